// norm_kernels.cuh -- the CUDA kernels of the fused RMSNorm / LayerNorm path.
//
// Definitions followed (web pages):
//  * "SOTA normalization performance with torch.compile", section "How Did
//    Torch.compile Catch Quack?": LayerNorm subtracts the row mean, divides by
//    the standard deviation, scales by gamma and adds beta; RMSNorm divides by
//    the root mean square and scales by gamma; the row statistics are stored
//    for the backward.  Its backward paragraph names dX, dW (gamma), dB (beta).
//  * "Fused RMSNorm", sections "What it is" / "How it works": read the row
//    once, keep it on chip, accumulate in fp32, write the result once.
//  * "Fused RMSNorm", sections "What didn't work" / "Next": dgamma partials go
//    to a workspace and a second kernel reduces them; no contended atomics.
//
// Three kernel families:
//  1. fwd_rows / bwd_rows: a row group of TPR threads (x CL CTAs of a
//     cluster) holds whole rows in registers as 16-byte vectors.  Thread t of
//     CTA rank c owns vectors (k*CL + c)*TPR + t, k < VPT, of every row it
//     touches, so each warp's loads and stores are contiguous 512-byte runs
//     and each thread always owns the same columns (which is what lets the
//     backward keep its dgamma/dbeta partials in registers across rows).
//     The grid is persistent: CTAs (or clusters) stride over rows; every
//     thread runs the same number of iterations, so barriers stay uniform.
//  2. fwd_elem / bwd_elem: one CTA per row, element-wise loads; serves any N
//     and any alignment (the row is re-read from L1/L2 between passes).
//  3. colreduce: sums the per-block partial rows of the workspace, column by
//     column, in a fixed order.
#pragma once

#include "device_common.cuh"
#include "params.h"

namespace gbn {

// ============================================================================ forward, row-resident
template <typename T, bool LN, int TPR, int VPT, int R, int CL, int CTA>
__global__ void __launch_bounds__(CTA) fwd_rows(const FwdParams p) {
    static_assert(CTA % TPR == 0 && (TPR <= 32 || TPR % 32 == 0), "bad row-group shape");
    static_assert(CL == 1 || TPR == CTA, "a cluster row uses whole CTAs");
    constexpr int E = VecTraits<T>::E;
    constexpr int RPC = CTA / TPR;
    // LayerNorm rows that fill the row group exactly (no cluster) take one
    // equal-count (mean, M2) combine; otherwise the mean first, then the
    // centred sum of squares.
    constexpr bool MERGE = LN && CL == 1;
    __shared__ RowReduceSmem<TPR, RPC, CL, MERGE ? 2 * R : 1> red2;
    __shared__ RowReduceSmem<TPR, RPC, CL, R> red;

    const int t = threadIdx.x % TPR;
    const int grp = threadIdx.x / TPR;
    const int rank = CL > 1 ? (int)cluster_ctarank() : 0;
    const int64_t nv = p.N / E;
    const float n = (float)p.N;
    const bool full = nv == (int64_t)TPR * VPT * CL;  // uniform over the grid

    int64_t vid[VPT];
    bool vok[VPT];
    uint4 gv[VPT], bv[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        vid[k] = ((int64_t)k * CL + rank) * TPR + t;
        vok[k] = vid[k] < nv;
        gv[k] = vok[k] ? param_vec<T>(p.gamma, vid[k], true) : make_uint4(0, 0, 0, 0);
        if constexpr (LN) bv[k] = vok[k] ? param_vec<T>(p.beta, vid[k], false) : make_uint4(0, 0, 0, 0);
    }

    int parity = 0;
    const int64_t start = CL > 1 ? (int64_t)cluster_id_x() * R : (int64_t)blockIdx.x * RPC * R;
    const int64_t step = CL > 1 ? (int64_t)cluster_count_x() * R : (int64_t)gridDim.x * RPC * R;
    for (int64_t base = start; base < p.M; base += step) {
        int64_t row[R];
        bool rok[R];
        uint4 xv[R][VPT];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            row[r] = base + (CL > 1 ? r : r * RPC + grp);
            rok[r] = row[r] < p.M;
#pragma unroll
            for (int k = 0; k < VPT; ++k)
                xv[r][k] = (rok[r] && vok[k]) ? ld_vec(p.x, row[r] * nv + vid[k])
                                              : make_uint4(0, 0, 0, 0);
        }
        // Pass 1: sum of squares (RMSNorm) or sum (LayerNorm), fp32.
        float s[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            s[r] = 0.f;
#pragma unroll
            for (int k = 0; k < VPT; ++k)
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float f = vget<T>(xv[r][k], e);
                    s[r] += LN ? f : f * f;
                }
        }
        float mean[R], rstd[R];
        if (MERGE && full) {
            // Every thread holds VPT * E elements of each row: local mean and
            // M2 from the registers, then one equal-count combine over the row.
            constexpr float kC = (float)(VPT * E);
            float m2[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                mean[r] = s[r] * (1.f / kC);
                m2[r] = 0.f;
#pragma unroll
                for (int k = 0; k < VPT; ++k)
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float d = vget<T>(xv[r][k], e) - mean[r];
                        m2[r] += d * d;
                    }
            }
            if constexpr (MERGE) row_meanvar_equal<TPR, RPC, R>(mean, m2, kC, red2, parity);
#pragma unroll
            for (int r = 0; r < R; ++r) rstd[r] = rsqrtf(m2[r] / n + p.eps);
        } else {
        row_allreduce<TPR, RPC, CL, R>(s, red, parity);
        if constexpr (LN) {
            // Pass 2 over the registers: centred sum of squares (no cancellation).
#pragma unroll
            for (int r = 0; r < R; ++r) {
                mean[r] = s[r] / n;
                s[r] = 0.f;
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    if (!vok[k]) continue;
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float d = vget<T>(xv[r][k], e) - mean[r];
                        s[r] += d * d;
                    }
                }
            }
            row_allreduce<TPR, RPC, CL, R>(s, red, parity);
#pragma unroll
            for (int r = 0; r < R; ++r) rstd[r] = rsqrtf(s[r] / n + p.eps);
        } else {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                mean[r] = 0.f;
                rstd[r] = rsqrtf(s[r] / n + p.eps);
            }
        }
        }
        if (t == 0 && rank == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (!rok[r]) continue;
                if (p.rstd) p.rstd[row[r]] = rstd[r];
                if (LN && p.mean) p.mean[row[r]] = mean[r];
            }
        }
        // Apply: y = ((x - mean) * rstd) * gamma (+ beta), rounded once.
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                if (!(rok[r] && vok[k])) continue;
                float o[E];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float xh = (vget<T>(xv[r][k], e) - mean[r]) * rstd[r];
                    o[e] = xh * vget<T>(gv[k], e);
                    if constexpr (LN) o[e] += vget<T>(bv[k], e);
                }
                st_vec(p.y, row[r] * nv + vid[k], vpack<T>(o));
            }
        }
    }
    // No CTA of a cluster may exit while a peer could still write into its
    // shared memory; every such write precedes the last barrier above, and
    // this final barrier makes the exit order irrelevant.
    if constexpr (CL > 1) cluster_sync_all();
}

// ============================================================================ forward, parameters in shared memory
// As fwd_rows (no cluster, one row per row group per iteration), with gamma
// (and beta) converted once per CTA to fp32 in shared memory (dynamic,
// [nv * E] floats each) instead of held packed in registers, and the row
// converted once to fp32 registers.  Fewer registers per thread (more warps
// per SM) and about half the instructions per element of fwd_rows for
// LayerNorm: x is converted once, gamma and beta not at all per row.
// RAW: gamma and beta staged in their storage type ([nv] 16-byte vectors
// each) and converted per use: a quarter of the fp32 planes' shared memory
// for 16-bit types, so more CTAs fit on an SM.
template <typename T, bool LN, int TPR, int VPT, int CTA, int MINB, bool RAW = false>
__global__ void __launch_bounds__(CTA, MINB) fwd_rows_s(const FwdParams p) {
    static_assert(CTA % TPR == 0 && TPR % 32 == 0, "bad row-group shape");
    constexpr int E = VecTraits<T>::E;
    constexpr int H = E / 4;  // float4 per 16-byte vector
    constexpr int RPC = CTA / TPR;
    // gamma as [H][nv] float4 (plane-major: a warp's 16-byte reads are
    // consecutive, no bank conflicts), then beta likewise
    extern __shared__ __align__(16) float4 pars[];
    uint4 *const parr = reinterpret_cast<uint4 *>(pars);  // RAW: gamma [nv], then beta [nv]
    __shared__ RowReduceSmem<TPR, RPC, 1, 2> red2;
    __shared__ RowReduceSmem<TPR, RPC, 1, 1> red1;

    const int t = threadIdx.x % TPR;
    const int grp = threadIdx.x / TPR;
    const int64_t nv = p.N / E;
    const float n = (float)p.N;
    const bool full = nv == (int64_t)TPR * VPT;  // uniform over the grid

    for (int64_t v = threadIdx.x; v < nv; v += CTA) {
        const uint4 g = param_vec<T>(p.gamma, v, true);
        uint4 b = make_uint4(0, 0, 0, 0);
        if constexpr (LN) b = param_vec<T>(p.beta, v, false);
        if constexpr (RAW) {
            parr[v] = g;
            if constexpr (LN) parr[nv + v] = b;
        } else {
#pragma unroll
            for (int h = 0; h < H; ++h) {
                pars[h * nv + v] = make_float4(vget<T>(g, 4 * h), vget<T>(g, 4 * h + 1), vget<T>(g, 4 * h + 2),
                                               vget<T>(g, 4 * h + 3));
                if constexpr (LN)
                    pars[(H + h) * nv + v] = make_float4(vget<T>(b, 4 * h), vget<T>(b, 4 * h + 1),
                                                         vget<T>(b, 4 * h + 2), vget<T>(b, 4 * h + 3));
            }
        }
    }
    __syncthreads();

    int64_t vid[VPT];
    bool vok[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        vid[k] = (int64_t)k * TPR + t;
        vok[k] = vid[k] < nv;
    }
    int parity = 0;
    for (int64_t base = (int64_t)blockIdx.x * RPC; base < p.M; base += (int64_t)gridDim.x * RPC) {
        const int64_t row = base + grp;
        const bool rok = row < p.M;
        float2 xf[VPT][E / 2];  // the row's elements of this thread, as pairs
        {
            uint4 q[VPT];
#pragma unroll
            for (int k = 0; k < VPT; ++k)
                q[k] = (rok && vok[k]) ? ld_vec(p.x, row * nv + vid[k]) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int k = 0; k < VPT; ++k)
#pragma unroll
                for (int e = 0; e < E / 2; ++e) xf[k][e] = vpair<T>(q[k], e);
        }
        // four independent accumulation chains per thread (two pairs)
        float2 sa[2] = {f2s(0.f), f2s(0.f)};
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < E / 2; ++e)
                sa[e & 1] = LN ? f2add(sa[e & 1], xf[k][e]) : f2fma(xf[k][e], xf[k][e], sa[e & 1]);
        const float s = (sa[0].x + sa[1].x) + (sa[0].y + sa[1].y);
        float mean = 0.f, rstd;
        if (LN && full) {
            // equal per-thread counts: local mean and M2, one combine (fwd_rows)
            constexpr float kC = (float)(VPT * E);
            float mm[1] = {s * (1.f / kC)}, m2[1];
            const float2 nmm = f2s(-mm[0]);
            float2 qa[2] = {f2s(0.f), f2s(0.f)};
#pragma unroll
            for (int k = 0; k < VPT; ++k)
#pragma unroll
                for (int e = 0; e < E / 2; ++e) {
                    const float2 d = f2add(xf[k][e], nmm);
                    qa[e & 1] = f2fma(d, d, qa[e & 1]);
                }
            m2[0] = (qa[0].x + qa[1].x) + (qa[0].y + qa[1].y);
            row_meanvar_equal<TPR, RPC, 1>(mm, m2, kC, red2, parity);
            mean = mm[0];
            rstd = rsqrtf(m2[0] / n + p.eps);
        } else {
            float a[1] = {s};
            row_allreduce<TPR, RPC, 1, 1>(a, red1, parity);
            if constexpr (LN) {
                mean = a[0] / n;
                const float2 nm = f2s(-mean);
                float2 q2 = f2s(0.f);
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    if (!vok[k]) continue;
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) {
                        const float2 d = f2add(xf[k][e], nm);
                        q2 = f2fma(d, d, q2);
                    }
                }
                a[0] = q2.x + q2.y;
                row_allreduce<TPR, RPC, 1, 1>(a, red1, parity);
            }
            rstd = rsqrtf(a[0] / n + p.eps);
        }
        if (t == 0 && rok) {
            if (p.rstd) p.rstd[row] = rstd;
            if (LN && p.mean) p.mean[row] = mean;
        }
        // y = ((x - mean) * rstd) * gamma (+ beta)
        const float2 nm = f2s(-mean), rs = f2s(rstd);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            if (!(rok && vok[k])) continue;
            float2 o[E / 2];
            if constexpr (RAW) {
                const uint4 g = parr[vid[k]];
                uint4 b = make_uint4(0, 0, 0, 0);
                if constexpr (LN) b = parr[nv + vid[k]];
#pragma unroll
                for (int e = 0; e < E / 2; ++e) {
                    o[e] = f2mul(f2mul(f2add(xf[k][e], nm), rs), vpair<T>(g, e));
                    if constexpr (LN) o[e] = f2add(o[e], vpair<T>(b, e));
                }
            } else {
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float4 g = pars[h * nv + vid[k]];
                    o[2 * h] = f2mul(f2mul(f2add(xf[k][2 * h], nm), rs), make_float2(g.x, g.y));
                    o[2 * h + 1] = f2mul(f2mul(f2add(xf[k][2 * h + 1], nm), rs), make_float2(g.z, g.w));
                    if constexpr (LN) {
                        const float4 b = pars[(H + h) * nv + vid[k]];
                        o[2 * h] = f2add(o[2 * h], make_float2(b.x, b.y));
                        o[2 * h + 1] = f2add(o[2 * h + 1], make_float2(b.z, b.w));
                    }
                }
            }
            st_vec(p.y, row * nv + vid[k], vpack2<T>(o));
        }
    }
}

// ============================================================================ backward, row-resident
// Per row: xhat = (x - mean) * rstd, g = dy * gamma, c2 = mean(g * xhat),
// c1 = mean(g) (LayerNorm), dx = rstd * (g - c1 - xhat * c2).  Each thread
// adds dy * xhat (and dy) into fp32 registers for the columns it owns; at the
// end the CTA (or each CTA of a cluster) writes one partial row per block into
// ws[P, N] (and ws[P, N] after it for dbeta).
template <typename T, bool LN, int TPR, int VPT, int R, int CL, int CTA>
__global__ void __launch_bounds__(CTA) bwd_rows(const BwdParams p) {
    static_assert(CTA % TPR == 0 && (TPR <= 32 || TPR % 32 == 0), "bad row-group shape");
    pdl_launch_dependents();  // the column reduce waits for this grid's completion
    static_assert(CL == 1 || TPR == CTA, "a cluster row uses whole CTAs");
    constexpr int E = VecTraits<T>::E;
    constexpr int RPC = CTA / TPR;
    constexpr int NS = LN ? 2 * R : R;  // sums reduced per row batch
    __shared__ RowReduceSmem<TPR, RPC, CL, NS> red;
    // Row-group combine buffer for the epilogue: one row of partials (x2 for LN).
    __shared__ float comb[RPC > 1 ? TPR * VPT * E * (LN ? 2 : 1) : 1];

    const int t = threadIdx.x % TPR;
    const int grp = threadIdx.x / TPR;
    const int rank = CL > 1 ? (int)cluster_ctarank() : 0;
    const int64_t nv = p.N / E;
    const float n = (float)p.N;

    int64_t vid[VPT];
    bool vok[VPT];
    uint4 gv[VPT];
    float accg[VPT][E], accb[LN ? VPT : 1][E];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        vid[k] = ((int64_t)k * CL + rank) * TPR + t;
        vok[k] = vid[k] < nv;
        gv[k] = vok[k] ? param_vec<T>(p.gamma, vid[k], true) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            accg[k][e] = 0.f;
            if constexpr (LN) accb[k][e] = 0.f;
        }
    }

    int parity = 0;
    const int64_t start = CL > 1 ? (int64_t)cluster_id_x() * R : (int64_t)blockIdx.x * RPC * R;
    const int64_t step = CL > 1 ? (int64_t)cluster_count_x() * R : (int64_t)gridDim.x * RPC * R;
    for (int64_t base = start; base < p.M; base += step) {
        int64_t row[R];
        bool rok[R];
        uint4 xv[R][VPT], dv[R][VPT];
        float mean[R], rstd[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            row[r] = base + (CL > 1 ? r : r * RPC + grp);
            rok[r] = row[r] < p.M;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const bool ok = rok[r] && vok[k];
                xv[r][k] = ok ? ld_vec(p.x, row[r] * nv + vid[k]) : make_uint4(0, 0, 0, 0);
                dv[r][k] = ok ? ld_vec(p.dy, row[r] * nv + vid[k]) : make_uint4(0, 0, 0, 0);
            }
            rstd[r] = rok[r] ? __ldg(p.rstd + row[r]) : 0.f;
            mean[r] = (LN && rok[r]) ? __ldg(p.mean + row[r]) : 0.f;
        }
        // Row sums: s[r] = sum g * xhat, s[R + r] = sum g (LayerNorm).
        float s[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i) s[i] = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int k = 0; k < VPT; ++k)
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float xh = (vget<T>(xv[r][k], e) - mean[r]) * rstd[r];
                    const float g = vget<T>(dv[r][k], e) * vget<T>(gv[k], e);
                    s[r] += g * xh;
                    if constexpr (LN) s[R + r] += g;
                }
        row_allreduce<TPR, RPC, CL, NS>(s, red, parity);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float c2 = s[r] / n;
            const float c1 = LN ? s[LN ? R + r : 0] / n : 0.f;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                float o[E];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float xh = (vget<T>(xv[r][k], e) - mean[r]) * rstd[r];
                    const float dyv = vget<T>(dv[r][k], e);
                    const float g = dyv * vget<T>(gv[k], e);
                    o[e] = rstd[r] * (g - c1 - xh * c2);
                    // Masked slots hold dy = 0, so they add nothing.
                    accg[k][e] += dyv * xh;
                    if constexpr (LN) accb[k][e] += dyv;
                }
                if (rok[r] && vok[k]) st_vec(p.dx, row[r] * nv + vid[k], vpack<T>(o));
            }
        }
    }

    // Epilogue: one partial row per block (CTA, or cluster), columns in order.
    const int64_t prow = CL > 1 ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
    const int64_t P = CL > 1 ? (int64_t)cluster_count_x() : (int64_t)gridDim.x;
    float *wsg = p.ws + prow * p.N;
    float *wsb = p.ws + (P + prow) * p.N;
    if constexpr (RPC > 1) {
        // Row groups of this CTA own the same columns: add them in group order.
        constexpr int CAP = TPR * VPT * E;
        for (int gi = 0; gi < RPC; ++gi) {
            if (grp == gi) {
#pragma unroll
                for (int k = 0; k < VPT; ++k)
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const int c = (k * TPR + t) * E + e;
                        comb[c] = gi == 0 ? accg[k][e] : comb[c] + accg[k][e];
                        if constexpr (LN)
                            comb[CAP + c] = gi == 0 ? accb[k][e] : comb[CAP + c] + accb[k][e];
                    }
            }
            __syncthreads();
        }
        // Write the combined row: CTA threads stride over its vectors.
        for (int i = threadIdx.x; i < TPR * VPT; i += CTA) {
            const int k = i / TPR, tt = i % TPR;
            const int64_t v = (int64_t)k * TPR + tt;  // CL == 1 here
            if (v >= nv) continue;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                wsg[v * E + e] = comb[i * E + e];
                if constexpr (LN) wsb[v * E + e] = comb[CAP + i * E + e];
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            if (!vok[k]) continue;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                wsg[vid[k] * E + e] = accg[k][e];
                if constexpr (LN) wsb[vid[k] * E + e] = accb[k][e];
            }
        }
    }
    if constexpr (CL > 1) cluster_sync_all();
}

// ============================================================================ element-wise path (any N, any alignment)
template <typename T, bool LN>
__global__ void __launch_bounds__(kElemCTA) fwd_elem(const FwdParams p) {
    __shared__ float red[2 * 1 * (kElemCTA / 32)];
    const T *x = static_cast<const T *>(p.x);
    const T *gamma = static_cast<const T *>(p.gamma);
    const T *beta = static_cast<const T *>(p.beta);
    T *y = static_cast<T *>(p.y);
    const float n = (float)p.N;
    int parity = 0;
    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
        const T *xr = x + row * p.N;
        float s[1] = {0.f};
        for (int64_t j = threadIdx.x; j < p.N; j += kElemCTA) {
            const float f = to_f(xr[j]);
            s[0] += LN ? f : f * f;
        }
        cta_allreduce<kElemCTA, 1>(s, red, parity);
        float mean = 0.f, rstd;
        if constexpr (LN) {
            mean = s[0] / n;
            s[0] = 0.f;
            for (int64_t j = threadIdx.x; j < p.N; j += kElemCTA) {
                const float d = to_f(xr[j]) - mean;
                s[0] += d * d;
            }
            cta_allreduce<kElemCTA, 1>(s, red, parity);
        }
        rstd = rsqrtf(s[0] / n + p.eps);
        if (threadIdx.x == 0) {
            if (p.rstd) p.rstd[row] = rstd;
            if (LN && p.mean) p.mean[row] = mean;
        }
        T *yr = y + row * p.N;
        for (int64_t j = threadIdx.x; j < p.N; j += kElemCTA) {
            float o = ((to_f(xr[j]) - mean) * rstd) * (gamma ? to_f(gamma[j]) : 1.f);
            if (LN && beta) o += to_f(beta[j]);
            yr[j] = from_f<T>(o);
        }
    }
}

// Each CTA accumulates its partial dgamma/dbeta row directly in its own row
// of the workspace (no other CTA touches it), zeroed first.
template <typename T, bool LN>
__global__ void __launch_bounds__(kElemCTA) bwd_elem(const BwdParams p) {
    pdl_launch_dependents();  // the column reduce waits for this grid's completion
    __shared__ float red[2 * 2 * (kElemCTA / 32)];
    const T *x = static_cast<const T *>(p.x);
    const T *dy = static_cast<const T *>(p.dy);
    const T *gamma = static_cast<const T *>(p.gamma);
    T *dx = static_cast<T *>(p.dx);
    const float n = (float)p.N;
    const int64_t P = gridDim.x;
    float *wsg = p.ws + (int64_t)blockIdx.x * p.N;
    float *wsb = p.ws + (P + blockIdx.x) * p.N;
    for (int64_t j = threadIdx.x; j < p.N; j += kElemCTA) {
        wsg[j] = 0.f;
        if constexpr (LN) wsb[j] = 0.f;
    }
    int parity = 0;
    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
        const T *xr = x + row * p.N;
        const T *dyr = dy + row * p.N;
        const float rstd = __ldg(p.rstd + row);
        const float mean = LN ? __ldg(p.mean + row) : 0.f;
        float s[2] = {0.f, 0.f};
        for (int64_t j = threadIdx.x; j < p.N; j += kElemCTA) {
            const float xh = (to_f(xr[j]) - mean) * rstd;
            const float g = to_f(dyr[j]) * (gamma ? to_f(gamma[j]) : 1.f);
            s[0] += g * xh;
            s[1] += g;
        }
        cta_allreduce<kElemCTA, 2>(s, red, parity);
        const float c2 = s[0] / n;
        const float c1 = LN ? s[1] / n : 0.f;
        T *dxr = dx + row * p.N;
        for (int64_t j = threadIdx.x; j < p.N; j += kElemCTA) {
            const float xh = (to_f(xr[j]) - mean) * rstd;
            const float dyv = to_f(dyr[j]);
            const float g = dyv * (gamma ? to_f(gamma[j]) : 1.f);
            dxr[j] = from_f<T>(rstd * (g - c1 - xh * c2));
            wsg[j] += dyv * xh;
            if constexpr (LN) wsb[j] += dyv;
        }
    }
}

// ============================================================================ column reduce
// out_s[j] = sum_{p < P} ws[s][p][j] for s = blockIdx.y (0: dgamma, 1: dbeta).
// A CTA owns 32 column groups of VW columns; its W warps each sum a fixed,
// contiguous band of rows, and the W band sums are added in warp order, so
// the result does not depend on timing.
template <int VW>  // 4: float4 columns (N % 4 == 0), 1: scalar columns
__global__ void __launch_bounds__(kColCTA) colreduce(const float *ws, int64_t P, int64_t N,
                                                     float *out0, float *out1) {
    constexpr int W = kColCTA / 32;
    __shared__ float part[W][32 * VW];
    // Launched right behind the backward row kernel that writes `ws`.
    pdl_wait_primary();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *src = ws + (int64_t)blockIdx.y * P * N;
    float *out = blockIdx.y ? out1 : out0;
    if (out == nullptr) return;  // that sum is not wanted
    const int64_t col = ((int64_t)blockIdx.x * 32 + lane) * VW;
    const bool ok = col < N;
    const int64_t p0 = P * warp / W, p1 = P * (warp + 1) / W;
    float acc[VW];
#pragma unroll
    for (int v = 0; v < VW; ++v) acc[v] = 0.f;
    if (ok) {
        // Bands of up to kColBatch rows: all loads of a batch are issued before
        // any is added, so a band costs one memory latency, not one per row.
        constexpr int kColBatch = 16;
        for (int64_t q0 = p0; q0 < p1; q0 += kColBatch) {
            if constexpr (VW == 4) {
                const float4 *s4 = reinterpret_cast<const float4 *>(src + col);
                const int64_t stride = N / 4;
                float4 a[kColBatch];
#pragma unroll
                for (int i = 0; i < kColBatch; ++i)
                    a[i] = q0 + i < p1 ? __ldg(s4 + (q0 + i) * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int i = 0; i < kColBatch; ++i) {
                    acc[0] += a[i].x;
                    acc[1] += a[i].y;
                    acc[2] += a[i].z;
                    acc[3] += a[i].w;
                }
            } else {
                float a[kColBatch];
#pragma unroll
                for (int i = 0; i < kColBatch; ++i) a[i] = q0 + i < p1 ? __ldg(src + (q0 + i) * N + col) : 0.f;
#pragma unroll
                for (int i = 0; i < kColBatch; ++i) acc[0] += a[i];
            }
        }
    }
#pragma unroll
    for (int v = 0; v < VW; ++v) part[warp][lane * VW + v] = acc[v];
    __syncthreads();
    if (warp == 0 && ok) {
        float r[VW];
#pragma unroll
        for (int v = 0; v < VW; ++v) {
            r[v] = 0.f;
            for (int w = 0; w < W; ++w) r[v] += part[w][lane * VW + v];
        }
        if constexpr (VW == 4) {
            if ((reinterpret_cast<uintptr_t>(out + col) & 15) == 0) {
                *reinterpret_cast<float4 *>(out + col) = make_float4(r[0], r[1], r[2], r[3]);
            } else {
#pragma unroll
                for (int v = 0; v < 4; ++v) out[col + v] = r[v];
            }
        } else {
            out[col] = r[0];
        }
    }
}

}  // namespace gbn
