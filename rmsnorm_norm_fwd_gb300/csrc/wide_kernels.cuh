// wide_kernels.cuh -- RMSNorm / LayerNorm forward for wide rows without a
// thread-block cluster: one CTA owns a whole row at a time and reads it twice.
//
// Same arithmetic as norm_kernels.cuh (the definitions on "SOTA normalization
// performance with torch.compile", section "How Did Torch.compile Catch
// Quack?", and "Fused RMSNorm", sections "What it is" / "How it works").
//
// A row too wide for one SM's registers and shared memory is normally split
// across a cluster, but a cluster of 8 or 16 CTAs only fits on part of the
// GPU (whole clusters per GPC) and every row then waits on a cross-CTA
// exchange.  Here each CTA streams its row from DRAM for the statistics
// (pass 1, loads marked L2 evict_last), reduces over the CTA, and streams the
// row again for the output (pass 2, the same lines now hit in L2 and are
// marked evict_first; y is written evict_first).  The L2 holds the rows in
// flight: CTAs x row bytes (about 40 MB for 152 CTAs of 256 KB rows).  Rows
// are independent, every SM works, and two or more CTAs per SM overlap one
// row's reduction with another's streaming.
//
// LayerNorm statistics: each thread reduces its batches of U vectors exactly
// (batch mean, then the batch's centred sum of squares from the registers),
// folds them into a running (count, mean, M2) with the pairwise update of
// Chan, Golub and LeVeque (1979), and the CTA combines the threads' triples
// with the same update -- no E[x^2] - mean^2 cancellation.
#pragma once

#include "device_common.cuh"
#include "params.h"

namespace gbn {

// L2 eviction-priority policies (createpolicy, PTX ISA "Cache Eviction
// Priority Hints"), applied per access with .L2::cache_hint.
__device__ __forceinline__ uint64_t l2_policy_keep() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_drop() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// 16-byte read-only load with an L2 policy (not kept in L1).
__device__ __forceinline__ uint4 ld_l2hint(const uint4 *p, uint64_t pol) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ void st_l2hint(uint4 *p, const uint4 &v, uint64_t pol) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;"
                 :
                 : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

// Bulk prefetch of bytes (a multiple of 16) at a 16-byte-aligned global
// address into L2, kept there (evict_last); no registers or shared memory.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes, uint64_t pol) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;"
                 :
                 : "l"(p), "r"(bytes), "l"(pol)
                 : "memory");
}
// Warp-cooperative bulk prefetch of one row (row_bytes a multiple of 16) in
// chunks of at most 16 KB.
__device__ __forceinline__ void prefetch_row(const void *row, size_t row_bytes, int lane, uint64_t pol) {
    constexpr size_t kChunk = 16384;
    for (size_t off = (size_t)lane * kChunk; off < row_bytes; off += 32 * kChunk) {
        const size_t b = row_bytes - off < kChunk ? row_bytes - off : kChunk;
        prefetch_l2_bulk(static_cast<const unsigned char *>(row) + off, (uint32_t)b, pol);
    }
}

// Combine of groups' (count n_g, mean m_g, M2_g) into the union's:
// n = sum n_g, mean = (sum n_g m_g) / n, M2 = sum (M2_g + n_g (m_g - mean)^2)
// (the group form of the update of Chan, Golub and LeVeque, 1979; exact in
// exact arithmetic and centred on the union's mean).  Over the 32 lanes of a
// warp: three butterfly sums, every lane ends with identical bits (each
// butterfly step adds two operands in either order).  An empty union gives
// (0, 0, 0).
template <int G = 32>
__device__ __forceinline__ void warp_combine(float &n, float &mean, float &m2) {
    float tn = n, ts = n * mean;
#pragma unroll
    for (int o = 1; o < G; o <<= 1) {
        tn += __shfl_xor_sync(0xffffffffu, tn, o);
        ts += __shfl_xor_sync(0xffffffffu, ts, o);
    }
    const float mu = tn > 0.f ? ts / tn : 0.f;
    const float d = mean - mu;
    float tm = m2 + n * (d * d);
#pragma unroll
    for (int o = 1; o < G; o <<= 1) tm += __shfl_xor_sync(0xffffffffu, tm, o);
    n = tn;
    mean = mu;
    m2 = tm;
}

// PF (prefetch): 0 none; 1 each row is bulk-prefetched into L2 as its pass 1
// starts; 2 as 1 for the first rows, then the CTA's next rows are prefetched
// as the current rows' pass 2 starts (twice the rows per CTA resident in L2).
// R rows per CTA at a time: their pass-1 loads share the batches, their
// statistics one CTA barrier, and their pass 2 one load of gamma (and beta)
// per vector, which halves (R = 2) the L2 reads of the parameters.
template <typename T, bool LN, int NT, int UV, int MINB, int PF, int R>
__global__ void __launch_bounds__(NT, MINB) fwd_wide(const FwdParams p) {
    constexpr int E = VecTraits<T>::E;
    constexpr int W = NT / 32;
    constexpr bool kRoomy = 65536 / (NT * MINB) >= 128;  // registers per thread >= 128
    // Vectors per thread per load batch (all R rows together at most 8, and
    // at most 4 for the LayerNorm batch, read twice from registers, when
    // registers are short).
    constexpr int UR = UV * R > 8 ? (8 / R > 0 ? 8 / R : 1) : UV;
    constexpr int U = (LN && !kRoomy && UR * R > 4) ? (4 / R > 0 ? 4 / R : 1) : UR;
    // Pass 2 loads x of R rows and gamma (and beta) per vector: fewer vectors
    // per batch unless the register budget is roomy.
    constexpr int U2r = LN ? U / 2 : (kRoomy ? U : U / 2);
    constexpr int U2 = U2r > 0 ? U2r : 1;
    // Independent partial sums per thread and row in pass 1.
    constexpr int A0 = (LN && !kRoomy) ? 2 : (R > 1 ? 2 : 4);
    constexpr int A = U < A0 ? U : A0;
    static_assert(NT % 32 == 0 && NT <= 1024 && R >= 1 && R <= 2, "CTA shape");
    __shared__ float red[2][3][R][W];

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int64_t nv = p.N / E;
    const float n = (float)p.N;
    const size_t row_bytes = (size_t)nv * 16;
    const uint64_t keep = l2_policy_keep(), drop = l2_policy_drop();
    const uint4 *gam = static_cast<const uint4 *>(p.gamma);
    const uint4 *bet = static_cast<const uint4 *>(p.beta);
    const uint4 *xg = static_cast<const uint4 *>(p.x);
    int parity = 0;
    const int64_t step = (int64_t)gridDim.x * R;

    auto prefetch_rows = [&](int64_t base) {
        if (warp == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (base + r < p.M) prefetch_row(xg + (base + r) * nv, row_bytes, lane, keep);
        }
    };
    if (PF == 2) prefetch_rows((int64_t)blockIdx.x * R);

    for (int64_t base = (int64_t)blockIdx.x * R; base < p.M; base += step) {
        bool ok[R];
        const uint4 *xr[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            ok[r] = base + r < p.M;
            xr[r] = xg + (ok[r] ? base + r : base) * nv;
        }
        if (PF == 1) prefetch_rows(base);

        // ---- pass 1: statistics (rows from DRAM, kept in L2)
        float cnt[R], mean[R], acc[R];  // acc: sum x^2 (RMS) or M2 (LN)
        float2 pa[R][A];                // RMS partial sums of squares, as pairs
#pragma unroll
        for (int r = 0; r < R; ++r) {
            cnt[r] = mean[r] = acc[r] = 0.f;
#pragma unroll
            for (int a = 0; a < A; ++a) pa[r][a] = f2s(0.f);
        }
        for (int64_t b = t; b < nv; b += (int64_t)NT * U) {
            uint4 q[R][U];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t v = b + (int64_t)u * NT;
                    q[r][u] = (ok[r] && v < nv) ? ld_l2hint(xr[r] + v, keep) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if constexpr (!LN) {
#pragma unroll
                    for (int u = 0; u < U; ++u)
#pragma unroll
                        for (int e = 0; e < E / 2; ++e) {
                            const float2 f = vpair<T>(q[r][u], e);
                            pa[r][u % A] = f2fma(f, f, pa[r][u % A]);
                        }
                } else {
                    float2 ps[A], pm[A];
                    int nb = 0;
#pragma unroll
                    for (int a = 0; a < A; ++a) ps[a] = pm[a] = f2s(0.f);
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        if (b + (int64_t)u * NT < nv) {
                            nb += E;
#pragma unroll
                            for (int e = 0; e < E / 2; ++e) ps[u % A] = f2add(ps[u % A], vpair<T>(q[r][u], e));
                        }
                    }
                    float s = ps[0].x + ps[0].y;
#pragma unroll
                    for (int a = 1; a < A; ++a) s += ps[a].x + ps[a].y;
                    const float fb = (float)nb;
                    const float mb = __fdiv_rn(s, fb);
                    const float2 nmb = f2s(-mb);
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        if (b + (int64_t)u * NT < nv) {
#pragma unroll
                            for (int e = 0; e < E / 2; ++e) {
                                const float2 d = f2add(vpair<T>(q[r][u], e), nmb);
                                pm[u % A] = f2fma(d, d, pm[u % A]);
                            }
                        }
                    }
                    float m2b = pm[0].x + pm[0].y;
#pragma unroll
                    for (int a = 1; a < A; ++a) m2b += pm[a].x + pm[a].y;
                    if (cnt[r] == 0.f) {
                        cnt[r] = fb;
                        mean[r] = mb;
                        acc[r] = m2b;
                    } else {
                        // running += batch (one division per batch of U vectors)
                        const float tot = cnt[r] + fb;
                        const float d = mb - mean[r];
                        const float rr = __fdiv_rn(fb, tot);
                        mean[r] += d * rr;
                        acc[r] += m2b + d * d * cnt[r] * rr;
                        cnt[r] = tot;
                    }
                }
            }
        }
        if constexpr (!LN) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                acc[r] = pa[r][0].x + pa[r][0].y;
#pragma unroll
                for (int a = 1; a < A; ++a) acc[r] += pa[r][a].x + pa[r][a].y;
            }
        }

        // ---- CTA reduction (identical bits in every thread)
        float (*buf)[R][W] = red[parity];
        parity ^= 1;
        if constexpr (!LN) {
#pragma unroll
            for (int o = 1; o < 32; o <<= 1)
#pragma unroll
                for (int r = 0; r < R; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < R; ++r) buf[0][r][warp] = acc[r];
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < R; ++r) {
                acc[r] = 0.f;
#pragma unroll 4
                for (int w = 0; w < W; ++w) acc[r] += buf[0][r][w];
            }
        } else {
#pragma unroll
            for (int r = 0; r < R; ++r) warp_combine(cnt[r], mean[r], acc[r]);
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    buf[0][r][warp] = cnt[r];
                    buf[1][r][warp] = mean[r];
                    buf[2][r][warp] = acc[r];
                }
            }
            __syncthreads();
            // the same group combine over the W warps, in warp order
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float tn = 0.f, ts = 0.f;
#pragma unroll 4
                for (int w = 0; w < W; ++w) {
                    tn += buf[0][r][w];
                    ts += buf[0][r][w] * buf[1][r][w];
                }
                mean[r] = ts / tn;  // tn = N > 0
                float a2 = 0.f;
#pragma unroll 4
                for (int w = 0; w < W; ++w) {
                    const float d = buf[1][r][w] - mean[r];
                    a2 += buf[2][r][w] + buf[0][r][w] * (d * d);
                }
                acc[r] = a2;
            }
        }
        float rstd[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            rstd[r] = rsqrtf(acc[r] / n + p.eps);
            if (!LN) mean[r] = 0.f;
            if (t == 0 && ok[r]) {
                if (p.rstd) p.rstd[base + r] = rstd[r];
                if (LN && p.mean) p.mean[base + r] = mean[r];
            }
        }

        if (PF == 2) prefetch_rows(base + step);

        // ---- pass 2: y = (x - mean) * rstd * gamma (+ beta), x from L2
        for (int64_t b = t; b < nv; b += (int64_t)NT * U2) {
            uint4 q[R][U2], g[U2], bb[LN ? U2 : 1];
#pragma unroll
            for (int u = 0; u < U2; ++u) {
                const int64_t v = b + (int64_t)u * NT;
                if (v < nv) {
                    g[u] = gam ? ld_l2hint(gam + v, keep) : ones_vec<T>();
                    if constexpr (LN) bb[u] = bet ? ld_l2hint(bet + v, keep) : make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        if (ok[r]) q[r][u] = ld_l2hint(xr[r] + v, drop);
                }
            }
#pragma unroll
            for (int u = 0; u < U2; ++u) {
                const int64_t v = b + (int64_t)u * NT;
                if (v >= nv) continue;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (!ok[r]) continue;
                    float2 o[E / 2];
                    const float2 nm = f2s(-mean[r]), rs = f2s(rstd[r]);
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) {
                        o[e] = f2mul(f2mul(f2add(vpair<T>(q[r][u], e), nm), rs), vpair<T>(g[u], e));
                        if constexpr (LN) o[e] = f2add(o[e], vpair<T>(bb[u], e));
                    }
                    st_l2hint(static_cast<uint4 *>(p.y) + (base + r) * nv + v, vpack2<T>(o), drop);
                }
            }
        }
    }
}

}  // namespace gbn

namespace gbn {

// ============================================================================ backward
// Backward for wide rows: a cluster of CL CTAs (CL = 1, 2, 4, 8 or 16) shares each
// row; CTA `rank` owns a contiguous column slice and keeps its dgamma (and
// dbeta) partial sums for that slice in shared memory across all the rows it
// visits.  Per row: pass 1 streams the slice of x and dy from DRAM (L2
// evict_last) for the partial sums sum g xhat and sum g (g = dy gamma), the
// CTA reduces them and sends them to every CTA of the cluster through
// distributed shared memory; pass 2 re-reads the slice from L2, writes
// dx = rstd (g - c1 - xhat c2) and adds dy xhat (and dy) into the shared
// accumulators.  At the end each CTA writes its slice of the cluster's
// partial row; the column-reduce kernel sums the partial rows.
//
// Pipeline: iteration j of a CTA sweeps its slice once for both pass 1 of
// its row j and pass 2 of its row j - 2 (gamma loaded once for both), so each
// batch has two rows' loads in flight; then it reduces and sends row j's
// partials and waits for row j - 1's exchange, which has had a whole sweep to
// complete.
//
// Exchange: each CTA stores its partials of row k into slot [k % 4][rank] of
// every CTA (st.shared::cluster) and arrives with release semantics on that
// CTA's barrier xch[k % 4]; it waits (acquire, bounded) for CL arrivals,
// then adds the CL partials in rank order, so every CTA gets identical bits.
// Reuse is safe with four slots: a peer sends row k + 4 only after it has
// received this CTA's row k + 2, which this CTA sends after a CTA barrier
// that follows its reads of row k's slots (and its completed wait for row k).

// One sweep of a CTA over its slice: pass 1 of one row (P1) and pass 2 of
// another (P2), batch by batch.  v: this thread's pass-1 partial sums.
template <typename T, bool LN, int NT, int U, bool P1, bool P2>
__device__ __forceinline__ void wide_bwd_sweep(int t, int cnt, int64_t slice, const uint4 *gr,
                                               float4 *accs, const uint4 *x1, const uint4 *d1,
                                               float mean1, float rstd1, float (&v)[LN ? 2 : 1],
                                               const uint4 *x2, const uint4 *d2, uint4 *dx2,
                                               float mean2, float rstd2, float c1, float c2,
                                               uint64_t keep, uint64_t drop) {
    constexpr int E = VecTraits<T>::E;
    constexpr int H = E / 4;
    constexpr int A = U < 2 ? U : 2;  // independent partial-sum chains
    float a2[A], a1[A];
#pragma unroll
    for (int a = 0; a < A; ++a) a2[a] = a1[a] = 0.f;
    for (int b = t; b < cnt; b += NT * U) {
        uint4 px[U], pd[U], qx[U], qd[U], g[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int vv = b + u * NT;
            if (vv < cnt) {
                g[u] = gr ? ld_l2hint(gr + vv, keep) : ones_vec<T>();
                if constexpr (P1) {
                    px[u] = ld_l2hint(x1 + vv, keep);
                    pd[u] = ld_l2hint(d1 + vv, keep);
                }
                if constexpr (P2) {
                    qx[u] = ld_l2hint(x2 + vv, drop);
                    qd[u] = ld_l2hint(d2 + vv, drop);
                }
            } else {
                g[u] = px[u] = pd[u] = make_uint4(0, 0, 0, 0);
            }
        }
        if constexpr (P2) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int vv = b + u * NT;
                if (vv < cnt) {
                    float o[E], dg[E], dyv[E];
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float xh = (vget<T>(qx[u], e) - mean2) * rstd2;
                        dyv[e] = vget<T>(qd[u], e);
                        const float gg = dyv[e] * vget<T>(g[u], e);
                        o[e] = rstd2 * (gg - c1 - xh * c2);
                        dg[e] = dyv[e] * xh;
                    }
                    st_l2hint(dx2 + vv, vpack<T>(o), drop);
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        float4 &ag = accs[h * slice + vv];
                        float4 a = ag;
                        a.x += dg[4 * h];
                        a.y += dg[4 * h + 1];
                        a.z += dg[4 * h + 2];
                        a.w += dg[4 * h + 3];
                        ag = a;
                        if constexpr (LN) {
                            float4 &ab = accs[(H + h) * slice + vv];
                            float4 q = ab;
                            q.x += dyv[4 * h];
                            q.y += dyv[4 * h + 1];
                            q.z += dyv[4 * h + 2];
                            q.w += dyv[4 * h + 3];
                            ab = q;
                        }
                    }
                }
            }
        }
        if constexpr (P1) {
            // lanes past the slice hold zeros: g = 0 adds nothing
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float xh = (vget<T>(px[u], e) - mean1) * rstd1;
                    const float gg = vget<T>(pd[u], e) * vget<T>(g[u], e);
                    a2[u % A] += gg * xh;
                    if constexpr (LN) a1[u % A] += gg;
                }
        }
    }
    if constexpr (P1) {
        v[0] = a2[0];
#pragma unroll
        for (int a = 1; a < A; ++a) v[0] += a2[a];
        if constexpr (LN) {
            v[1] = a1[0];
#pragma unroll
            for (int a = 1; a < A; ++a) v[1] += a1[a];
        }
    }
}

// FUSE: 1 the schedule above; 0 pass 1 of row k + 1 (and its send), then the
// wait for row k's exchange, then pass 2 of row k (one row's loads per batch,
// larger batches).
// MINB: CTAs per SM the launch bound asks for (registers 65536 / (NT * MINB)).
template <typename T, bool LN, int NT, int U, int CL, int PF, int FUSE, int MINB>
__global__ void __launch_bounds__(NT, MINB) bwd_wide(const BwdParams p) {
    pdl_launch_dependents();  // the column reduce waits for this grid's completion
    constexpr int E = VecTraits<T>::E;
    constexpr int W = NT / 32;
    constexpr int H = E / 4;          // float4 accumulators per 16-byte vector
    constexpr int NVAL = LN ? 2 : 1;  // partial sums per row; accumulator planes
    constexpr int NS = 4;             // exchange slots
    static_assert(NT % 32 == 0 && NT <= 1024 && CL >= 1 && CL <= 16, "shape");
    extern __shared__ __align__(16) float4 accs[];  // [NVAL][H][slice]
    __shared__ float red[2][NVAL][W];
    __shared__ float slot[NS][CL][NVAL];
    __shared__ __align__(8) uint64_t xch[NS];
    __shared__ int abort_flag;

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int rank = CL > 1 ? (int)cluster_ctarank() : 0;
    const int64_t cid = CL > 1 ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
    const int64_t ncl = CL > 1 ? (int64_t)cluster_count_x() : (int64_t)gridDim.x;
    const int64_t M = p.M, nv = p.N / E;
    const int64_t slice = (nv + CL - 1) / CL;
    const int64_t v0 = rank * slice;
    const int cnt = (int)(nv - v0 < slice ? nv - v0 : slice);
    const float n = (float)p.N;
    const uint64_t keep = l2_policy_keep(), drop = l2_policy_drop();
    const uint4 *gr = p.gamma ? static_cast<const uint4 *>(p.gamma) + v0 : nullptr;  // null: gamma = 1
    const size_t slice_bytes = (size_t)cnt * 16;

    for (int64_t i = t; i < (int64_t)NVAL * H * slice; i += NT) accs[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t == 0) {
        abort_flag = 0;
        if (CL > 1) {
            for (int j = 0; j < NS; ++j) mbar_init(&xch[j], CL);
            fence_mbar_init();
        }
    }
    // Every CTA's barriers exist before any peer arrives on them.
    if constexpr (CL > 1) cluster_sync_all();
    else __syncthreads();

    const int64_t nrows = cid < M ? (M - cid + ncl - 1) / ncl : 0;
    auto row_of = [&](int64_t k) { return cid + k * ncl; };
    auto row_x = [&](int64_t k) { return static_cast<const uint4 *>(p.x) + row_of(k) * nv + v0; };
    auto row_dy = [&](int64_t k) { return static_cast<const uint4 *>(p.dy) + row_of(k) * nv + v0; };
    auto prefetch = [&](int64_t k) {
        if (warp == 0 && k < nrows) {
            prefetch_row(row_x(k), slice_bytes, lane, keep);
            prefetch_row(row_dy(k), slice_bytes, lane, keep);
        }
    };
    int parity = 0;
    float cst[3][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};  // (c1, c2) of row k at [k % 3], once known

    // Row k's pass-1 partials v, summed over the CTA (identical bits in every
    // thread), then sent to the cluster (or, without one, turned into c1, c2).
    auto finish_pass1 = [&](int64_t k, float (&v)[NVAL]) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1)
#pragma unroll
            for (int i = 0; i < NVAL; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < NVAL; ++i) red[parity][i][warp] = v[i];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < NVAL; ++i) {
            float s = 0.f;
#pragma unroll 4
            for (int w = 0; w < W; ++w) s += red[parity][i][w];
            v[i] = s;
        }
        parity ^= 1;
        if constexpr (CL > 1) {
            if (t < CL) {
                const int sp = (int)(k % NS);
                const uint32_t dst = map_to_rank(smem_u32(&slot[sp][rank][0]), (uint32_t)t);
#pragma unroll
                for (int i = 0; i < NVAL; ++i) st_cluster_f32(dst + 4u * i, v[i]);
                mbar_arrive_remote(map_to_rank(smem_u32(&xch[sp]), (uint32_t)t));
            }
        } else {
            cst[k % 3][0] = LN ? v[NVAL - 1] / n : 0.f;
            cst[k % 3][1] = v[0] / n;
        }
    };
    // Row k's exchange: wait for the CL partials, sum them in rank order.
    auto recv = [&](int64_t k) {
        if constexpr (CL > 1) {
            const int sp = (int)(k % NS);
            mbar_wait_cluster_bounded(&xch[sp], (uint32_t)((k / NS) & 1), &abort_flag, p.tc.fault);
            float s[NVAL];
#pragma unroll
            for (int i = 0; i < NVAL; ++i) {
                s[i] = 0.f;
#pragma unroll
                for (int c = 0; c < CL; ++c) s[i] += slot[sp][c][i];
            }
            cst[k % 3][0] = LN ? s[NVAL - 1] / n : 0.f;
            cst[k % 3][1] = s[0] / n;
        }
    };
    auto rstd_of = [&](int64_t k) { return __ldg(p.rstd + row_of(k)); };
    auto mean_of = [&](int64_t k) { return LN ? __ldg(p.mean + row_of(k)) : 0.f; };
    auto dx_of = [&](int64_t k) { return static_cast<uint4 *>(p.dx) + row_of(k) * nv + v0; };

    if (PF == 2) prefetch(0);
    if constexpr (FUSE) {
        for (int64_t j = 0; j < nrows + 2; ++j) {
            const bool has1 = j < nrows, has2 = j >= 2;
            if (PF == 1) prefetch(j);
            if (PF == 2) prefetch(j + 1);
            float v[NVAL];
            const int64_t k1 = has1 ? j : 0, k2 = has2 ? j - 2 : 0;
            const float rstd1 = has1 ? rstd_of(k1) : 0.f, mean1 = has1 ? mean_of(k1) : 0.f;
            const float rstd2 = has2 ? rstd_of(k2) : 0.f, mean2 = has2 ? mean_of(k2) : 0.f;
            const float c1 = cst[k2 % 3][0], c2 = cst[k2 % 3][1];
            if (has1 && has2)
                wide_bwd_sweep<T, LN, NT, U, true, true>(t, cnt, slice, gr, accs, row_x(k1), row_dy(k1),
                                                         mean1, rstd1, v, row_x(k2), row_dy(k2), dx_of(k2),
                                                         mean2, rstd2, c1, c2, keep, drop);
            else if (has1)
                wide_bwd_sweep<T, LN, NT, U, true, false>(t, cnt, slice, gr, accs, row_x(k1), row_dy(k1),
                                                          mean1, rstd1, v, nullptr, nullptr, nullptr, 0.f,
                                                          0.f, 0.f, 0.f, keep, drop);
            else if (has2)
                wide_bwd_sweep<T, LN, NT, U, false, true>(t, cnt, slice, gr, accs, nullptr, nullptr, 0.f,
                                                          0.f, v, row_x(k2), row_dy(k2), dx_of(k2), mean2,
                                                          rstd2, c1, c2, keep, drop);
            if (has1) finish_pass1(j, v);
            if (j >= 1 && j - 1 < nrows) recv(j - 1);
        }
    } else {
        float v[NVAL];
        if (nrows > 0) {
            if (PF == 1) prefetch(0);
            wide_bwd_sweep<T, LN, NT, U, true, false>(t, cnt, slice, gr, accs, row_x(0), row_dy(0),
                                                      mean_of(0), rstd_of(0), v, nullptr, nullptr, nullptr,
                                                      0.f, 0.f, 0.f, 0.f, keep, drop);
            finish_pass1(0, v);
        }
        for (int64_t k = 0; k < nrows; ++k) {
            if (k + 1 < nrows) {
                if (PF == 1) prefetch(k + 1);
                if (PF == 2) prefetch(k + 2);
                wide_bwd_sweep<T, LN, NT, U, true, false>(t, cnt, slice, gr, accs, row_x(k + 1),
                                                          row_dy(k + 1), mean_of(k + 1), rstd_of(k + 1), v,
                                                          nullptr, nullptr, nullptr, 0.f, 0.f, 0.f, 0.f,
                                                          keep, drop);
                finish_pass1(k + 1, v);
            }
            recv(k);
            wide_bwd_sweep<T, LN, NT, U, false, true>(t, cnt, slice, gr, accs, nullptr, nullptr, 0.f, 0.f,
                                                      v, row_x(k), row_dy(k), dx_of(k), mean_of(k),
                                                      rstd_of(k), cst[k % 3][0], cst[k % 3][1], keep, drop);
        }
    }
    // No CTA leaves while a peer could still write into its shared memory
    // (this matters only after an aborted wait).
    if constexpr (CL > 1) cluster_sync_all();

    // This CTA's slice of the cluster's partial row (P = clusters).
    float4 *wsg = reinterpret_cast<float4 *>(p.ws + cid * p.N + v0 * E);
    float4 *wsb = reinterpret_cast<float4 *>(p.ws + (ncl + cid) * p.N + v0 * E);
    for (int vv = t; vv < cnt; vv += NT) {
#pragma unroll
        for (int h = 0; h < H; ++h) {
            wsg[vv * H + h] = accs[h * slice + vv];
            if constexpr (LN) wsb[vv * H + h] = accs[(H + h) * slice + vv];
        }
    }
}

}  // namespace gbn

namespace gbn {

// ============================================================================ backward, register sums
// As bwd_wide (a cluster of CL CTAs per row, CTA `rank` owning a contiguous
// column slice; pass 1 from DRAM, exchange of the row sums through
// distributed shared memory in four slots, pass 2 from L2; pass 1 of row k + 1
// before pass 2 of row k), with the dgamma/dbeta sums in registers instead of
// shared memory: thread t owns vectors t + k * NT (k < K) of the slice, so
// each element's sums cost two FMAs instead of shared-memory read-modify-
// writes, and gamma of the slice is widened once to fp32 in shared memory
// (plane-major float4).  Per element: two conversions, the pass-1 partials
// and, in pass 2, dx and the two sums -- about half the instructions of
// bwd_wide, whose sums live in shared memory.  Loads go in batches of KB
// vectors per tensor (registers: K * E sums per plane plus 2 * KB vectors).
// MINB: CTAs per SM of the launch bound (registers 65536 / (NT * MINB)); two
// CTAs of a cluster on one SM let one CTA's exchange or memory wait overlap
// the other's work.
// FUSE: 1 pass 1 of row j in the same sweep as pass 2 of row j - 2 (both
// rows' loads in flight together); 0 pass 1 of row k + 1, the exchange of row
// k, then pass 2 of row k.
// DB (LayerNorm): 1 the dbeta sums in shared memory (each thread's own fp32
// plane entries, a read-modify-write per vector) and gamma kept there in its
// storage type, which frees K * E registers for a larger K or a second CTA
// per SM; 2 as 1 with gamma read from global memory (L1/L2) per use instead,
// a third less shared memory per CTA (more L1 beside it for the loads in
// flight); 0 both sums in registers, gamma widened to fp32.
template <typename T, bool LN, int NT, int K, int CL, int PF, int MINB, int FUSE, int DB = 0>
__global__ void __launch_bounds__(NT, MINB) bwd_wider(const BwdParams p) {
    pdl_launch_dependents();  // the column reduce waits for this grid's completion
    constexpr int E = VecTraits<T>::E;
    constexpr int H = E / 4;
    constexpr int W = NT / 32;
    constexpr int NVAL = LN ? 2 : 1;
    constexpr int NS = 4;
    constexpr int KB = FUSE ? (K < 2 ? K : 2) : (K < 4 ? K : 4);  // vectors per tensor per batch
    static_assert(NT % 32 == 0 && NT <= 1024 && CL >= 1 && CL <= 16 && K % KB == 0, "shape");
    static_assert(!DB || LN, "dbeta sums only for LayerNorm");
    static_assert((W & (W - 1)) == 0 && (CL & (CL - 1)) == 0, "warps per CTA, CTAs per row: powers of two");
    // gamma of the slice: [H][K * NT] float4 (DB: [K * NT] raw vectors), then
    // (DB) the dbeta sums [H][K * NT] float4
    extern __shared__ __align__(16) float4 gsm[];
    __shared__ float red[2][NVAL][W];
    __shared__ float slot[NS][CL][NVAL];
    __shared__ __align__(8) uint64_t xch[NS];
    __shared__ int abort_flag;

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int rank = CL > 1 ? (int)cluster_ctarank() : 0;
    const int64_t cid = CL > 1 ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
    const int64_t ncl = CL > 1 ? (int64_t)cluster_count_x() : (int64_t)gridDim.x;
    const int64_t M = p.M, nv = p.N / E;
    const int64_t slice = (nv + CL - 1) / CL;
    const int64_t v0 = rank * slice;
    const int64_t cnt = nv - v0 < slice ? (nv - v0 > 0 ? nv - v0 : 0) : slice;
    const float n = (float)p.N;
    const uint64_t keep = l2_policy_keep(), drop = l2_policy_drop();
    constexpr int KNT = K * NT;

    uint4 *graw = reinterpret_cast<uint4 *>(gsm);
    float4 *dbs = gsm + (DB == 1 ? KNT : 0);  // DB: this slice's dbeta sums
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int64_t lv = (int64_t)k * NT + t;
        const uint4 g = lv < cnt ? param_vec<T>(p.gamma, v0 + lv, true) : make_uint4(0, 0, 0, 0);
        if constexpr (DB) {
            if constexpr (DB == 1) graw[lv] = g;
#pragma unroll
            for (int h = 0; h < H; ++h) dbs[h * KNT + lv] = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
#pragma unroll
            for (int h = 0; h < H; ++h)
                gsm[h * KNT + lv] = make_float4(vget<T>(g, 4 * h), vget<T>(g, 4 * h + 1), vget<T>(g, 4 * h + 2),
                                                vget<T>(g, 4 * h + 3));
        }
    }
    if (t == 0) {
        abort_flag = 0;
        if (CL > 1) {
            for (int j = 0; j < NS; ++j) mbar_init(&xch[j], CL);
            fence_mbar_init();
        }
    }
    // every CTA's barriers exist before any peer arrives on them
    if constexpr (CL > 1) cluster_sync_all();
    else __syncthreads();

    // dgamma (and dbeta) sums of this thread's columns, as pairs of elements
    float2 accg[K][E / 2], accb[(LN && !DB) ? K : 1][E / 2];
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
        for (int e = 0; e < E / 2; ++e) {
            accg[k][e] = f2s(0.f);
            if constexpr (LN && !DB) accb[k][e] = f2s(0.f);
        }

    const int64_t nrows = cid < M ? (M - cid + ncl - 1) / ncl : 0;
    auto row_of = [&](int64_t k) { return cid + k * ncl; };
    auto row_x = [&](int64_t k) { return static_cast<const uint4 *>(p.x) + row_of(k) * nv + v0; };
    auto row_dy = [&](int64_t k) { return static_cast<const uint4 *>(p.dy) + row_of(k) * nv + v0; };
    auto prefetch = [&](int64_t k) {
        if (warp == 0 && k < nrows && cnt > 0) {
            prefetch_row(row_x(k), (size_t)cnt * 16, lane, keep);
            prefetch_row(row_dy(k), (size_t)cnt * 16, lane, keep);
        }
    };
    auto gam = [&](int k, float2 (&g)[E / 2]) {
        const int64_t lv = (int64_t)k * NT + t;
        if constexpr (DB == 2) {
            const uint4 q = lv < cnt ? param_vec<T>(p.gamma, v0 + lv, true) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int e = 0; e < E / 2; ++e) g[e] = vpair<T>(q, e);
        } else if constexpr (DB) {
            const uint4 q = graw[lv];
#pragma unroll
            for (int e = 0; e < E / 2; ++e) g[e] = vpair<T>(q, e);
        } else {
#pragma unroll
            for (int h = 0; h < H; ++h) {
                const float4 q = gsm[h * KNT + lv];
                g[2 * h] = make_float2(q.x, q.y);
                g[2 * h + 1] = make_float2(q.z, q.w);
            }
        }
    };
    int parity = 0;
    float cst[3][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};  // (c1, c2) of row k at [k % 3]

    // The CTA's sum of this thread's pass-1 partials (identical bits in every
    // thread), sent to the cluster (or, alone, turned into c1, c2).
    auto finish1 = [&](int64_t kr, float (&v)[NVAL]) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1)
#pragma unroll
            for (int i = 0; i < NVAL; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < NVAL; ++i) red[parity][i][warp] = v[i];
        }
        __syncthreads();
        // every warp runs the same butterfly over the warps' sums (lane l
        // takes warp l % W's): identical bits in every thread
#pragma unroll
        for (int i = 0; i < NVAL; ++i) {
            float s = red[parity][i][lane & (W - 1)];
#pragma unroll
            for (int o = 1; o < W; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            v[i] = s;
        }
        parity ^= 1;
        if constexpr (CL > 1) {
            if (t < CL) {
                const int sp = (int)(kr % NS);
                const uint32_t dst = map_to_rank(smem_u32(&slot[sp][rank][0]), (uint32_t)t);
#pragma unroll
                for (int i = 0; i < NVAL; ++i) st_cluster_f32(dst + 4u * i, v[i]);
                mbar_arrive_remote(map_to_rank(smem_u32(&xch[sp]), (uint32_t)t));
            }
        } else {
            cst[kr % 3][0] = LN ? v[NVAL - 1] / n : 0.f;
            cst[kr % 3][1] = v[0] / n;
        }
    };
    auto recv = [&](int64_t kr) {
        if constexpr (CL > 1) {
            const int sp = (int)(kr % NS);
            mbar_wait_cluster_bounded(&xch[sp], (uint32_t)((kr / NS) & 1), &abort_flag, p.tc.fault);
            // a butterfly over the CL partials (lane l takes rank l % CL's):
            // identical bits in every thread of every CTA
            float s[NVAL];
#pragma unroll
            for (int i = 0; i < NVAL; ++i) {
                s[i] = slot[sp][lane & (CL - 1)][i];
#pragma unroll
                for (int o = 1; o < CL; o <<= 1) s[i] += __shfl_xor_sync(0xffffffffu, s[i], o);
            }
            cst[kr % 3][0] = LN ? s[NVAL - 1] / n : 0.f;
            cst[kr % 3][1] = s[0] / n;
        }
    };
    // One sweep over the slice: pass 1 of row k1 (if has1: this thread's
    // partials into v) and pass 2 of row k2 (if has2: dx and the sums), their
    // loads in the same batches so that both rows' latencies overlap.  The
    // branches are uniform over the CTA.  fullc: every thread holds all K
    // vectors of its share (a literal in each inlined copy of the body).
    auto sweep = [&](bool has1, int64_t k1, bool has2, int64_t k2, float (&v)[NVAL], bool fullc) {
        const float rstd1 = has1 ? __ldg(p.rstd + row_of(k1)) : 0.f;
        const float mean1 = (LN && has1) ? __ldg(p.mean + row_of(k1)) : 0.f;
        const float rstd2 = has2 ? __ldg(p.rstd + row_of(k2)) : 0.f;
        const float mean2 = (LN && has2) ? __ldg(p.mean + row_of(k2)) : 0.f;
        const float rc1 = rstd2 * cst[k2 % 3][0], rc2 = rstd2 * cst[k2 % 3][1];
        // the row constants as pairs (negations are exact: x + (-m) = x - m)
        const float2 nm1 = f2s(-mean1), nm2 = f2s(-mean2), r2 = f2s(rstd2), nrc1 = f2s(-rc1), nrc2 = f2s(-rc2);
        const uint4 *x1 = row_x(has1 ? k1 : 0), *d1 = row_dy(has1 ? k1 : 0);
        const uint4 *x2 = row_x(has2 ? k2 : 0), *d2 = row_dy(has2 ? k2 : 0);
        uint4 *dx2 = static_cast<uint4 *>(p.dx) + row_of(has2 ? k2 : 0) * nv + v0;
        // pass-1 partials: lane 0 the even elements, lane 1 the odd ones
        float2 a2 = f2s(0.f), a1 = f2s(0.f);
#pragma unroll
        for (int kb = 0; kb < K; kb += KB) {
            uint4 px[KB], pd[KB], qx[KB], qd[KB];
#pragma unroll
            for (int i = 0; i < KB; ++i) {
                const int64_t lv = (int64_t)(kb + i) * NT + t;
                const bool ok = fullc || lv < cnt;
                px[i] = (has1 && ok) ? ld_l2hint(x1 + lv, keep) : make_uint4(0, 0, 0, 0);
                pd[i] = (has1 && ok) ? ld_l2hint(d1 + lv, keep) : make_uint4(0, 0, 0, 0);
                qx[i] = (has2 && ok) ? ld_l2hint(x2 + lv, drop) : make_uint4(0, 0, 0, 0);
                qd[i] = (has2 && ok) ? ld_l2hint(d2 + lv, drop) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int i = 0; i < KB; ++i) {
                const int64_t lv = (int64_t)(kb + i) * NT + t;
                float2 g[E / 2];
                gam(kb + i, g);
                if (has2) {
                    float2 o[E / 2];
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) {
                        const float2 xh = f2mul(f2add(vpair<T>(qx[i], e), nm2), r2);
                        const float2 dyv = vpair<T>(qd[i], e);
                        // dx = rstd g - rstd c1 - (rstd c2) xhat
                        o[e] = f2fma(nrc2, xh, f2fma(r2, f2mul(dyv, g[e]), nrc1));
                        accg[kb + i][e] = f2fma(dyv, xh, accg[kb + i][e]);  // zero past the slice (dy = 0)
                        if constexpr (LN && !DB) accb[kb + i][e] = f2add(accb[kb + i][e], dyv);
                    }
                    if constexpr (DB) {
                        // this thread's own dbeta entries: no other thread touches them
#pragma unroll
                        for (int h = 0; h < H; ++h) {
                            float4 &b4 = dbs[h * KNT + lv];
                            const float2 lo = f2add(make_float2(b4.x, b4.y), vpair<T>(qd[i], 2 * h));
                            const float2 hi = f2add(make_float2(b4.z, b4.w), vpair<T>(qd[i], 2 * h + 1));
                            b4 = make_float4(lo.x, lo.y, hi.x, hi.y);
                        }
                    }
                    if (fullc || lv < cnt) st_l2hint(dx2 + lv, vpack2<T>(o), drop);
                }
                if (has1) {
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) {
                        const float2 gg = f2mul(vpair<T>(pd[i], e), g[e]);  // zero past the slice
                        a2 = f2fma(gg, f2add(vpair<T>(px[i], e), nm1), a2);
                        if constexpr (LN) a1 = f2add(a1, gg);
                    }
                }
            }
        }
        v[0] = (a2.x + a2.y) * rstd1;  // sum g xhat = rstd sum g (x - mean)
        if constexpr (LN) v[NVAL - 1] = a1.x + a1.y;
    };

    // the body once per case, so that with every vector of the share present
    // the bound checks drop out of the compiled loops
    auto run = [&](bool fullc) {
        float v[NVAL];
        if constexpr (FUSE) {
            // step j: pass 1 of row j with pass 2 of row j - 2, then row j's
            // partials go out and row j - 1's come in (a whole sweep after they
            // were sent)
            if (PF == 2) prefetch(0);
            for (int64_t j = 0; j < nrows + 2; ++j) {
                const bool has1 = j < nrows, has2 = j >= 2;
                if (PF >= 1) prefetch(j + (PF == 2 ? 1 : 0));
                sweep(has1, j, has2, j - 2, v, fullc);
                if (has1) finish1(j, v);
                if (j >= 1 && j - 1 < nrows) recv(j - 1);
            }
        } else {
            // pass 1 of row k + 1, then row k's exchange, then pass 2 of row k
            if (PF == 2) prefetch(0);
            if (nrows > 0) {
                if (PF == 1) prefetch(0);
                sweep(true, 0, false, 0, v, fullc);
                finish1(0, v);
            }
            for (int64_t kr = 0; kr < nrows; ++kr) {
                if (kr + 1 < nrows) {
                    if (PF == 1) prefetch(kr + 1);
                    if (PF == 2) prefetch(kr + 2);
                    sweep(true, kr + 1, false, 0, v, fullc);
                    finish1(kr + 1, v);
                }
                recv(kr);
                sweep(false, 0, true, kr, v, fullc);
            }
        }
    };
    if (cnt == (int64_t)KNT) run(true);
    else run(false);
    // no CTA leaves while a peer could still write into its shared memory
    if constexpr (CL > 1) cluster_sync_all();

    // this CTA's slice of the cluster's partial row (P = clusters)
    float *wsg = p.ws + cid * p.N + v0 * E;
    float *wsb = p.ws + (ncl + cid) * p.N + v0 * E;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int64_t lv = (int64_t)k * NT + t;
        if (lv >= cnt) continue;
#pragma unroll
        for (int h = 0; h < H; ++h) {
            reinterpret_cast<float4 *>(wsg + lv * E)[h] =
                make_float4(accg[k][2 * h].x, accg[k][2 * h].y, accg[k][2 * h + 1].x, accg[k][2 * h + 1].y);
            if constexpr (LN && DB)
                reinterpret_cast<float4 *>(wsb + lv * E)[h] = dbs[h * KNT + lv];
            else if constexpr (LN)
                reinterpret_cast<float4 *>(wsb + lv * E)[h] =
                    make_float4(accb[k][2 * h].x, accb[k][2 * h].y, accb[k][2 * h + 1].x, accb[k][2 * h + 1].y);
        }
    }
}

}  // namespace gbn

namespace gbn {

// ============================================================================ forward, cluster slices
// Wide-row forward on the layout of bwd_wider: a cluster of CL CTAs shares
// each row, CTA `rank` always owns the same column slice, so gamma (and
// beta) of the slice sit in its shared memory for the whole call (in their
// storage type) and pass 2 re-reads only x from L2 -- fwd_wide re-reads x,
// gamma and beta per row, three L2 loads per vector.  Per row: pass 1
// streams the slice from DRAM (L2 evict_last) for this thread's statistics
// (RMS: the sum of squares; LN: count, mean and M2 per batch of KB vectors,
// merged with the update of Chan, Golub and LeVeque), the CTA combines them
// (every warp runs the same butterfly over the warps' partials) and sends
// them to every CTA of the cluster through distributed shared memory (four
// slots); the row's exchange is collected (a butterfly over the CL partials
// in rank positions: identical bits in every CTA) a whole sweep later, then
// pass 2 writes y from the slice re-read from L2 (evict_first).
// Thread t owns vectors t + k * NT (k < K) of the slice.
// FUSE: 0 pass 1 of row k + 1, the exchange of row k, then pass 2 of row k;
// 1 pass 1 of row j in the same sweep as pass 2 of row j - 2 (both rows'
// loads in flight together, KB = 4 vectors of each per batch); 2 one pass:
// the slice stays in registers from its DRAM read to its y (no L2 re-read),
// two rows per thread, the next row's loads issued before this row's
// statistics.  In every mode the four exchange slots are safe to reuse: a
// peer sends row k + 4 only after it has received this CTA's row k + 2,
// which this CTA sends after the CTA barrier in its statistics step, and
// that barrier follows its reads of row k's slot.
template <typename T, bool LN, int NT, int K, int CL, int PF, int MINB, int FUSE = 0>
__global__ void __launch_bounds__(NT, MINB) fwd_wider(const FwdParams p) {
    constexpr int E = VecTraits<T>::E;
    constexpr int W = NT / 32;
    constexpr int NVAL = LN ? 3 : 1;  // exchanged: (count, mean, M2) or the sum of squares
    constexpr int NS = 4;
    // vectors per batch: the whole of a thread's slice up to 8, 4 when fused
    constexpr int KB = FUSE == 1 ? (K < 4 ? K : 4) : (K < 8 ? K : 8);
    static_assert(NT % 32 == 0 && NT <= 1024 && CL >= 1 && CL <= 16 && K % KB == 0, "shape");
    static_assert(((KB * E) & (KB * E - 1)) == 0, "a whole batch holds a power-of-two count");
    static_assert((W & (W - 1)) == 0 && (CL & (CL - 1)) == 0, "warps per CTA, CTAs per row: powers of two");
    extern __shared__ __align__(16) uint4 psm[];  // gamma of the slice [K * NT], then beta
    __shared__ float red[2][3][W];
    __shared__ float slot[NS][CL][NVAL];
    __shared__ __align__(8) uint64_t xch[NS];
    __shared__ int abort_flag;

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int rank = CL > 1 ? (int)cluster_ctarank() : 0;
    const int64_t cid = CL > 1 ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
    const int64_t ncl = CL > 1 ? (int64_t)cluster_count_x() : (int64_t)gridDim.x;
    const int64_t M = p.M, nv = p.N / E;
    const int64_t slice = (nv + CL - 1) / CL;
    const int64_t v0 = rank * slice;
    const int64_t cnt = nv - v0 < slice ? (nv - v0 > 0 ? nv - v0 : 0) : slice;
    const float n = (float)p.N;
    const uint64_t keep = l2_policy_keep(), drop = l2_policy_drop();
    constexpr int KNT = K * NT;

#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int64_t lv = (int64_t)k * NT + t;
        psm[lv] = lv < cnt ? param_vec<T>(p.gamma, v0 + lv, true) : make_uint4(0, 0, 0, 0);
        if constexpr (LN) psm[KNT + lv] = lv < cnt ? param_vec<T>(p.beta, v0 + lv, false) : make_uint4(0, 0, 0, 0);
    }
    if (t == 0) {
        abort_flag = 0;
        if (CL > 1) {
            for (int j = 0; j < NS; ++j) mbar_init(&xch[j], CL);
            fence_mbar_init();
        }
    }
    // every CTA's barriers exist before any peer arrives on them
    if constexpr (CL > 1) cluster_sync_all();
    else __syncthreads();

    const int64_t nrows = cid < M ? (M - cid + ncl - 1) / ncl : 0;
    auto row_of = [&](int64_t k) { return cid + k * ncl; };
    auto row_x = [&](int64_t k) { return static_cast<const uint4 *>(p.x) + row_of(k) * nv + v0; };
    auto prefetch = [&](int64_t k) {
        if (warp == 0 && k < nrows && cnt > 0) prefetch_row(row_x(k), (size_t)cnt * 16, lane, keep);
    };
    int parity = 0;
    float cst[3][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};  // (mean, rstd) of row k at [k % 3]

    // The CTA's statistics of row k from this thread's (identical bits in
    // every thread), sent to the cluster (or, alone, turned into mean, rstd).
    // v: RMS {sum x^2}; LN {count, mean, M2}.
    auto finish1 = [&](int64_t k, float (&v)[NVAL]) {
        // The warps' partials are combined by every warp at once: lane l
        // takes warp l % W's, then a butterfly over W lanes (identical bits
        // in every lane of every warp).
        const int wl = lane & (W - 1);
        if constexpr (!LN) {
            float acc = v[0];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) red[parity][0][warp] = acc;
            __syncthreads();
            acc = red[parity][0][wl];
#pragma unroll
            for (int o = 1; o < W; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            v[0] = acc;
        } else {
            warp_combine(v[0], v[1], v[2]);
            if (lane == 0) {
                red[parity][0][warp] = v[0];
                red[parity][1][warp] = v[1];
                red[parity][2][warp] = v[2];
            }
            __syncthreads();
            v[0] = red[parity][0][wl];
            v[1] = red[parity][1][wl];
            v[2] = red[parity][2][wl];
            warp_combine<W>(v[0], v[1], v[2]);
        }
        parity ^= 1;
        if constexpr (CL > 1) {
            if (t < CL) {
                const int sp = (int)(k % NS);
                const uint32_t dst = map_to_rank(smem_u32(&slot[sp][rank][0]), (uint32_t)t);
#pragma unroll
                for (int i = 0; i < NVAL; ++i) st_cluster_f32(dst + 4u * i, v[i]);
                mbar_arrive_remote(map_to_rank(smem_u32(&xch[sp]), (uint32_t)t));
            }
        } else {
            cst[k % 3][0] = LN ? v[1] : 0.f;
            cst[k % 3][1] = rsqrtf((LN ? v[2] : v[0]) / n + p.eps);
        }
    };
    // The exchange of row k: CL partials combined in rank order.
    auto recv = [&](int64_t k) {
        if constexpr (CL > 1) {
            const int sp = (int)(k % NS);
            mbar_wait_cluster_bounded(&xch[sp], (uint32_t)((k / NS) & 1), &abort_flag, p.tc.fault);
            // lane l takes rank l % CL's partial, then a butterfly over CL
            // lanes: identical bits in every thread of every CTA
            const int cl = lane & (CL - 1);
            if constexpr (!LN) {
                float s = slot[sp][cl][0];
#pragma unroll
                for (int o = 1; o < CL; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                cst[k % 3][0] = 0.f;
                cst[k % 3][1] = rsqrtf(s / n + p.eps);
            } else {
                float tn = slot[sp][cl][0], mu = slot[sp][cl][1], a2 = slot[sp][cl][2];
                warp_combine<CL>(tn, mu, a2);
                cst[k % 3][0] = mu;
                cst[k % 3][1] = rsqrtf(a2 / n + p.eps);
            }
        }
    };
    // One accumulation chain per pair position of a vector (E / 2 chains),
    // summed pairwise at the end of the batch.
    auto chains = [&](float2 (&c)[E / 2]) {
#pragma unroll
        for (int w = 1; w < E / 2; w <<= 1)
#pragma unroll
            for (int e = 0; e + w < E / 2; e += 2 * w) c[e] = f2add(c[e], c[e + w]);
        return c[0];
    };
    // This thread's statistics of KB vectors q (vectors kb .. kb + KB - 1 of
    // its share) folded into the running RMS sum of squares a, or the LN
    // running count, mean and M2.  fullc: every thread holds all K vectors
    // of its share (no per-vector bound checks; a literal in each inlined
    // copy of the body below).
    auto stat_batch = [&](const uint4 (&q)[KB], int kb, float2 &a, float &cn, float &mean, float &m2, bool fullc) {
        const bool FULL = fullc;
        if constexpr (!LN) {
            float2 c[E / 2];
#pragma unroll
            for (int e = 0; e < E / 2; ++e) c[e] = f2s(0.f);
#pragma unroll
            for (int i = 0; i < KB; ++i)
#pragma unroll
                for (int e = 0; e < E / 2; ++e) {
                    const float2 f = vpair<T>(q[i], e);
                    c[e] = f2fma(f, f, c[e]);
                }
            a = f2add(a, chains(c));
        } else {
            int nb = 0;
            float2 c[E / 2];
#pragma unroll
            for (int e = 0; e < E / 2; ++e) c[e] = f2s(0.f);
#pragma unroll
            for (int i = 0; i < KB; ++i) {
                if (FULL || (int64_t)(kb + i) * NT + t < cnt) nb += E;
#pragma unroll
                for (int e = 0; e < E / 2; ++e) c[e] = f2add(c[e], vpair<T>(q[i], e));
            }
            if (nb > 0) {
                const float fb = (float)nb;
                const float2 s2 = chains(c);
                // a whole batch holds a power-of-two count: the product by its
                // reciprocal is the correctly rounded quotient
                const float mb = nb == KB * E ? (s2.x + s2.y) * (1.f / (float)(KB * E)) : __fdiv_rn(s2.x + s2.y, fb);
                const float2 nmb = f2s(-mb);
#pragma unroll
                for (int e = 0; e < E / 2; ++e) c[e] = f2s(0.f);
#pragma unroll
                for (int i = 0; i < KB; ++i) {
                    if (!FULL && (int64_t)(kb + i) * NT + t >= cnt) continue;
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) {
                        const float2 d = f2add(vpair<T>(q[i], e), nmb);
                        c[e] = f2fma(d, d, c[e]);
                    }
                }
                const float2 d2 = chains(c);
                const float m2b = d2.x + d2.y;
                if (cn == 0.f) {
                    cn = fb;
                    mean = mb;
                    m2 = m2b;
                } else {
                    // running += batch
                    const float tot = cn + fb;
                    const float d = mb - mean;
                    const float rr = __fdiv_rn(fb, tot);
                    mean += d * rr;
                    m2 += m2b + d * d * cn * rr;
                    cn = tot;
                }
            }
        }
    };
    auto stat_out = [&](const float2 &a, float cn, float mean, float m2, float (&v)[NVAL]) {
        if constexpr (!LN) {
            v[0] = a.x + a.y;
        } else {
            v[0] = cn;
            v[1] = mean;
            v[2] = m2;
        }
    };
    // The row's (mean and) rstd, stored by one thread of rank 0.
    auto put_stats = [&](int64_t k, float mean2, float rstd2) {
        if (rank == 0 && t == 0) {
            const int64_t row = row_of(k);
            if (p.rstd) p.rstd[row] = rstd2;
            if (LN && p.mean) p.mean[row] = mean2;
        }
    };
    // y of vector lv of the slice from its x (q).
    auto out_vec = [&](const uint4 &q, int64_t lv, uint4 *yr, float2 nm, float2 rs) {
        const uint4 g = psm[lv];
        uint4 b = make_uint4(0, 0, 0, 0);
        if constexpr (LN) b = psm[KNT + lv];
        float2 o[E / 2];
#pragma unroll
        for (int e = 0; e < E / 2; ++e) {
            const float2 xh = f2mul(f2add(vpair<T>(q, e), nm), rs);
            // LN: xhat * gamma + beta in one rounding
            o[e] = LN ? f2fma(xh, vpair<T>(g, e), vpair<T>(b, e)) : f2mul(xh, vpair<T>(g, e));
        }
        st_l2hint(yr + lv, vpack2<T>(o), drop);
    };
    // One sweep over the slice: pass 1 of row k1 (if has1: this thread's
    // statistics into v) and pass 2 of row k2 (if has2: y), their loads in
    // the same batches.  Branches uniform over the CTA.
    auto sweep = [&](bool has1, int64_t k1, bool has2, int64_t k2, float (&v)[NVAL], bool fullc) {
        const bool FULL = fullc;
        const uint4 *x1 = row_x(has1 ? k1 : 0), *x2 = row_x(has2 ? k2 : 0);
        const float mean2 = cst[(has2 ? k2 : 0) % 3][0], rstd2 = cst[(has2 ? k2 : 0) % 3][1];
        const float2 nm = f2s(-mean2), rs = f2s(rstd2);
        if (has2) put_stats(k2, mean2, rstd2);
        uint4 *yr = static_cast<uint4 *>(p.y) + row_of(has2 ? k2 : 0) * nv + v0;
        float2 a = f2s(0.f);                 // RMS: sum of squares
        float cn = 0.f, mean = 0.f, m2 = 0.f;  // LN: running count, mean, M2
#pragma unroll
        for (int kb = 0; kb < K; kb += KB) {
            uint4 q1[KB], q2[KB];
#pragma unroll
            for (int i = 0; i < KB; ++i) {
                const int64_t lv = (int64_t)(kb + i) * NT + t;
                const bool ok = FULL || lv < cnt;
                q1[i] = (has1 && ok) ? ld_l2hint(x1 + lv, keep) : make_uint4(0, 0, 0, 0);
                q2[i] = (has2 && ok) ? ld_l2hint(x2 + lv, drop) : make_uint4(0, 0, 0, 0);
            }
            if (has2) {
#pragma unroll
                for (int i = 0; i < KB; ++i) {
                    const int64_t lv = (int64_t)(kb + i) * NT + t;
                    if (FULL || lv < cnt) out_vec(q2[i], lv, yr, nm, rs);
                }
            }
            if (has1) stat_batch(q1, kb, a, cn, mean, m2, fullc);
        }
        stat_out(a, cn, mean, m2, v);
    };
    // Register-resident rows (FUSE 2): the slice of row k, read once from
    // DRAM, stays in this thread's registers (q) until its y is written.
    auto load_r = [&](int64_t k, uint4 (&q)[K], bool fullc) {
        const bool FULL = fullc;
        const bool has = k < nrows;
        const uint4 *xr = row_x(has ? k : 0);
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const int64_t lv = (int64_t)i * NT + t;
            q[i] = (has && (FULL || lv < cnt)) ? ld_l2hint(xr + lv, drop) : make_uint4(0, 0, 0, 0);
        }
    };
    auto stats_r = [&](const uint4 (&q)[K], float (&v)[NVAL], bool fullc) {
        float2 a = f2s(0.f);
        float cn = 0.f, mean = 0.f, m2 = 0.f;
#pragma unroll
        for (int kb = 0; kb < K; kb += KB) {
            uint4 qb[KB];
#pragma unroll
            for (int i = 0; i < KB; ++i) qb[i] = q[kb + i];
            stat_batch(qb, kb, a, cn, mean, m2, fullc);
        }
        stat_out(a, cn, mean, m2, v);
    };
    auto write_r = [&](int64_t k, const uint4 (&q)[K], bool fullc) {
        const bool FULL = fullc;
        const float mean2 = cst[k % 3][0], rstd2 = cst[k % 3][1];
        put_stats(k, mean2, rstd2);
        uint4 *yr = static_cast<uint4 *>(p.y) + row_of(k) * nv + v0;
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const int64_t lv = (int64_t)i * NT + t;
            if (FULL || lv < cnt) out_vec(q[i], lv, yr, f2s(-mean2), f2s(rstd2));
        }
    };

    // Every thread holds all K vectors of its share (uniform over the CTA):
    // the body is inlined once per case, so with fullc true the bound checks
    // drop out of the compiled loops.
    auto run = [&](bool fullc) {
        float v[NVAL];
        if constexpr (FUSE == 2) {
            // row k + 1's loads go out before row k's statistics, so they are in
            // flight through row k's reduction, exchange and y
            uint4 qa[K], qb[K];
            load_r(0, qa, fullc);
            for (int64_t k = 0; k < nrows; k += 2) {
                load_r(k + 1, qb, fullc);
                stats_r(qa, v, fullc);
                finish1(k, v);
                recv(k);
                write_r(k, qa, fullc);
                if (k + 1 < nrows) {
                    load_r(k + 2, qa, fullc);
                    stats_r(qb, v, fullc);
                    finish1(k + 1, v);
                    recv(k + 1);
                    write_r(k + 1, qb, fullc);
                }
            }
        } else if constexpr (FUSE) {

            // step j: pass 1 of row j with pass 2 of row j - 2, then row j's
            // statistics go out and row j - 1's come in (a whole sweep after
            // they were sent)
            for (int64_t j = 0; j < nrows + 2; ++j) {
                const bool has1 = j < nrows, has2 = j >= 2;
                if (PF >= 1) prefetch(j + 1);
                sweep(has1, j, has2, j - 2, v, fullc);
                if (has1) finish1(j, v);
                if (j >= 1 && j - 1 < nrows) recv(j - 1);
            }
        } else {
            // pass 1 of row k + 1, then row k's exchange, then pass 2 of row k
            if (PF >= 1) prefetch(0);
            if (nrows > 0) {
                sweep(true, 0, false, 0, v, fullc);
                finish1(0, v);
            }
            for (int64_t kr = 0; kr < nrows; ++kr) {
                if (kr + 1 < nrows) {
                    if (PF >= 1) prefetch(kr + 1);
                    sweep(true, kr + 1, false, 0, v, fullc);
                    finish1(kr + 1, v);
                }
                recv(kr);
                sweep(false, 0, true, kr, v, fullc);
            }
        }
    };
    if (cnt == (int64_t)KNT) run(true);
    else run(false);
    // no CTA leaves while a peer could still write into its shared memory
    if constexpr (CL > 1) cluster_sync_all();
}

}  // namespace gbn
