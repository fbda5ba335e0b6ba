// ex_kernels.cuh -- RMSNorm / LayerNorm forward and backward for the general
// form of the call: rows with their own strides, a storage type per tensor
// (rows x, parameters gamma / beta, output y), and an optional residual add
// fused in front of the norm.
//
// Same arithmetic as norm_kernels.cuh (the definitions on "SOTA
// normalization performance with torch.compile", section "How Did
// Torch.compile Catch Quack?", and "Fused RMSNorm", sections "What it is" /
// "How it works": fp16/bf16 storage, fp32 accumulation, one rounding per
// output).  The fusion follows the torch.compile page's paragraphs on
// Inductor fusing a norm with its neighbouring operations: the residual sum
// h = x + r is formed in fp32, rounded once to the storage type of x and r,
// stored if asked for, and normalised -- the values an unfused h = x + r
// followed by the norm would give, with one read of x and r instead of a
// write and a re-read of h.  Backward: dx = rstd (g - c1 - xhat c2) + dres,
// where dres is the gradient reaching h from the residual stream; dx is the
// gradient of both x and r.
//
// Storage types are runtime arguments: every load and store of a row goes
// through ld8 / st8 (eight elements: one 16-byte vector of 16-bit values, two
// of fp32), whose branch on the type is uniform over the grid, so one kernel
// serves every combination of types.  Rows are held in fp32 registers by row
// groups of TPR threads (thread t owns 8-element chunks k * TPR + t), gamma
// (and beta) are widened once per CTA into shared memory (plane-major float4,
// conflict-free), the grid is persistent and the backward keeps its
// dgamma/dbeta partials in registers, one partial row per CTA, summed by the
// column-reduce kernel.  fwd_exr / bwd_exr: the same row groups fed through
// a shared-memory ring by bulk asynchronous copies (one copy per row, or one
// per tile when the rows are dense), for rows whose 16-byte vectors allow it.
// fwd_exe / bwd_exe: one CTA per row, element by element, for any N, stride
// and alignment.
#pragma once

#include "device_common.cuh"
#include "params.h"
#include "tma_kernels.cuh"

namespace gbn {

// Storage type codes (gbnorm_dtype_t).
constexpr int kF32 = 0, kF16 = 1, kBF16 = 2;

// 16-byte load through the coherent path: an output of these kernels may
// overwrite the row it was computed from (in place), so rows are not read as
// read-only data.
__device__ __forceinline__ uint4 ld_row_vec(const void *base, int64_t idx) {
    return reinterpret_cast<const uint4 *>(base)[idx];
}

// Eight consecutive elements of a row starting at element `off` (a multiple
// of 8; the row 16-byte aligned), widened to fp32.
__device__ __forceinline__ void ld8(const void *row, int64_t off, int dt, float (&f)[8]) {
    if (dt == kF32) {
        const uint4 a = ld_row_vec(row, off / 4), b = ld_row_vec(row, off / 4 + 1);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[e] = vget<float>(a, e);
            f[4 + e] = vget<float>(b, e);
        }
    } else {
        const uint4 a = ld_row_vec(row, off / 8);
        if (dt == kBF16) {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = vget<__nv_bfloat16>(a, e);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = vget<__half>(a, e);
        }
    }
}
__device__ __forceinline__ void st8(void *row, int64_t off, int dt, const float (&f)[8]) {
    if (dt == kF32) {
        st_vec(row, off / 4, vpack<float>(f));
        st_vec(row, off / 4 + 1, vpack<float>(f + 4));
    } else if (dt == kBF16) {
        st_vec(row, off / 8, vpack<__nv_bfloat16>(f));
    } else {
        st_vec(row, off / 8, vpack<__half>(f));
    }
}
// One element, any alignment.
__device__ __forceinline__ float ld1(const void *row, int64_t j, int dt) {
    if (dt == kF32) return static_cast<const float *>(row)[j];
    if (dt == kBF16) return to_f(static_cast<const __nv_bfloat16 *>(row)[j]);
    return to_f(static_cast<const __half *>(row)[j]);
}
__device__ __forceinline__ void st1(void *row, int64_t j, int dt, float v) {
    if (dt == kF32) static_cast<float *>(row)[j] = v;
    else if (dt == kBF16) static_cast<__nv_bfloat16 *>(row)[j] = from_f<__nv_bfloat16>(v);
    else static_cast<__half *>(row)[j] = from_f<__half>(v);
}
// v rounded to storage type dt (round to nearest even) and widened back.
__device__ __forceinline__ float round_to(float v, int dt) {
    if (dt == kBF16) return __bfloat162float(__float2bfloat16_rn(v));
    if (dt == kF16) return __half2float(__float2half_rn(v));
    return v;
}
__device__ __forceinline__ int esize(int dt) { return dt == kF32 ? 4 : 2; }
__device__ __forceinline__ const void *row_ptr(const void *base, int64_t row, int64_t ld, int dt) {
    return static_cast<const unsigned char *>(base) + row * ld * esize(dt);
}
__device__ __forceinline__ void *row_ptr(void *base, int64_t row, int64_t ld, int dt) {
    return static_cast<unsigned char *>(base) + row * ld * esize(dt);
}

// gamma (and beta) of the whole row, widened to fp32 into shared memory as
// two planes of float4 per parameter: chunk c's elements 0-3 at [c], 4-7 at
// [nc + c].  A null parameter row is the constant 1 (gamma) or 0 (beta).
template <bool LN, int CTA>
__device__ __forceinline__ void ex_load_params(float4 *pars, const void *gamma, const void *beta, int pdt,
                                               int64_t nc) {
    for (int64_t c = threadIdx.x; c < nc; c += CTA) {
        float g[8], b[8];
        if (gamma) {
            ld8(gamma, 8 * c, pdt, g);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) g[e] = 1.f;
        }
        pars[c] = make_float4(g[0], g[1], g[2], g[3]);
        pars[nc + c] = make_float4(g[4], g[5], g[6], g[7]);
        if constexpr (LN) {
            if (beta) {
                ld8(beta, 8 * c, pdt, b);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) b[e] = 0.f;
            }
            pars[2 * nc + c] = make_float4(b[0], b[1], b[2], b[3]);
            pars[3 * nc + c] = make_float4(b[4], b[5], b[6], b[7]);
        }
    }
}
__device__ __forceinline__ void ex_par8(const float4 *plane, int64_t nc, int64_t c, float (&f)[8]) {
    const float4 a = plane[c], b = plane[nc + c];
    f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w;
    f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
}

// ============================================================================ forward
template <bool LN, int TPR, int VPT, int CTA, int MINB>
__global__ void __launch_bounds__(CTA, MINB) fwd_ex(const ExFwdParams p) {
    static_assert(CTA % TPR == 0 && TPR % 32 == 0, "row-group shape");
    constexpr int RPC = CTA / TPR;
    extern __shared__ __align__(16) float4 pars[];  // gamma planes, then beta planes
    __shared__ RowReduceSmem<TPR, RPC, 1, 2> red2;
    __shared__ RowReduceSmem<TPR, RPC, 1, 1> red1;
    const int64_t nc = p.N / 8;
    const int t = threadIdx.x % TPR, grp = threadIdx.x / TPR;
    const float n = (float)p.N;
    const bool full = nc == (int64_t)TPR * VPT;  // every thread holds VPT chunks (uniform)
    ex_load_params<LN, CTA>(pars, p.gamma, p.beta, p.pdt, nc);
    __syncthreads();
    int parity = 0;
    for (int64_t base = (int64_t)blockIdx.x * RPC; base < p.M; base += (int64_t)gridDim.x * RPC) {
        const int64_t row = base + grp;
        const bool rok = row < p.M;
        const int64_t rr = rok ? row : base;
        float xf[VPT][8];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int64_t c = (int64_t)k * TPR + t;
            if (rok && c < nc) {
                ld8(row_ptr(p.x, rr, p.ldx, p.xdt), 8 * c, p.xdt, xf[k]);
                if (p.res) {
                    // h = x + r in fp32, rounded once to the storage type
                    float r8[8];
                    ld8(row_ptr(p.res, rr, p.ldr, p.xdt), 8 * c, p.xdt, r8);
#pragma unroll
                    for (int e = 0; e < 8; ++e) xf[k][e] = round_to(xf[k][e] + r8[e], p.xdt);
                    if (p.h) st8(row_ptr(p.h, rr, p.ldh, p.xdt), 8 * c, p.xdt, xf[k]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) xf[k][e] = 0.f;
            }
        }
        float sa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e) sa[e & 3] += LN ? xf[k][e] : xf[k][e] * xf[k][e];
        const float s = (sa[0] + sa[1]) + (sa[2] + sa[3]);
        float mean = 0.f, rstd;
        if (LN && full) {
            // equal per-thread counts: local mean and M2, one exact combine
            constexpr float kC = (float)(VPT * 8);
            float mm[1] = {s * (1.f / kC)}, m2[1];
            float qa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < VPT; ++k)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float d = xf[k][e] - mm[0];
                    qa[e & 3] += d * d;
                }
            m2[0] = (qa[0] + qa[1]) + (qa[2] + qa[3]);
            row_meanvar_equal<TPR, RPC, 1>(mm, m2, kC, red2, parity);
            mean = mm[0];
            rstd = rsqrtf(m2[0] / n + p.eps);
        } else {
            float a[1] = {s};
            row_allreduce<TPR, RPC, 1, 1>(a, red1, parity);
            if constexpr (LN) {
                // mean first, then the centred sum of squares from the registers
                mean = a[0] / n;
                a[0] = 0.f;
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    if ((int64_t)k * TPR + t >= nc) continue;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float d = xf[k][e] - mean;
                        a[0] += d * d;
                    }
                }
                row_allreduce<TPR, RPC, 1, 1>(a, red1, parity);
            }
            rstd = rsqrtf(a[0] / n + p.eps);
        }
        if (!rok) continue;  // uniform per row group; no collective below
        if (t == 0) {
            if (p.rstd) p.rstd[row] = rstd;
            if (LN && p.mean) p.mean[row] = mean;
        }
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int64_t c = (int64_t)k * TPR + t;
            if (c >= nc) continue;
            float g[8], o[8];
            ex_par8(pars, nc, c, g);
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = ((xf[k][e] - mean) * rstd) * g[e];
            if constexpr (LN) {
                float b[8];
                ex_par8(pars + 2 * nc, nc, c, b);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] += b[e];
            }
            st8(row_ptr(p.y, row, p.ldy, p.ydt), 8 * c, p.ydt, o);
        }
    }
}

// ============================================================================ backward
template <bool LN, int TPR, int VPT, int CTA, int MINB>
__global__ void __launch_bounds__(CTA, MINB) bwd_ex(const ExBwdParams p) {
    static_assert(CTA % TPR == 0 && TPR % 32 == 0, "row-group shape");
    pdl_launch_dependents();  // the column reduce waits for this grid's completion
    constexpr int RPC = CTA / TPR;
    constexpr int NS = LN ? 2 : 1;
    extern __shared__ __align__(16) float4 pars[];  // gamma planes; later the row groups' partials
    __shared__ RowReduceSmem<TPR, RPC, 1, NS> red;
    const int64_t nc = p.N / 8;
    const int t = threadIdx.x % TPR, grp = threadIdx.x / TPR;
    const float n = (float)p.N;
    ex_load_params<false, CTA>(pars, p.gamma, nullptr, p.pdt, nc);
    __syncthreads();
    float accg[VPT][8], accb[LN ? VPT : 1][8];
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            accg[k][e] = 0.f;
            if constexpr (LN) accb[k][e] = 0.f;
        }
    int parity = 0;
    for (int64_t base = (int64_t)blockIdx.x * RPC; base < p.M; base += (int64_t)gridDim.x * RPC) {
        const int64_t row = base + grp;
        const bool rok = row < p.M;
        const int64_t rr = rok ? row : base;
        const float rstd = rok ? __ldg(p.rstd + row) : 0.f;
        const float mean = (LN && rok) ? __ldg(p.mean + row) : 0.f;
        // x - mean and dy of this thread's chunks (zeros outside the row)
        float xc[VPT][8], dyv[VPT][8];
        float sum[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i) sum[i] = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int64_t c = (int64_t)k * TPR + t;
            if (rok && c < nc) {
                ld8(row_ptr(p.x, rr, p.ldx, p.xdt), 8 * c, p.xdt, xc[k]);
                ld8(row_ptr(p.dy, rr, p.lddy, p.ydt), 8 * c, p.ydt, dyv[k]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) xc[k][e] = dyv[k][e] = 0.f;
            }
            float g8[8];
            ex_par8(pars, nc, c < nc ? c : 0, g8);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                xc[k][e] -= mean;
                const float gg = dyv[k][e] * g8[e];
                sum[0] += gg * xc[k][e];
                if constexpr (LN) sum[NS - 1] += gg;
            }
        }
        // masked slots hold dy = 0 and contribute nothing
        row_allreduce<TPR, RPC, 1, NS>(sum, red, parity);
        if (!rok) continue;  // uniform per row group; no collective below
        // dx = rstd g - rstd c1 - (rstd c2) xhat (+ dres), c2 = rstd sum g (x - mean) / n
        const float c2 = rstd * sum[0] / n;
        const float rc1 = LN ? rstd * (sum[NS - 1] / n) : 0.f;
        const float rc2 = rstd * c2;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int64_t c = (int64_t)k * TPR + t;
            if (c >= nc) continue;
            float g8[8], o[8];
            ex_par8(pars, nc, c, g8);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float xh = xc[k][e] * rstd;
                o[e] = fmaf(-rc2, xh, fmaf(rstd, dyv[k][e] * g8[e], -rc1));
                accg[k][e] += dyv[k][e] * xh;
                if constexpr (LN) accb[k][e] += dyv[k][e];
            }
            if (p.dres) {
                float r8[8];
                ld8(row_ptr(p.dres, row, p.lddres, p.xdt), 8 * c, p.xdt, r8);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] += r8[e];
            }
            st8(row_ptr(p.dx, row, p.lddx, p.xdt), 8 * c, p.xdt, o);
        }
    }
    // Epilogue: one partial row per CTA; the row groups (same columns) are
    // added in group order through shared memory (the parameters are no
    // longer needed).
    float *wsg = p.ws + (int64_t)blockIdx.x * p.N;
    float *wsb = p.ws + ((int64_t)gridDim.x + blockIdx.x) * p.N;
    float *comb = reinterpret_cast<float *>(pars);  // [NS][N]
    __syncthreads();
    for (int gi = 0; gi < RPC; ++gi) {
        if (grp == gi) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int64_t c = (int64_t)k * TPR + t;
                if (c >= nc) continue;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int64_t j = 8 * c + e;
                    comb[j] = gi == 0 ? accg[k][e] : comb[j] + accg[k][e];
                    if constexpr (LN) comb[p.N + j] = gi == 0 ? accb[k][e] : comb[p.N + j] + accb[k][e];
                }
            }
        }
        __syncthreads();
    }
    for (int64_t j = threadIdx.x; j < p.N; j += CTA) {
        wsg[j] = comb[j];
        if constexpr (LN) wsb[j] = comb[p.N + j];
    }
}

// ============================================================================ element-wise (any N, stride, alignment)
template <bool LN>
__global__ void __launch_bounds__(kElemCTA) fwd_exe(const ExFwdParams p) {
    __shared__ float red[2 * 1 * (kElemCTA / 32)];
    const float n = (float)p.N;
    int parity = 0;
    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
        const void *xr = row_ptr(p.x, row, p.ldx, p.xdt);
        const void *rr = p.res ? row_ptr(p.res, row, p.ldr, p.xdt) : nullptr;
        void *hr = p.h ? row_ptr(p.h, row, p.ldh, p.xdt) : nullptr;
        // the (rounded) residual sum of an element; once stored (pass 1) it is
        // read back, which stays right when h overwrites x or r in place
        // (each thread reads back only the elements it wrote)
        auto hsum = [&](int64_t j) {
            const float v = ld1(xr, j, p.xdt);
            return rr ? round_to(v + ld1(rr, j, p.xdt), p.xdt) : v;
        };
        auto hval = [&](int64_t j) { return hr ? ld1(hr, j, p.xdt) : hsum(j); };
        float s[1] = {0.f};
        for (int64_t j = threadIdx.x; j < p.N; j += kElemCTA) {
            const float f = hsum(j);
            if (hr) st1(hr, j, p.xdt, f);
            s[0] += LN ? f : f * f;
        }
        cta_allreduce<kElemCTA, 1>(s, red, parity);
        float mean = 0.f;
        if constexpr (LN) {
            mean = s[0] / n;
            s[0] = 0.f;
            for (int64_t j = threadIdx.x; j < p.N; j += kElemCTA) {
                const float d = hval(j) - mean;
                s[0] += d * d;
            }
            cta_allreduce<kElemCTA, 1>(s, red, parity);
        }
        const float rstd = rsqrtf(s[0] / n + p.eps);
        if (threadIdx.x == 0) {
            if (p.rstd) p.rstd[row] = rstd;
            if (LN && p.mean) p.mean[row] = mean;
        }
        void *yr = row_ptr(p.y, row, p.ldy, p.ydt);
        for (int64_t j = threadIdx.x; j < p.N; j += kElemCTA) {
            float o = ((hval(j) - mean) * rstd) * (p.gamma ? ld1(p.gamma, j, p.pdt) : 1.f);
            if (LN && p.beta) o += ld1(p.beta, j, p.pdt);
            st1(yr, j, p.ydt, o);
        }
    }
}

// Each CTA accumulates its partial dgamma/dbeta row in its own workspace row.
template <bool LN>
__global__ void __launch_bounds__(kElemCTA) bwd_exe(const ExBwdParams p) {
    pdl_launch_dependents();
    __shared__ float red[2 * 2 * (kElemCTA / 32)];
    const float n = (float)p.N;
    const int64_t P = gridDim.x;
    float *wsg = p.ws + (int64_t)blockIdx.x * p.N;
    float *wsb = p.ws + (P + blockIdx.x) * p.N;
    for (int64_t j = threadIdx.x; j < p.N; j += kElemCTA) {
        wsg[j] = 0.f;
        if constexpr (LN) wsb[j] = 0.f;
    }
    auto gam = [&](int64_t j) { return p.gamma ? ld1(p.gamma, j, p.pdt) : 1.f; };
    int parity = 0;
    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
        const void *xr = row_ptr(p.x, row, p.ldx, p.xdt);
        const void *dyr = row_ptr(p.dy, row, p.lddy, p.ydt);
        const float rstd = __ldg(p.rstd + row);
        const float mean = LN ? __ldg(p.mean + row) : 0.f;
        float s[2] = {0.f, 0.f};
        for (int64_t j = threadIdx.x; j < p.N; j += kElemCTA) {
            const float xh = (ld1(xr, j, p.xdt) - mean) * rstd;
            const float g = ld1(dyr, j, p.ydt) * gam(j);
            s[0] += g * xh;
            s[1] += g;
        }
        cta_allreduce<kElemCTA, 2>(s, red, parity);
        const float c2 = s[0] / n;
        const float c1 = LN ? s[1] / n : 0.f;
        void *dxr = row_ptr(p.dx, row, p.lddx, p.xdt);
        const void *drr = p.dres ? row_ptr(p.dres, row, p.lddres, p.xdt) : nullptr;
        for (int64_t j = threadIdx.x; j < p.N; j += kElemCTA) {
            const float xh = (ld1(xr, j, p.xdt) - mean) * rstd;
            const float dyv = ld1(dyr, j, p.ydt);
            float o = rstd * (dyv * gam(j) - c1 - xh * c2);
            if (drr) o += ld1(drr, j, p.xdt);
            st1(dxr, j, p.xdt, o);
            wsg[j] += dyv * xh;
            if constexpr (LN) wsb[j] += dyv;
        }
    }
}

// ============================================================================ ring kernels
// Rows are brought into a shared-memory ring by cp.async.bulk: a tile of RT
// rows per stage, every row tensor of the tile in its own section of the
// stage (rows packed at N * element-size bytes, each section 128-byte
// aligned).  As in fwd_tmp / bwd_tmp, the CTA's NT threads form RPP = NT / TPR
// row groups; group g walks the CTA's tiles g, g + RPP, ... through its own
// SG = stages / RPP stages, and its first thread refills the stage of tile
// j - 1 right after the group barrier of tile j's first row reduction (every
// thread of the group has read tile j - 1 by then).  gamma (and beta) are
// bulk-copied once per CTA in their storage type and widened on use; the
// saved statistics of a backward tile come in with the tile (stat_window).

struct ExRingHeader {
    uint64_t full[kExRingMaxStages];
    uint64_t pbar;  // gamma (and beta) landed
    int abort;
    int pad;
    float red[(kTmaHeaderBytes - 8 * kExRingMaxStages - 16) / 4];  // row-group scratch
};
static_assert(sizeof(ExRingHeader) == kTmaHeaderBytes, "header layout");

// Eight elements (8-element chunk c) of a row staged in shared memory in
// storage type dt, widened to fp32.
__device__ __forceinline__ void lds8(const unsigned char *row, int64_t c, int dt, float (&f)[8]) {
    if (dt == kF32) {
        const uint4 a = lds128(row + 32 * c), b = lds128(row + 32 * c + 16);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[e] = vget<float>(a, e);
            f[4 + e] = vget<float>(b, e);
        }
    } else {
        const uint4 a = lds128(row + 16 * c);
        if (dt == kBF16) {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = vget<__nv_bfloat16>(a, e);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = vget<__half>(a, e);
        }
    }
}
// A parameter chunk from shared memory, or the constant a null row stands for.
__device__ __forceinline__ void par8(const unsigned char *row, bool present, int64_t c, int dt, float one,
                                     float (&f)[8]) {
    if (present) {
        lds8(row, c, dt, f);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = one;
    }
}

// The same chunk as four pairs (elements 2i, 2i + 1) for the two-lane fp32
// operations.
__device__ __forceinline__ void lds8p(const unsigned char *row, int64_t c, int dt, float2 (&f)[4]) {
    if (dt == kF32) {
        const uint4 a = lds128(row + 32 * c), b = lds128(row + 32 * c + 16);
        f[0] = vpair<float>(a, 0);
        f[1] = vpair<float>(a, 1);
        f[2] = vpair<float>(b, 0);
        f[3] = vpair<float>(b, 1);
    } else {
        const uint4 a = lds128(row + 16 * c);
        if (dt == kBF16) {
#pragma unroll
            for (int i = 0; i < 4; ++i) f[i] = vpair<__nv_bfloat16>(a, i);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) f[i] = vpair<__half>(a, i);
        }
    }
}
__device__ __forceinline__ void par8p(const unsigned char *row, bool present, int64_t c, int dt, float one,
                                      float2 (&f)[4]) {
    if (present) {
        lds8p(row, c, dt, f);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) f[i] = f2s(one);
    }
}
// Parameter chunk c as pairs: from fp32 planes (element 0-3 at [c], 4-7 at
// [nc + c]; conflict-free, nothing to convert) or from the raw row.
__device__ __forceinline__ void parp(bool planes, const float4 *pl, const unsigned char *raw, bool present,
                                     int64_t nc, int64_t c, int dt, float one, float2 (&f)[4]) {
    if (planes) {
        const float4 a = pl[c], b = pl[nc + c];
        f[0] = make_float2(a.x, a.y);
        f[1] = make_float2(a.z, a.w);
        f[2] = make_float2(b.x, b.y);
        f[3] = make_float2(b.z, b.w);
    } else {
        par8p(raw, present, c, dt, one, f);
    }
}
__device__ __forceinline__ void st8p(void *row, int64_t off, int dt, const float2 (&f)[4]) {
    const float o[8] = {f[0].x, f[0].y, f[1].x, f[1].y, f[2].x, f[2].y, f[3].x, f[3].y};
    st8(row, off, dt, o);
}

// Rows [r0, r0 + rows) of a row tensor (row stride ld elements, row_bytes =
// N * element size) into dst, packed at row_bytes: one copy when the rows are
// dense, else one per row.  Every source row starts on a 16-byte boundary
// (aligned base and row stride) and row_bytes is a multiple of 16.
__device__ __forceinline__ void ex_copy_rows(unsigned char *dst, const void *base, int64_t ld, int es,
                                             int64_t r0, int rows, size_t row_bytes, uint64_t *bar) {
    const unsigned char *src = static_cast<const unsigned char *>(base) + r0 * ld * es;
    const size_t pitch = (size_t)ld * (size_t)es;
    if (pitch == row_bytes) {
        bulk_g2s(dst, src, (uint32_t)(rows * row_bytes), bar);
    } else {
        for (int r = 0; r < rows; ++r) bulk_g2s(dst + r * row_bytes, src + r * pitch, (uint32_t)row_bytes, bar);
    }
}

// Waits (bounded, regardless of the abort flag) for the copies a group leader
// issued into its stages, so that none is still landing when the CTA exits.
__device__ __forceinline__ void exr_drain(ExRingHeader &h, int grp, int SG, int issued) {
    int zero = 0;
    for (int j = issued > SG ? issued - SG : 0; j < issued; ++j)
        mbar_wait_bounded(&h.full[grp * SG + j % SG], (uint32_t)((j / SG) & 1),
                          reinterpret_cast<volatile int *>(&zero), nullptr);
}

// XT: the storage type of x (and of y, dy, h, dres, dx) fixed at compile
// time (kF32 / kF16 / kBF16), which folds every conversion branch; -1 reads
// the types from the call (any combination).
template <bool LN, int TPR, int VPT, int NT, int XT = -1>
__global__ void __launch_bounds__(NT, 1) fwd_exr(const ExFwdParams p) {
    constexpr int RPP = NT / TPR;
    constexpr int WPR = TPR / 32;
    static_assert(NT % TPR == 0 && TPR % 32 == 0 && TPR > 32 && 2 * RPP <= kExRingMaxStages, "CTA shape");
    static_assert(RPP * 2 * 2 * WPR <= (int)(sizeof(ExRingHeader::red) / 4), "scratch");
    extern __shared__ __align__(128) unsigned char smem[];
    ExRingHeader &h = *reinterpret_cast<ExRingHeader *>(smem);
    const int xdt = XT >= 0 ? XT : p.xdt, ydt = XT >= 0 ? XT : p.ydt;
    const int64_t M = p.M, nc = p.N / 8;
    const int xes = esize(xdt);
    const size_t xrb = (size_t)p.N * xes;
    const bool planes = p.planes != 0;
    unsigned char *gsm = smem + kTmaHeaderBytes;  // gamma, then beta
    unsigned char *bsm = gsm + exr_param_bytes(p.N, p.pdt, false, planes);
    unsigned char *stages = smem + kTmaHeaderBytes + exr_param_bytes(p.N, p.pdt, LN, planes);
    const float4 *gpl = reinterpret_cast<const float4 *>(gsm);  // planes: gamma, then beta at + 2 * nc
    const int SG = p.tc.stages / RPP, RT = p.tc.rows;
    const size_t xsec = exr_section(RT, p.N, xdt);
    const int64_t ntiles = (M + RT - 1) / RT;
    const int t = threadIdx.x % TPR, grp = threadIdx.x / TPR;
    float *scratch = h.red + grp * (2 * 2 * WPR);
    volatile int *abort_flag = &h.abort;
    int issued = 0;

    auto tile_of = [&](int64_t j) {
        const int64_t tile = blockIdx.x + (grp + j * RPP) * (int64_t)gridDim.x;
        return tile < ntiles ? tile : (int64_t)-1;
    };
    auto issue = [&](int64_t j) {
        const int64_t tile = tile_of(j);
        if (tile < 0) return;
        const int s = grp * SG + (int)(j % SG);
        const int64_t r0 = tile * RT;
        const int rows = (int)(M - r0 < RT ? M - r0 : RT);
        unsigned char *dst = stages + (size_t)s * p.tc.stride;
        mbar_arrive_expect_tx(&h.full[s], (uint32_t)(rows * xrb) * (p.res ? 2u : 1u));
        ex_copy_rows(dst, p.x, p.ldx, xes, r0, rows, xrb, &h.full[s]);
        if (p.res) ex_copy_rows(dst + xsec, p.res, p.ldr, xes, r0, rows, xrb, &h.full[s]);
        ++issued;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < RPP * SG; ++s) mbar_init(&h.full[s], 1);
        mbar_init(&h.pbar, 1);
        h.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !planes)
        load_params(&h.pbar, gsm, bsm, p.gamma, LN ? p.beta : nullptr,
                    (uint32_t)((size_t)p.N * esize(p.pdt)));
    if (t == 0)
        for (int j = 0; j < SG; ++j) issue(j);
    if (planes) {
        // gamma (beta) planes: [0, 2 nc) then, for LayerNorm, [2 nc, 4 nc)
        ex_load_params<LN, NT>(reinterpret_cast<float4 *>(gsm), p.gamma, p.beta, p.pdt, nc);
        __syncthreads();
    } else {
        mbar_wait_bounded(&h.pbar, 0, abort_flag, p.tc.fault);
    }

    const float n = (float)p.N;
    const bool full = nc == (int64_t)TPR * VPT;  // every thread holds VPT chunks (uniform)
    const bool has_g = p.gamma != nullptr, has_b = LN && p.beta != nullptr;
    int parity = 0;
    for (int64_t j = 0;; ++j) {
        const int64_t tile = tile_of(j);
        if (tile < 0) break;  // uniform per group (named barriers only)
        const int s = grp * SG + (int)(j % SG);
        mbar_wait_bounded(&h.full[s], (uint32_t)((j / SG) & 1), abort_flag, p.tc.fault);
        const int64_t r0 = tile * RT;
        const int rows = (int)(M - r0 < RT ? M - r0 : RT);
        const unsigned char *tb = stages + (size_t)s * p.tc.stride;
        for (int r = 0; r < rows; ++r) {  // every thread of the group works on the same row
            const int64_t row = r0 + r;
            const unsigned char *xs = tb + (size_t)r * xrb;
            float2 xf[VPT][4];
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int64_t c = (int64_t)k * TPR + t;
                if (c < nc) {
                    lds8p(xs, c, xdt, xf[k]);
                    if (p.res) {
                        // h = x + r in fp32, rounded once to the storage type
                        float2 r8[4];
                        lds8p(xs + xsec, c, xdt, r8);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 hs = f2add(xf[k][e], r8[e]);
                            xf[k][e] = make_float2(round_to(hs.x, xdt), round_to(hs.y, xdt));
                        }
                        if (p.h) st8p(row_ptr(p.h, row, p.ldh, xdt), 8 * c, xdt, xf[k]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) xf[k][e] = f2s(0.f);
                }
            }
            float2 a2 = f2s(0.f);
#pragma unroll
            for (int k = 0; k < VPT; ++k)
#pragma unroll
                for (int e = 0; e < 4; ++e) a2 = LN ? f2add(a2, xf[k][e]) : f2fma(xf[k][e], xf[k][e], a2);
            float acc = a2.x + a2.y;
            float mean = 0.f;
            if (LN && full) {
                constexpr float kC = (float)(VPT * 8);
                mean = acc * (1.f / kC);
                const float2 nm = f2s(-mean);
                float2 q2 = f2s(0.f);
#pragma unroll
                for (int k = 0; k < VPT; ++k)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 d = f2add(xf[k][e], nm);
                        q2 = f2fma(d, d, q2);
                    }
                float m2 = q2.x + q2.y;
                group_meanvar_equal<TPR>(mean, m2, kC, scratch, parity, 1 + grp);
                acc = m2;
            } else {
                float a[1] = {acc};
                group_allreduce<TPR, 1>(a, scratch, parity, 1 + grp);
                acc = a[0];
                if constexpr (LN) {
                    mean = acc / n;
                    const float2 nm = f2s(-mean);
                    float2 q2 = f2s(0.f);
#pragma unroll
                    for (int k = 0; k < VPT; ++k) {
                        if ((int64_t)k * TPR + t >= nc) continue;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 d = f2add(xf[k][e], nm);
                            q2 = f2fma(d, d, q2);
                        }
                    }
                    a[0] = q2.x + q2.y;
                    group_allreduce<TPR, 1>(a, scratch, parity, 1 + grp);
                    acc = a[0];
                }
            }
            if (r == 0 && j >= 1 && t == 0) {
                // every thread of the group is past its last read of tile
                // j - 1's stage: order those reads before the copy's writes
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(j - 1 + SG);
            }
            const float rstd = rsqrtf(acc / n + p.eps);
            if (t == 0) {
                if (p.rstd) p.rstd[row] = rstd;
                if (LN && p.mean) p.mean[row] = mean;
            }
            const float2 nm = f2s(-mean), rs = f2s(rstd);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int64_t c = (int64_t)k * TPR + t;
                if (c >= nc) continue;
                float2 g[4], o[4];
                parp(planes, gpl, gsm, has_g, nc, c, p.pdt, 1.f, g);
#pragma unroll
                for (int e = 0; e < 4; ++e) o[e] = f2mul(f2mul(f2add(xf[k][e], nm), rs), g[e]);
                if constexpr (LN) {
                    float2 b[4];
                    parp(planes, gpl + 2 * nc, bsm, has_b, nc, c, p.pdt, 0.f, b);
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[e] = f2add(o[e], b[e]);
                }
                st8p(row_ptr(p.y, row, p.ldy, ydt), 8 * c, ydt, o);
            }
        }
    }
    if (t == 0 && *abort_flag) exr_drain(h, grp, SG, issued);
}

template <bool LN, int TPR, int VPT, int NT, int XT = -1>
__global__ void __launch_bounds__(NT, 1) bwd_exr(const ExBwdParams p) {
    pdl_launch_dependents();  // the column reduce waits for this grid's completion
    constexpr int NS = LN ? 2 : 1;
    constexpr int RPP = NT / TPR;
    constexpr int WPR = TPR / 32;
    // pass-1 values kept in registers for pass 2 where the dgamma/dbeta sums
    // leave room for them (LayerNorm: two chunks only with one row group per
    // CTA, whose scratch addressing is simplest; otherwise they spill)
    constexpr bool HOLD = LN ? (VPT == 1 || (VPT == 2 && TPR == NT)) : VPT <= 2;
    static_assert(NT % TPR == 0 && TPR % 32 == 0 && TPR > 32 && 2 * RPP <= kExRingMaxStages, "CTA shape");
    static_assert(RPP * 2 * NS * WPR <= (int)(sizeof(ExRingHeader::red) / 4), "scratch");
    extern __shared__ __align__(128) unsigned char smem[];
    ExRingHeader &h = *reinterpret_cast<ExRingHeader *>(smem);
    const int xdt = XT >= 0 ? XT : p.xdt, ydt = XT >= 0 ? XT : p.ydt;
    const int64_t M = p.M, nc = p.N / 8;
    const int xes = esize(xdt), yes = esize(ydt);
    const size_t xrb = (size_t)p.N * xes, yrb = (size_t)p.N * yes;
    const bool planes = p.planes != 0;
    unsigned char *gsm = smem + kTmaHeaderBytes;  // gamma: fp32 planes, or its storage type
    unsigned char *stages = smem + kTmaHeaderBytes + exr_param_bytes(p.N, p.pdt, false, planes);
    const float4 *gpl = reinterpret_cast<const float4 *>(gsm);
    const int SG = p.tc.stages / RPP, RT = p.tc.rows;
    // stage: x | dy | dres (if any) | rstd, mean windows
    const size_t xsec = exr_section(RT, p.N, xdt), ysec = exr_section(RT, p.N, ydt);
    const size_t rsec = p.dres ? xsec : 0;
    const int64_t ntiles = (M + RT - 1) / RT;
    const int t = threadIdx.x % TPR, grp = threadIdx.x / TPR;
    float *scratch = h.red + grp * (2 * NS * WPR);
    volatile int *abort_flag = &h.abort;
    int issued = 0;

    auto tile_of = [&](int64_t j) {
        const int64_t tile = blockIdx.x + (grp + j * RPP) * (int64_t)gridDim.x;
        return tile < ntiles ? tile : (int64_t)-1;
    };
    auto issue = [&](int64_t j) {
        const int64_t tile = tile_of(j);
        if (tile < 0) return;
        const int s = grp * SG + (int)(j % SG);
        const int64_t r0 = tile * RT;
        const int rows = (int)(M - r0 < RT ? M - r0 : RT);
        unsigned char *dst = stages + (size_t)s * p.tc.stride;
        int64_t wa, wb;
        stat_window(r0, rows, M, &wa, &wb);
        const uint32_t tx = (uint32_t)(rows * xrb) * (p.dres ? 2u : 1u) + (uint32_t)(rows * yrb) +
                            (uint32_t)(wb - wa) * 4u * (LN ? 2u : 1u);
        mbar_arrive_expect_tx(&h.full[s], tx);
        ex_copy_rows(dst, p.x, p.ldx, xes, r0, rows, xrb, &h.full[s]);
        ex_copy_rows(dst + xsec, p.dy, p.lddy, yes, r0, rows, yrb, &h.full[s]);
        if (p.dres) ex_copy_rows(dst + xsec + ysec, p.dres, p.lddres, xes, r0, rows, xrb, &h.full[s]);
        if (wb > wa) {
            float *sd = reinterpret_cast<float *>(dst + xsec + ysec + rsec);
            bulk_g2s(sd, p.rstd + wa, (uint32_t)(wb - wa) * 4u, &h.full[s]);
            if constexpr (LN) bulk_g2s(sd + exr_stat_floats(RT), p.mean + wa, (uint32_t)(wb - wa) * 4u, &h.full[s]);
        }
        ++issued;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < RPP * SG; ++s) mbar_init(&h.full[s], 1);
        mbar_init(&h.pbar, 1);
        h.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !planes)
        load_params(&h.pbar, gsm, nullptr, p.gamma, nullptr, (uint32_t)((size_t)p.N * esize(p.pdt)));
    if (t == 0)
        for (int j = 0; j < SG; ++j) issue(j);
    if (planes) {
        ex_load_params<false, NT>(reinterpret_cast<float4 *>(gsm), p.gamma, nullptr, p.pdt, nc);
        __syncthreads();
    } else {
        mbar_wait_bounded(&h.pbar, 0, abort_flag, p.tc.fault);
    }

    const float n = (float)p.N;
    const bool has_g = p.gamma != nullptr;
    // dgamma (and dbeta) sums of this thread's columns, as pairs
    float2 accg[VPT][4], accb[LN ? VPT : 1][4];
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            accg[k][e] = f2s(0.f);
            if constexpr (LN) accb[k][e] = f2s(0.f);
        }
    int parity = 0;
    // Trip count uniform over the CTA (the epilogue's barriers); groups past
    // their last tile leave the loop early.
    const int64_t my_tiles = blockIdx.x < ntiles ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    for (int64_t j = 0; j < (my_tiles + RPP - 1) / RPP; ++j) {
        const int64_t tile = tile_of(j);
        if (tile < 0) break;  // uniform per group (named barriers only below)
        const int s = grp * SG + (int)(j % SG);
        mbar_wait_bounded(&h.full[s], (uint32_t)((j / SG) & 1), abort_flag, p.tc.fault);
        const int64_t r0 = tile * RT;
        const int rows = (int)(M - r0 < RT ? M - r0 : RT);
        int64_t wa, wb;
        stat_window(r0, rows, M, &wa, &wb);
        const unsigned char *tb = stages + (size_t)s * p.tc.stride;
        const float *st = reinterpret_cast<const float *>(tb + xsec + ysec + rsec) - wa;
        for (int r = 0; r < rows; ++r) {  // every thread of the group works on the same row
            const int64_t row = r0 + r;
            const unsigned char *xs = tb + (size_t)r * xrb;
            const unsigned char *ds = tb + xsec + (size_t)r * yrb;
            const bool in_win = row < wb;
            const float rstd = in_win ? st[row] : __ldg(p.rstd + row);
            const float mean = LN ? (in_win ? st[exr_stat_floats(RT) + row] : __ldg(p.mean + row)) : 0.f;
            const float2 nm = f2s(-mean);
            float2 s2 = f2s(0.f), s1 = f2s(0.f);
            float2 hx[HOLD ? VPT : 1][4], hg[HOLD ? VPT : 1][4], hd[HOLD ? VPT : 1][4];
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int64_t c = (int64_t)k * TPR + t;
                float2 x8[4], d8[4], g8[4];
                if (c < nc) {
                    lds8p(xs, c, xdt, x8);
                    lds8p(ds, c, ydt, d8);
                    parp(planes, gpl, gsm, has_g, nc, c, p.pdt, 1.f, g8);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) x8[e] = d8[e] = g8[e] = f2s(0.f);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 xc = f2add(x8[e], nm);
                    const float2 gg = f2mul(d8[e], g8[e]);
                    if constexpr (HOLD) {
                        hx[k][e] = xc;
                        hg[k][e] = gg;
                        hd[k][e] = d8[e];
                    }
                    s2 = f2fma(gg, xc, s2);
                    if constexpr (LN) s1 = f2add(s1, gg);
                }
            }
            float sum[NS];
            sum[0] = s2.x + s2.y;
            if constexpr (LN) sum[NS - 1] = s1.x + s1.y;
            group_allreduce<TPR, NS>(sum, scratch, parity, 1 + grp);
            if (r == 0 && j >= 1 && t == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(j - 1 + SG);
            }
            // dx = rstd g - rstd c1 - (rstd c2) xhat (+ dres), c2 = rstd sum g (x - mean) / n
            const float c2 = rstd * sum[0] / n;
            const float rc1 = LN ? rstd * (sum[NS - 1] / n) : 0.f;
            const float rc2 = rstd * c2;
            const float2 r2 = f2s(rstd), nrc1 = f2s(-rc1), nrc2 = f2s(-rc2);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int64_t c = (int64_t)k * TPR + t;
                if (c >= nc) continue;
                float2 xc[4], gg[4], dv[4], o[4];
                if constexpr (HOLD) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        xc[e] = hx[k][e];
                        gg[e] = hg[k][e];
                        dv[e] = hd[k][e];
                    }
                } else {
                    float2 x8[4], g8[4];
                    lds8p(xs, c, xdt, x8);
                    lds8p(ds, c, ydt, dv);
                    parp(planes, gpl, gsm, has_g, nc, c, p.pdt, 1.f, g8);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        xc[e] = f2add(x8[e], nm);
                        gg[e] = f2mul(dv[e], g8[e]);
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 xh = f2mul(xc[e], r2);
                    o[e] = f2fma(nrc2, xh, f2fma(r2, gg[e], nrc1));
                    accg[k][e] = f2fma(dv[e], xh, accg[k][e]);
                    if constexpr (LN) accb[k][e] = f2add(accb[k][e], dv[e]);
                }
                if (p.dres) {
                    float2 r8[4];
                    lds8p(tb + xsec + ysec + (size_t)r * xrb, c, xdt, r8);
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[e] = f2add(o[e], r8[e]);
                }
                st8p(row_ptr(p.dx, row, p.lddx, xdt), 8 * c, xdt, o);
            }
        }
    }
    if (t == 0 && *abort_flag) exr_drain(h, grp, SG, issued);

    // Epilogue: this CTA's partial row.  With several row groups (same
    // columns), every group writes its partials to the idle ring, then each
    // thread adds, for its columns, the groups' values in group order.
    float *wsg = p.ws + (int64_t)blockIdx.x * p.N;
    float *wsb = p.ws + ((int64_t)gridDim.x + blockIdx.x) * p.N;
    if constexpr (RPP > 1) {
        constexpr int CAP = TPR * VPT * 8;
        float *comb = reinterpret_cast<float *>(stages);  // [NS][RPP][CAP]
        __syncthreads();  // every group is done with the ring
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = (k * TPR + t) * 8 + 2 * e;
                comb[grp * CAP + c] = accg[k][e].x;
                comb[grp * CAP + c + 1] = accg[k][e].y;
                if constexpr (LN) {
                    comb[(RPP + grp) * CAP + c] = accb[k][e].x;
                    comb[(RPP + grp) * CAP + c + 1] = accb[k][e].y;
                }
            }
        __syncthreads();
        const int64_t ncol = p.N < CAP ? p.N : CAP;
        for (int c = threadIdx.x; c < ncol; c += NT) {
            float sg = 0.f, sb = 0.f;
#pragma unroll
            for (int gi = 0; gi < RPP; ++gi) {
                sg += comb[gi * CAP + c];
                if constexpr (LN) sb += comb[(RPP + gi) * CAP + c];
            }
            wsg[c] = sg;
            if constexpr (LN) wsb[c] = sb;
        }
    } else {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int64_t c = (int64_t)k * TPR + t;
            if (c >= nc) continue;
            float4 *g4 = reinterpret_cast<float4 *>(wsg + 8 * c);
            float4 *b4 = reinterpret_cast<float4 *>(wsb + 8 * c);
            g4[0] = make_float4(accg[k][0].x, accg[k][0].y, accg[k][1].x, accg[k][1].y);
            g4[1] = make_float4(accg[k][2].x, accg[k][2].y, accg[k][3].x, accg[k][3].y);
            if constexpr (LN) {
                b4[0] = make_float4(accb[k][0].x, accb[k][0].y, accb[k][1].x, accb[k][1].y);
                b4[1] = make_float4(accb[k][2].x, accb[k][2].y, accb[k][3].x, accb[k][3].y);
            }
        }
    }
}

}  // namespace gbn
