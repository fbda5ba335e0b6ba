// tma_kernels.cuh -- RMSNorm / LayerNorm forward and backward with rows staged
// through a shared-memory ring by bulk asynchronous copies (TMA engine).
//
// Same arithmetic as the row-resident kernels in norm_kernels.cuh (the
// definitions on "SOTA normalization performance with torch.compile", section
// "How Did Torch.compile Catch Quack?", and "Fused RMSNorm", sections "What it
// is" / "How it works" / "What didn't work"); what differs is how bytes reach
// the SM.  Rows of one tensor are contiguous, so a tile of consecutive rows is
// one contiguous block: one cp.async.bulk per tensor per tile, no tensor map.
//
// CTA layout: CW consumer warps + 1 producer warp, one CTA per SM, persistent.
// The producer's lane 0 keeps up to `stages` tiles in flight; each tile lands
// in its stage and completes that stage's "full" mbarrier (transaction bytes).
// Consumers split the tile's rows over row groups of TPR threads, read their
// slice of each row from shared memory once, reduce, and write y (or dx) with
// 16-byte stores straight to global memory; one lane per consumer warp then
// arrives on the stage's "empty" mbarrier so the producer may refill it.
// The backward also streams dy and the saved statistics, keeps per-thread
// dgamma/dbeta partials in registers (each thread owns fixed columns) and
// writes one partial row per CTA into the workspace.
//
// Every mbarrier wait is bounded (mbar_wait_bounded): on a timeout the CTA
// raises its abort flag and the device fault word, skips all further waits and
// runs to completion, and the producer waits (bounded) for its copies still in
// flight before the CTA exits.
#pragma once

#include "device_common.cuh"
#include "params.h"

namespace gbn {

constexpr int kTmaBarAll = 15;         // named barrier over all consumer threads

struct TmaHeader {
    uint64_t full[kTmaMaxStages];
    uint64_t empty[kTmaMaxStages];
    uint64_t pbar;  // gamma (and beta) landed in shared memory
    int abort;
    int pad;
    float red[(kTmaHeaderBytes - 16 * kTmaMaxStages - 16) / 4];  // row-group scratch
};
static_assert(sizeof(TmaHeader) == kTmaHeaderBytes, "header layout");

// The saved statistics (rstd, mean) of a tile's rows [r0, r0 + rows) come in
// by bulk copy in 16-byte units: the window [wa, wb) is the tile's rows
// widened to multiples of 4 and clipped to the last multiple of 4 <= M, so it
// never reads past the arrays (16-byte-aligned bases).  Rows of the tile
// outside the window (only in the last < 4 rows of the matrix) are loaded
// directly by the consumers.
__host__ __device__ __forceinline__ void stat_window(int64_t r0, int rows, int64_t M, int64_t *wa,
                                                     int64_t *wb) {
    const int64_t a = r0 & ~(int64_t)3;
    int64_t b = (r0 + rows + 3) & ~(int64_t)3;
    const int64_t lim = M & ~(int64_t)3;
    if (b > lim) b = lim;
    *wa = a;
    *wb = b > a ? b : a;
}
// Floats reserved per statistic per stage: the widest window of a tile of RT rows.
__host__ __device__ constexpr int stat_stride(int RT) { return (RT + 7) & ~3; }

// Producer: lane 0 of the last warp.  `ntensors` row tensors per tile (x, or
// x and dy), plus the saved statistics for the backward.
template <bool BWD, bool LN>
__device__ __forceinline__ void tma_produce(TmaHeader &h, unsigned char *stages, const TileCfg &tc,
                                            int64_t M, size_t row_bytes, const void *t0,
                                            const void *t1, const float *st0, const float *st1,
                                            uint32_t tile_bytes) {
    const int S = tc.stages, RT = tc.rows;
    const int64_t ntiles = (M + RT - 1) / RT;
    volatile int *abort_flag = &h.abort;
    int issued = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++issued) {
        const int s = issued % S;
        if (issued >= S) mbar_wait_bounded(&h.empty[s], ((issued / S) - 1) & 1, abort_flag, tc.fault);
        if (*abort_flag) break;
        const int64_t r0 = tile * RT;
        const int rows = (int)(M - r0 < RT ? M - r0 : RT);
        const uint32_t bytes = (uint32_t)(rows * row_bytes);
        unsigned char *dst = stages + (size_t)s * tc.stride;
        uint32_t tx = bytes;
        int64_t wa = 0, wb = 0;
        if constexpr (BWD) {
            tx += bytes;
            stat_window(r0, rows, M, &wa, &wb);
            tx += (uint32_t)(wb - wa) * 4u * (LN ? 2u : 1u);
        }
        mbar_arrive_expect_tx(&h.full[s], tx);
        bulk_g2s(dst, static_cast<const unsigned char *>(t0) + r0 * row_bytes, bytes, &h.full[s]);
        if constexpr (BWD) {
            bulk_g2s(dst + tile_bytes, static_cast<const unsigned char *>(t1) + r0 * row_bytes, bytes,
                     &h.full[s]);
            if (wb > wa) {
                float *sd = reinterpret_cast<float *>(dst + 2 * (size_t)tile_bytes);
                bulk_g2s(sd, st0 + wa, (uint32_t)(wb - wa) * 4u, &h.full[s]);
                if constexpr (LN)
                    bulk_g2s(sd + stat_stride(RT), st1 + wa, (uint32_t)(wb - wa) * 4u, &h.full[s]);
            }
        }
    }
    if (*abort_flag) {
        // Copies this thread issued may still be landing: wait for each (bounded,
        // regardless of the abort flag) before the CTA may exit.
        int zero = 0;
        const int first = issued > S ? issued - S : 0;
        for (int j = first; j < issued; ++j)
            mbar_wait_bounded(&h.full[j % S], (j / S) & 1, reinterpret_cast<volatile int *>(&zero), nullptr);
    }
}

// gamma (and beta) for the whole row are brought into shared memory once per
// CTA by the producer's bulk copies, completing h.pbar: every row reads them
// again, and registers are kept for the backward's dgamma/dbeta partials.
__device__ __forceinline__ void load_params(uint64_t *pbar, void *gdst, void *bdst, const void *g,
                                            const void *b, uint32_t bytes) {
    mbar_arrive_expect_tx(pbar, bytes * (b ? 2u : 1u));
    bulk_g2s(gdst, g, bytes, pbar);
    if (b) bulk_g2s(bdst, b, bytes, pbar);
}

// Bytes of shared memory the TMA kernels keep for gamma (and beta).
__host__ __device__ constexpr size_t tma_param_bytes(int64_t n_bytes, bool two) {
    return (size_t)((n_bytes + 127) & ~(int64_t)127) * (two ? 2 : 1);
}

// ============================================================================ forward
template <typename T, bool LN, int TPR, int VPT, int CW>
__global__ void __launch_bounds__((CW + 1) * 32, 1) fwd_tma(const FwdParams p) {
    constexpr int E = VecTraits<T>::E;
    constexpr int NT = CW * 32;
    constexpr int RPP = NT / TPR;
    constexpr int WPR = TPR > 32 ? TPR / 32 : 1;
    static_assert(NT % TPR == 0 && (TPR <= 32 || TPR % 32 == 0), "row group shape");
    static_assert(TPR <= 32 || (RPP * 2 * 2 * WPR <= (int)(sizeof(TmaHeader::red) / 4) && RPP <= 14),
                  "scratch / named barrier ids");
    extern __shared__ __align__(128) unsigned char smem[];
    TmaHeader &h = *reinterpret_cast<TmaHeader *>(smem);
    const int64_t M = p.M, nv = p.N / E;
    const size_t row_bytes = (size_t)p.N * sizeof(T);
    uint4 *par = reinterpret_cast<uint4 *>(smem + kTmaHeaderBytes);  // gamma [nv], beta [nv]
    unsigned char *stages = smem + kTmaHeaderBytes + tma_param_bytes((int64_t)row_bytes, LN);
    const int S = p.tc.stages, RT = p.tc.rows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint4 *beta_s = par + (tma_param_bytes((int64_t)row_bytes, false) / 16);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&h.full[s], 1);
            mbar_init(&h.empty[s], CW);
        }
        mbar_init(&h.pbar, 1);
        h.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == CW) {
        if (lane == 0) {
            load_params(&h.pbar, par, beta_s, p.gamma, LN ? p.beta : nullptr, (uint32_t)row_bytes);
            tma_produce<false, LN>(h, stages, p.tc, M, row_bytes, p.x, nullptr, nullptr, nullptr, 0);
        }
        return;
    }

    mbar_wait_bounded(&h.pbar, 0, &h.abort, p.tc.fault);
    const uint4 *gs = par;
    const uint4 *bs = beta_s;
    const int t = threadIdx.x % TPR, grp = threadIdx.x / TPR;
    float *scratch = h.red + grp * (2 * 2 * WPR);
    const float n = (float)p.N;
    const bool full = nv == (int64_t)TPR * VPT;  // every thread holds VPT vectors of each row
    volatile int *abort_flag = &h.abort;
    int parity = 0, it = 0;
    const int64_t ntiles = (M + RT - 1) / RT;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
        const int s = it % S;
        mbar_wait_bounded(&h.full[s], (it / S) & 1, abort_flag, p.tc.fault);
        const int64_t r0 = tile * RT;
        const int rows = (int)(M - r0 < RT ? M - r0 : RT);
        const unsigned char *tb = stages + (size_t)s * p.tc.stride;
        // Uniform trip count for every thread of the CTA (row groups narrower
        // than a warp share shuffles); rows past the tile are predicated off.
        for (int rb = 0; rb < rows; rb += RPP) {
            const int r = rb + grp;
            const bool rok = r < rows;
            const uint4 *xs = reinterpret_cast<const uint4 *>(tb + (size_t)(rok ? r : 0) * row_bytes);
            float acc[1] = {0.f};
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * TPR + t;
                if (!rok || v >= nv) continue;
                const uint4 q = lds128(xs + v);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float f = vget<T>(q, e);
                    acc[0] += LN ? f : f * f;
                }
            }
            float mean = 0.f;
            if (LN && full) {
                // Every thread holds VPT * E elements of the row: local mean and
                // M2 from the staged row, then one equal-count merge.
                constexpr float kC = (float)(VPT * E);
                mean = acc[0] * (1.f / kC);
                float m2 = 0.f;
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = k * TPR + t;
                    if (!rok) continue;
                    const uint4 q = lds128(xs + v);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float d = vget<T>(q, e) - mean;
                        m2 += d * d;
                    }
                }
                group_merge_equal<TPR>(mean, m2, kC, scratch, parity, 1 + grp);
                acc[0] = m2;
            } else {
            group_allreduce<TPR, 1>(acc, scratch, parity, 1 + grp);
            if constexpr (LN) {
                // Second pass over the staged row: centred sum of squares.
                mean = acc[0] / n;
                acc[0] = 0.f;
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = k * TPR + t;
                    if (!rok || v >= nv) continue;
                    const uint4 q = lds128(xs + v);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float d = vget<T>(q, e) - mean;
                        acc[0] += d * d;
                    }
                }
                group_allreduce<TPR, 1>(acc, scratch, parity, 1 + grp);
            }
            }
            const float rstd = rsqrtf(acc[0] / n + p.eps);
            if (!rok) continue;  // uniform per row group: no collective below
            const int64_t row = r0 + r;
            if (t == 0) {
                if (p.rstd) p.rstd[row] = rstd;
                if (LN && p.mean) p.mean[row] = mean;
            }
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * TPR + t;
                if (v >= nv) continue;
                const uint4 q = lds128(xs + v), g = lds128(gs + v);
                uint4 b;
                if constexpr (LN) b = lds128(bs + v);
                float o[E];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    o[e] = ((vget<T>(q, e) - mean) * rstd) * vget<T>(g, e);
                    if constexpr (LN) o[e] += vget<T>(b, e);
                }
                st_vec(p.y, row * nv + v, vpack<T>(o));
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&h.empty[s]);
    }
}

// ============================================================================ backward
template <typename T, bool LN, int TPR, int VPT, int CW>
__global__ void __launch_bounds__((CW + 1) * 32, 1) bwd_tma(const BwdParams p) {
    pdl_launch_dependents();  // the column reduce waits for this grid's completion
    constexpr int E = VecTraits<T>::E;
    constexpr int NT = CW * 32;
    constexpr int RPP = NT / TPR;
    constexpr int WPR = TPR > 32 ? TPR / 32 : 1;
    constexpr int NS = LN ? 2 : 1;
    constexpr bool HOLD = VPT * E <= 24;  // keep pass-1 values in registers for pass 2
    static_assert(NT % TPR == 0 && (TPR <= 32 || TPR % 32 == 0), "row group shape");
    static_assert(TPR <= 32 || (RPP * 2 * NS * WPR <= (int)(sizeof(TmaHeader::red) / 4) && RPP <= 14),
                  "scratch / named barrier ids");
    extern __shared__ __align__(128) unsigned char smem[];
    TmaHeader &h = *reinterpret_cast<TmaHeader *>(smem);
    const int64_t M = p.M, nv = p.N / E;
    const size_t row_bytes = (size_t)p.N * sizeof(T);
    uint4 *par = reinterpret_cast<uint4 *>(smem + kTmaHeaderBytes);  // gamma [nv]
    unsigned char *stages = smem + kTmaHeaderBytes + tma_param_bytes((int64_t)row_bytes, false);
    const int S = p.tc.stages, RT = p.tc.rows;
    const uint32_t tile_bytes = (uint32_t)((RT * row_bytes + 127) & ~(size_t)127);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&h.full[s], 1);
            mbar_init(&h.empty[s], CW);
        }
        mbar_init(&h.pbar, 1);
        h.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == CW) {
        if (lane == 0) {
            load_params(&h.pbar, par, nullptr, p.gamma, nullptr, (uint32_t)row_bytes);
            tma_produce<true, LN>(h, stages, p.tc, M, row_bytes, p.x, p.dy, p.rstd, p.mean, tile_bytes);
        }
        return;
    }

    mbar_wait_bounded(&h.pbar, 0, &h.abort, p.tc.fault);
    const uint4 *gs = par;
    const int t = threadIdx.x % TPR, grp = threadIdx.x / TPR;
    float *scratch = h.red + grp * (2 * NS * WPR);
    // HOLD: this thread's gamma, widened once (its columns never change).
    float gf[HOLD ? VPT : 1][E];
    if constexpr (HOLD) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = k * TPR + t;
            const uint4 g = v < nv ? lds128(gs + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int e = 0; e < E; ++e) gf[k][e] = vget<T>(g, e);
        }
    }
    const float n = (float)p.N;
    float accg[VPT][E], accb[LN ? VPT : 1][E];
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int e = 0; e < E; ++e) {
            accg[k][e] = 0.f;
            if constexpr (LN) accb[k][e] = 0.f;
        }
    volatile int *abort_flag = &h.abort;
    int parity = 0, it = 0;
    const int64_t ntiles = (M + RT - 1) / RT;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
        const int s = it % S;
        mbar_wait_bounded(&h.full[s], (it / S) & 1, abort_flag, p.tc.fault);
        const int64_t r0 = tile * RT;
        const int rows = (int)(M - r0 < RT ? M - r0 : RT);
        int64_t wa, wb;
        stat_window(r0, rows, M, &wa, &wb);
        const unsigned char *tb = stages + (size_t)s * p.tc.stride;
        const float *st = reinterpret_cast<const float *>(tb + 2 * (size_t)tile_bytes) - wa;
        for (int rb = 0; rb < rows; rb += RPP) {  // uniform trip count, see the forward
            const int r = rb + grp;
            const bool rok = r < rows;
            const size_t off = (size_t)(rok ? r : 0) * row_bytes;
            const uint4 *xs = reinterpret_cast<const uint4 *>(tb + off);
            const uint4 *ds = reinterpret_cast<const uint4 *>(tb + tile_bytes + off);
            const int64_t row = r0 + r;
            float rstd = 0.f, mean = 0.f;
            if (rok) {
                const bool in_win = row < wb;  // row >= wa always holds
                rstd = in_win ? st[row] : __ldg(p.rstd + row);
                if constexpr (LN) mean = in_win ? st[stat_stride(RT) + row] : __ldg(p.mean + row);
            }
            // Pass 1: x-hat and g = dy * gamma, their products summed over the
            // row.  With at most 24 elements per thread (HOLD) x-hat, g and the
            // raw dy stay in registers for pass 2; otherwise pass 2 re-reads the
            // staged row.
            float sum[NS];
#pragma unroll
            for (int i = 0; i < NS; ++i) sum[i] = 0.f;
            float hx[HOLD ? VPT : 1][E], hg[HOLD ? VPT : 1][E];
            uint4 hd[HOLD ? VPT : 1];
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * TPR + t;
                const bool ok = rok && v < nv;
                const uint4 q = ok ? lds128(xs + v) : make_uint4(0, 0, 0, 0);
                const uint4 d = ok ? lds128(ds + v) : make_uint4(0, 0, 0, 0);
                uint4 g = make_uint4(0, 0, 0, 0);
                if constexpr (HOLD) {
                    hd[k] = d;
                } else {
                    g = ok ? lds128(gs + v) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float xh = (vget<T>(q, e) - mean) * rstd;
                    const float gg = vget<T>(d, e) * (HOLD ? gf[HOLD ? k : 0][e] : vget<T>(g, e));
                    if constexpr (HOLD) {
                        hx[k][e] = xh;
                        hg[k][e] = gg;
                    }
                    sum[0] += gg * xh;
                    if constexpr (LN) sum[NS - 1] += gg;
                }
            }
            group_allreduce<TPR, NS>(sum, scratch, parity, 1 + grp);
            if (!rok) continue;  // uniform per row group: no collective below
            const float c2 = sum[0] / n;
            const float c1 = LN ? sum[NS - 1] / n : 0.f;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * TPR + t;
                if (v >= nv) continue;
                float o[E];
                if constexpr (HOLD) {
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float dyv = vget<T>(hd[k], e);
                        o[e] = rstd * (hg[k][e] - c1 - hx[k][e] * c2);
                        accg[k][e] += dyv * hx[k][e];
                        if constexpr (LN) accb[k][e] += dyv;
                    }
                } else {
                    const uint4 q = lds128(xs + v), d = lds128(ds + v), g = lds128(gs + v);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float xh = (vget<T>(q, e) - mean) * rstd;
                        const float dyv = vget<T>(d, e);
                        const float gg = dyv * vget<T>(g, e);
                        o[e] = rstd * (gg - c1 - xh * c2);
                        accg[k][e] += dyv * xh;
                        if constexpr (LN) accb[k][e] += dyv;
                    }
                }
                st_vec(p.dx, row * nv + v, vpack<T>(o));
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&h.empty[s]);
    }

    // Epilogue: the CTA's row groups own the same columns.  Every group writes
    // its partials to shared memory (the stage ring is idle now: every copy
    // issued was waited for above), then each thread adds, for its columns,
    // the groups' values in group order, and writes the CTA's partial row.
    float *wsg = p.ws + (int64_t)blockIdx.x * p.N;
    float *wsb = p.ws + ((int64_t)gridDim.x + blockIdx.x) * p.N;
    if constexpr (RPP > 1) {
        constexpr int CAP = TPR * VPT * E;  // columns one row group covers
        float *comb = reinterpret_cast<float *>(stages);  // [NS][RPP][CAP]
        named_sync(kTmaBarAll, NT);  // all rows done with the ring
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int c = (k * TPR + t) * E + e;
                comb[grp * CAP + c] = accg[k][e];
                if constexpr (LN) comb[(RPP + grp) * CAP + c] = accb[k][e];
            }
        named_sync(kTmaBarAll, NT);
        const int64_t ncol = nv * E < CAP ? nv * E : CAP;
        for (int c = threadIdx.x; c < ncol; c += NT) {
            float sg = 0.f, sb = 0.f;
#pragma unroll 4
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
            const int64_t v = (int64_t)k * TPR + t;
            if (v >= nv) continue;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                wsg[v * E + e] = accg[k][e];
                if constexpr (LN) wsb[v * E + e] = accb[k][e];
            }
        }
    }
}

}  // namespace gbn
