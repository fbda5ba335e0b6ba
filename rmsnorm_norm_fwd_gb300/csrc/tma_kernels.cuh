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
// again, and registers are kept for the backward's dgamma/dbeta partials.  A
// null row is not copied (the consumers use the constant it stands for).
__device__ __forceinline__ void load_params(uint64_t *pbar, void *gdst, void *bdst, const void *g,
                                            const void *b, uint32_t bytes) {
    mbar_arrive_expect_tx(pbar, bytes * ((g ? 1u : 0u) + (b ? 1u : 0u)));
    if (g) bulk_g2s(gdst, g, bytes, pbar);
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
                // M2 from the staged row, then one equal-count combine.
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
                group_meanvar_equal<TPR>(mean, m2, kC, scratch, parity, 1 + grp);
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
                const uint4 q = lds128(xs + v);
                const uint4 g = p.gamma ? lds128(gs + v) : ones_vec<T>();
                uint4 b;
                if constexpr (LN) b = p.beta ? lds128(bs + v) : make_uint4(0, 0, 0, 0);
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

// ============================================================================ single-kernel column reduce
// The second stage of the dgamma/dbeta reduction run by the backward kernel
// itself ("Fused RMSNorm", sections "What didn't work" / "Next": per-block
// partials, then a vectorised column sum -- here without a second launch).
// The kernel is launched cooperatively, so all P CTAs are resident.  After
// writing its partial row, each CTA publishes the call's epoch in its flag
// word (release, after a fence by every thread); one warp per CTA waits,
// bounded, until all P flags carry the epoch (acquire), then the CTA sums its
// share of the columns over the P partial rows: column groups of 32 lanes x VW
// (4 floats, or 1 when N % 4 != 0), group c taken by CTA c mod P, the rows
// split into 16 bands summed in row order and the band sums added in band
// order -- the order of colreduce, so the result is bit-identical to the
// two-kernel path with the same P.  The flags sit after the partial rows in
// the workspace (after NB = 1 or 2 blocks of them); stale flags from earlier
// calls carry other epochs.  `part` is 16 x 128 floats of idle shared
// memory; NT threads (bar_id) take part.
template <int NT, int NB>
__device__ __forceinline__ void sk_column_reduce(const BwdParams &p, float *part, volatile int *abort,
                                                 int bar_id) {
    constexpr int W = NT / 32;
    constexpr int kBands = kColCTA / 32;
    const int64_t P = gridDim.x, N = p.N;
    if (!p.dgamma && !p.dbeta) return;  // uniform: nothing to sum
    uint32_t *flags = reinterpret_cast<uint32_t *>(p.ws + NB * P * N);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __threadfence();
    named_sync(bar_id, NT);
    if (threadIdx.x == 0) st_release_gpu(flags + blockIdx.x, p.epoch);
    if (warp == 0) {
        const long long t0 = clock64();
        while (true) {
            bool mine = true;
            for (int64_t q = lane; q < P; q += 32) mine = mine && ld_acquire_gpu(flags + q) == p.epoch;
            if (__all_sync(0xffffffffu, mine)) break;
            if (*abort || clock64() - t0 > kWaitLimitCycles) {
                if (lane == 0) {
                    *abort = 1;
                    if (p.tc.fault) atomicExch(p.tc.fault, 1);
                }
                break;
            }
        }
    }
    named_sync(bar_id, NT);
    if (*abort) return;
    __threadfence();
    const int VW = (N & 3) == 0 ? 4 : 1;
    const int64_t ngroups = (N + 32 * VW - 1) / (32 * VW);
    for (int64_t cg = blockIdx.x; cg < ngroups; cg += P) {
        const int64_t col = (cg * 32 + lane) * VW;
        const bool ok = col < N;
#pragma unroll 1
        for (int s = 0; s < NB; ++s) {
            float *out = s ? p.dbeta : p.dgamma;
            if (!out) continue;  // uniform
            const float *src = p.ws + (int64_t)s * P * N;
            for (int band = warp; band < kBands; band += W) {
                const int64_t p0 = P * band / kBands, p1 = P * (band + 1) / kBands;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                if (ok) {
                    constexpr int kB = 16;
                    for (int64_t q0 = p0; q0 < p1; q0 += kB) {
                        if (VW == 4) {
                            float4 a[kB];
#pragma unroll
                            for (int i = 0; i < kB; ++i)
                                a[i] = q0 + i < p1 ? __ldcg(reinterpret_cast<const float4 *>(src + (q0 + i) * N + col))
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                            for (int i = 0; i < kB; ++i) {
                                acc[0] += a[i].x;
                                acc[1] += a[i].y;
                                acc[2] += a[i].z;
                                acc[3] += a[i].w;
                            }
                        } else {
                            float a[kB];
#pragma unroll
                            for (int i = 0; i < kB; ++i) a[i] = q0 + i < p1 ? __ldcg(src + (q0 + i) * N + col) : 0.f;
#pragma unroll
                            for (int i = 0; i < kB; ++i) acc[0] += a[i];
                        }
                    }
                }
                for (int v = 0; v < VW; ++v) part[band * 128 + lane * VW + v] = acc[v];
            }
            named_sync(bar_id, NT);
            if (warp == 0 && ok) {
                float r[4];
                for (int v = 0; v < VW; ++v) {
                    r[v] = 0.f;
                    for (int b = 0; b < kBands; ++b) r[v] += part[b * 128 + lane * VW + v];
                }
                if (VW == 4 && (reinterpret_cast<uintptr_t>(out + col) & 15) == 0) {
                    *reinterpret_cast<float4 *>(out + col) = make_float4(r[0], r[1], r[2], r[3]);
                } else {
                    for (int v = 0; v < VW; ++v) out[col + v] = r[v];
                }
            }
            named_sync(bar_id, NT);
        }
    }
}

// ============================================================================ backward
template <typename T, bool LN, int TPR, int VPT, int CW, bool SK = false>
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
    constexpr int H = E / 4;  // float4 per 16-byte vector
    float4 *gpar = reinterpret_cast<float4 *>(smem + kTmaHeaderBytes);  // gamma as fp32 [H][nv]
    unsigned char *stages = smem + kTmaHeaderBytes + tma_param_bytes(p.N * 4, false);
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
        if (lane == 0)
            tma_produce<true, LN>(h, stages, p.tc, M, row_bytes, p.x, p.dy, p.rstd, p.mean, tile_bytes);
        return;
    }

    // gamma, widened to fp32 once per CTA by the consumers.
    for (int64_t v = threadIdx.x; v < nv; v += NT) {
        const uint4 g = param_vec<T>(p.gamma, v, true);
#pragma unroll
        for (int hh = 0; hh < H; ++hh)
            gpar[hh * nv + v] = make_float4(vget<T>(g, 4 * hh), vget<T>(g, 4 * hh + 1), vget<T>(g, 4 * hh + 2),
                                           vget<T>(g, 4 * hh + 3));
    }
    named_sync(kTmaBarAll, NT);
    const int t = threadIdx.x % TPR, grp = threadIdx.x / TPR;
    float *scratch = h.red + grp * (2 * NS * WPR);
    // gamma of vector v of this thread's columns, as E floats.
    auto gamma_of = [&](int v, float2 (&g)[E / 2]) {
#pragma unroll
        for (int hh = 0; hh < H; ++hh) {
            const float4 q = gpar[hh * nv + v];
            g[2 * hh] = make_float2(q.x, q.y);
            g[2 * hh + 1] = make_float2(q.z, q.w);
        }
    };
    // HOLD: this thread's gamma, kept in registers (its columns never change).
    float2 gf[HOLD ? VPT : 1][E / 2];
    if constexpr (HOLD) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = k * TPR + t;
            if (v < nv) {
                gamma_of(v, gf[k]);
            } else {
#pragma unroll
                for (int e = 0; e < E / 2; ++e) gf[k][e] = f2s(0.f);
            }
        }
    }
    const float n = (float)p.N;
    // dgamma (and dbeta) partials of this thread's columns, as pairs
    float2 accg[VPT][E / 2], accb[LN ? VPT : 1][E / 2];
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int e = 0; e < E / 2; ++e) {
            accg[k][e] = f2s(0.f);
            if constexpr (LN) accb[k][e] = f2s(0.f);
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
            // Pass 1: g = dy * gamma and the row sums of g (x - mean) and g;
            // sum g xhat = rstd * sum g (x - mean).  With at most 24 elements
            // per thread (HOLD) x - mean, g and the raw dy stay in registers for
            // pass 2; otherwise pass 2 re-reads the staged row.
            const float2 nm = f2s(-mean);
            float2 s2 = f2s(0.f), s1 = f2s(0.f);
            float2 hx[HOLD ? VPT : 1][E / 2], hg[HOLD ? VPT : 1][E / 2];
            uint4 hd[HOLD ? VPT : 1];
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * TPR + t;
                const bool ok = rok && v < nv;
                const uint4 q = ok ? lds128(xs + v) : make_uint4(0, 0, 0, 0);
                const uint4 d = ok ? lds128(ds + v) : make_uint4(0, 0, 0, 0);
                float2 gk[E / 2];
                if constexpr (HOLD) {
                    hd[k] = d;
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) gk[e] = gf[HOLD ? k : 0][e];
                } else if (ok) {
                    gamma_of(v, gk);
                } else {
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) gk[e] = f2s(0.f);
                }
#pragma unroll
                for (int e = 0; e < E / 2; ++e) {
                    const float2 xc = f2add(vpair<T>(q, e), nm);
                    const float2 gg = f2mul(vpair<T>(d, e), gk[e]);
                    if constexpr (HOLD) {
                        hx[k][e] = xc;
                        hg[k][e] = gg;
                    }
                    s2 = f2fma(gg, xc, s2);
                    if constexpr (LN) s1 = f2add(s1, gg);
                }
            }
            float sum[NS];
            sum[0] = s2.x + s2.y;
            if constexpr (LN) sum[NS - 1] = s1.x + s1.y;
            group_allreduce<TPR, NS>(sum, scratch, parity, 1 + grp);
            if (!rok) continue;  // uniform per row group: no collective below
            // dx = rstd (g - c1 - xhat c2) = rstd g - rstd c1 - (rstd c2) xhat,
            // c2 = rstd sum g (x - mean) / n, c1 = sum g / n.
            const float c2 = rstd * sum[0] / n;
            const float rc1 = LN ? rstd * (sum[NS - 1] / n) : 0.f;
            const float rc2 = rstd * c2;
            const float2 r2 = f2s(rstd), nrc1 = f2s(-rc1), nrc2 = f2s(-rc2);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * TPR + t;
                if (v >= nv) continue;
                float2 o[E / 2];
                if constexpr (HOLD) {
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) {
                        const float2 dyv = vpair<T>(hd[k], e);
                        const float2 xh = f2mul(hx[k][e], r2);
                        o[e] = f2fma(nrc2, xh, f2fma(r2, hg[k][e], nrc1));
                        accg[k][e] = f2fma(dyv, xh, accg[k][e]);
                        if constexpr (LN) accb[k][e] = f2add(accb[k][e], dyv);
                    }
                } else {
                    const uint4 q = lds128(xs + v), d = lds128(ds + v);
                    float2 gk[E / 2];
                    gamma_of(v, gk);
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) {
                        const float2 xh = f2mul(f2add(vpair<T>(q, e), nm), r2);
                        const float2 dyv = vpair<T>(d, e);
                        o[e] = f2fma(nrc2, xh, f2fma(r2, f2mul(dyv, gk[e]), nrc1));
                        accg[k][e] = f2fma(dyv, xh, accg[k][e]);
                        if constexpr (LN) accb[k][e] = f2add(accb[k][e], dyv);
                    }
                }
                st_vec(p.dx, row * nv + v, vpack2<T>(o));
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
            for (int e = 0; e < E / 2; ++e) {
                const int c = (k * TPR + t) * E + 2 * e;
                comb[grp * CAP + c] = accg[k][e].x;
                comb[grp * CAP + c + 1] = accg[k][e].y;
                if constexpr (LN) {
                    comb[(RPP + grp) * CAP + c] = accb[k][e].x;
                    comb[(RPP + grp) * CAP + c + 1] = accb[k][e].y;
                }
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
            for (int e = 0; e < E / 2; ++e) {
                wsg[v * E + 2 * e] = accg[k][e].x;
                wsg[v * E + 2 * e + 1] = accg[k][e].y;
                if constexpr (LN) {
                    wsb[v * E + 2 * e] = accb[k][e].x;
                    wsb[v * E + 2 * e + 1] = accb[k][e].y;
                }
            }
        }
    }
    if constexpr (SK) sk_column_reduce<NT, NS>(p, reinterpret_cast<float *>(stages), &h.abort, kTmaBarAll);
}

// ============================================================================ forward, no producer warp
// Forward counterpart of bwd_tmp: RPP = NT / TPR row groups, each streaming
// its share of the CTA's tiles of x through its own part of the ring (S /
// RPP stages), refilled by the group's first thread after the group barrier
// that follows the last read of the previous tile.  gamma (and beta) sit in
// shared memory as fp32, converted once per CTA; each row is converted once
// into fp32 registers.
template <typename T, bool LN, int TPR, int VPT, int NT>
__global__ void __launch_bounds__(NT, 1) fwd_tmp(const FwdParams p) {
    constexpr int E = VecTraits<T>::E;
    constexpr int H = E / 4;
    constexpr int RPP = NT / TPR;
    constexpr int WPR = TPR / 32;
    static_assert(NT % TPR == 0 && TPR % 32 == 0 && TPR > 32 && RPP <= 14, "CTA shape");
    static_assert(RPP * 2 * 2 * WPR <= (int)(sizeof(TmaHeader::red) / 4), "scratch");
    extern __shared__ __align__(128) unsigned char smem[];
    TmaHeader &h = *reinterpret_cast<TmaHeader *>(smem);
    const int64_t M = p.M, nv = p.N / E;
    const size_t row_bytes = (size_t)p.N * sizeof(T);
    float4 *gpar = reinterpret_cast<float4 *>(smem + kTmaHeaderBytes);  // gamma [H][nv], then beta
    float4 *bpar = gpar + tma_param_bytes(p.N * 4, false) / 16;
    unsigned char *stages = smem + kTmaHeaderBytes + tma_param_bytes(p.N * 4, LN);
    const int SG = p.tc.stages / RPP, RT = p.tc.rows;
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
        const uint32_t bytes = (uint32_t)(rows * row_bytes);
        mbar_arrive_expect_tx(&h.full[s], bytes);
        bulk_g2s(stages + (size_t)s * p.tc.stride, static_cast<const unsigned char *>(p.x) + r0 * row_bytes,
                 bytes, &h.full[s]);
        ++issued;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < RPP * SG; ++s) mbar_init(&h.full[s], 1);
        h.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (t == 0)
        for (int j = 0; j < SG; ++j) issue(j);
    for (int64_t v = threadIdx.x; v < nv; v += NT) {
        const uint4 g = param_vec<T>(p.gamma, v, true);
        uint4 b = make_uint4(0, 0, 0, 0);
        if constexpr (LN) b = param_vec<T>(p.beta, v, false);
#pragma unroll
        for (int hh = 0; hh < H; ++hh) {
            gpar[hh * nv + v] = make_float4(vget<T>(g, 4 * hh), vget<T>(g, 4 * hh + 1), vget<T>(g, 4 * hh + 2),
                                           vget<T>(g, 4 * hh + 3));
            if constexpr (LN)
                bpar[hh * nv + v] = make_float4(vget<T>(b, 4 * hh), vget<T>(b, 4 * hh + 1),
                                               vget<T>(b, 4 * hh + 2), vget<T>(b, 4 * hh + 3));
        }
    }
    __syncthreads();

    const float n = (float)p.N;
    const bool full = nv == (int64_t)TPR * VPT;  // every thread holds VPT vectors of each row
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
            const uint4 *xs = reinterpret_cast<const uint4 *>(tb + (size_t)r * row_bytes);
            const int64_t row = r0 + r;
            float2 xf[VPT][E / 2];  // the row's elements of this thread, as pairs
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * TPR + t;
                const uint4 q = v < nv ? lds128(xs + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int e = 0; e < E / 2; ++e) xf[k][e] = vpair<T>(q, e);
            }
            float2 a2 = f2s(0.f);
#pragma unroll
            for (int k = 0; k < VPT; ++k)
#pragma unroll
                for (int e = 0; e < E / 2; ++e) a2 = LN ? f2add(a2, xf[k][e]) : f2fma(xf[k][e], xf[k][e], a2);
            float acc = a2.x + a2.y;
            float mean = 0.f;
            if (LN && full) {
                constexpr float kC = (float)(VPT * E);
                mean = acc * (1.f / kC);
                const float2 nm = f2s(-mean);
                float2 q2 = f2s(0.f);
#pragma unroll
                for (int k = 0; k < VPT; ++k)
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) {
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
                        if (k * TPR + t >= nv) continue;
#pragma unroll
                        for (int e = 0; e < E / 2; ++e) {
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
                // Every thread of the group is past its last read of the stage
                // of its tile j - 1: order those reads before the bulk copy's
                // writes, then refill.
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
                const int v = k * TPR + t;
                if (v >= nv) continue;
                float2 o[E / 2];
#pragma unroll
                for (int hh = 0; hh < H; ++hh) {
                    const float4 g = gpar[hh * nv + v];
                    o[2 * hh] = f2mul(f2mul(f2add(xf[k][2 * hh], nm), rs), make_float2(g.x, g.y));
                    o[2 * hh + 1] = f2mul(f2mul(f2add(xf[k][2 * hh + 1], nm), rs), make_float2(g.z, g.w));
                    if constexpr (LN) {
                        const float4 b = bpar[hh * nv + v];
                        o[2 * hh] = f2add(o[2 * hh], make_float2(b.x, b.y));
                        o[2 * hh + 1] = f2add(o[2 * hh + 1], make_float2(b.z, b.w));
                    }
                }
                st_vec(p.y, row * nv + v, vpack2<T>(o));
            }
        }
    }
    if (t == 0 && *abort_flag) {
        int zero = 0;
        for (int j = issued > SG ? issued - SG : 0; j < issued; ++j)
            mbar_wait_bounded(&h.full[grp * SG + j % SG], (uint32_t)((j / SG) & 1),
                              reinterpret_cast<volatile int *>(&zero), nullptr);
    }
}

// ============================================================================ backward, no producer warp
// As bwd_tma without a producer warp: the CTA's NT threads form RPP = NT / TPR
// row groups, and each group runs its own pipeline over its share of the
// CTA's tiles (group g takes the CTA's tiles g, g + RPP, ...) through its own
// S / RPP stages of the ring, refilled by the group's first thread.  The
// group barrier inside the first row's reduction of the group's tile j
// follows every group thread's last read of tile j - 1's stage, so right
// after it that thread issues the copy of tile j - 1 + S / RPP into it.
// Without a 17th warp the register budget is 65536 / NT per thread (128 for
// 512 threads), which holds the dgamma and dbeta partials and, for up to 24
// elements per thread, the pass-1 values (x - mean, g and dy) for pass 2.
template <typename T, bool LN, int TPR, int VPT, int NT, bool SK = false>
__global__ void __launch_bounds__(NT, 1) bwd_tmp(const BwdParams p) {
    pdl_launch_dependents();  // the column reduce waits for this grid's completion
    constexpr int E = VecTraits<T>::E;
    constexpr int H = E / 4;
    constexpr int NS = LN ? 2 : 1;
    constexpr int RPP = NT / TPR;
    constexpr int WPR = TPR / 32;
    constexpr bool HOLD = VPT * E <= 24;
    // TPR > 32: the group reduction is a named barrier, which the refill relies on
    static_assert(NT % TPR == 0 && TPR % 32 == 0 && TPR > 32 && RPP <= 14, "CTA shape");
    static_assert(RPP * 2 * NS * WPR <= (int)(sizeof(TmaHeader::red) / 4), "scratch");
    extern __shared__ __align__(128) unsigned char smem[];
    TmaHeader &h = *reinterpret_cast<TmaHeader *>(smem);
    const int64_t M = p.M, nv = p.N / E;
    const size_t row_bytes = (size_t)p.N * sizeof(T);
    float4 *gpar = reinterpret_cast<float4 *>(smem + kTmaHeaderBytes);  // gamma as fp32 [H][nv]
    unsigned char *stages = smem + kTmaHeaderBytes + tma_param_bytes(p.N * 4, false);
    const int SG = p.tc.stages / RPP, RT = p.tc.rows;  // stages per row group
    const uint32_t tile_bytes = (uint32_t)((RT * row_bytes + 127) & ~(size_t)127);
    const int64_t ntiles = (M + RT - 1) / RT;
    const int t = threadIdx.x % TPR, grp = threadIdx.x / TPR;
    float *scratch = h.red + grp * (2 * NS * WPR);
    volatile int *abort_flag = &h.abort;
    int issued = 0;  // group leader: copies issued

    // The CTA tile of the group's j-th tile, or -1.
    auto tile_of = [&](int64_t j) {
        const int64_t tile = blockIdx.x + (grp + j * RPP) * (int64_t)gridDim.x;
        return tile < ntiles ? tile : (int64_t)-1;
    };
    // Copy the group's j-th tile into its stage j % SG (group leader).
    auto issue = [&](int64_t j) {
        const int64_t tile = tile_of(j);
        if (tile < 0) return;
        const int s = grp * SG + (int)(j % SG);
        const int64_t r0 = tile * RT;
        const int rows = (int)(M - r0 < RT ? M - r0 : RT);
        const uint32_t bytes = (uint32_t)(rows * row_bytes);
        unsigned char *dst = stages + (size_t)s * p.tc.stride;
        int64_t wa, wb;
        stat_window(r0, rows, M, &wa, &wb);
        mbar_arrive_expect_tx(&h.full[s], 2 * bytes + (uint32_t)(wb - wa) * 4u * (LN ? 2u : 1u));
        bulk_g2s(dst, static_cast<const unsigned char *>(p.x) + r0 * row_bytes, bytes, &h.full[s]);
        bulk_g2s(dst + tile_bytes, static_cast<const unsigned char *>(p.dy) + r0 * row_bytes, bytes, &h.full[s]);
        if (wb > wa) {
            float *sd = reinterpret_cast<float *>(dst + 2 * (size_t)tile_bytes);
            bulk_g2s(sd, p.rstd + wa, (uint32_t)(wb - wa) * 4u, &h.full[s]);
            if constexpr (LN) bulk_g2s(sd + stat_stride(RT), p.mean + wa, (uint32_t)(wb - wa) * 4u, &h.full[s]);
        }
        ++issued;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < RPP * SG; ++s) mbar_init(&h.full[s], 1);
        h.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (t == 0)
        for (int j = 0; j < SG; ++j) issue(j);
    for (int64_t v = threadIdx.x; v < nv; v += NT) {
        const uint4 g = param_vec<T>(p.gamma, v, true);
#pragma unroll
        for (int hh = 0; hh < H; ++hh)
            gpar[hh * nv + v] = make_float4(vget<T>(g, 4 * hh), vget<T>(g, 4 * hh + 1), vget<T>(g, 4 * hh + 2),
                                           vget<T>(g, 4 * hh + 3));
    }
    __syncthreads();
    // gamma of vector v of this thread's columns, as E / 2 pairs
    auto gamma_of = [&](int v, float2 (&g)[E / 2]) {
#pragma unroll
        for (int hh = 0; hh < H; ++hh) {
            const float4 q = gpar[hh * nv + v];
            g[2 * hh] = make_float2(q.x, q.y);
            g[2 * hh + 1] = make_float2(q.z, q.w);
        }
    };
    float2 gf[HOLD ? VPT : 1][E / 2];
    if constexpr (HOLD) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = k * TPR + t;
            if (v < nv) {
                gamma_of(v, gf[k]);
            } else {
#pragma unroll
                for (int e = 0; e < E / 2; ++e) gf[k][e] = f2s(0.f);
            }
        }
    }
    const float n = (float)p.N;
    float2 accg[VPT][E / 2], accb[LN ? VPT : 1][E / 2];
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int e = 0; e < E / 2; ++e) {
            accg[k][e] = f2s(0.f);
            if constexpr (LN) accb[k][e] = f2s(0.f);
        }
    int parity = 0;
    // Trip count uniform over the CTA (the epilogue's barriers); groups past
    // their last tile idle through the remaining iterations.
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
        const float *st = reinterpret_cast<const float *>(tb + 2 * (size_t)tile_bytes) - wa;
        for (int r = 0; r < rows; ++r) {  // every thread of the group works on the same row
            const uint4 *xs = reinterpret_cast<const uint4 *>(tb + (size_t)r * row_bytes);
            const uint4 *ds = reinterpret_cast<const uint4 *>(tb + tile_bytes + (size_t)r * row_bytes);
            const int64_t row = r0 + r;
            const bool in_win = row < wb;
            const float rstd = in_win ? st[row] : __ldg(p.rstd + row);
            const float mean = LN ? (in_win ? st[stat_stride(RT) + row] : __ldg(p.mean + row)) : 0.f;
            const float2 nm = f2s(-mean);
            float2 s2 = f2s(0.f), s1 = f2s(0.f);
            float2 hx[HOLD ? VPT : 1][E / 2], hg[HOLD ? VPT : 1][E / 2];
            uint4 hd[HOLD ? VPT : 1];
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * TPR + t;
                const bool ok = v < nv;
                const uint4 q = ok ? lds128(xs + v) : make_uint4(0, 0, 0, 0);
                const uint4 d = ok ? lds128(ds + v) : make_uint4(0, 0, 0, 0);
                float2 gk[E / 2];
                if constexpr (HOLD) {
                    hd[k] = d;
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) gk[e] = gf[HOLD ? k : 0][e];
                } else if (ok) {
                    gamma_of(v, gk);
                } else {
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) gk[e] = f2s(0.f);
                }
#pragma unroll
                for (int e = 0; e < E / 2; ++e) {
                    const float2 xc = f2add(vpair<T>(q, e), nm);
                    const float2 gg = f2mul(vpair<T>(d, e), gk[e]);
                    if constexpr (HOLD) {
                        hx[k][e] = xc;
                        hg[k][e] = gg;
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
                // Every thread of the group is past its last read of the
                // stage of its tile j - 1: order those reads before the bulk
                // copy's writes, then refill.
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(j - 1 + SG);
            }
            const float c2 = rstd * sum[0] / n;
            const float rc1 = LN ? rstd * (sum[NS - 1] / n) : 0.f;
            const float rc2 = rstd * c2;
            const float2 r2 = f2s(rstd), nrc1 = f2s(-rc1), nrc2 = f2s(-rc2);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * TPR + t;
                if (v >= nv) continue;
                float2 o[E / 2];
                if constexpr (HOLD) {
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) {
                        const float2 dyv = vpair<T>(hd[k], e);
                        const float2 xh = f2mul(hx[k][e], r2);
                        o[e] = f2fma(nrc2, xh, f2fma(r2, hg[k][e], nrc1));
                        accg[k][e] = f2fma(dyv, xh, accg[k][e]);
                        if constexpr (LN) accb[k][e] = f2add(accb[k][e], dyv);
                    }
                } else {
                    const uint4 q = lds128(xs + v), d = lds128(ds + v);
                    float2 gk[E / 2];
                    gamma_of(v, gk);
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) {
                        const float2 xh = f2mul(f2add(vpair<T>(q, e), nm), r2);
                        const float2 dyv = vpair<T>(d, e);
                        o[e] = f2fma(nrc2, xh, f2fma(r2, f2mul(dyv, gk[e]), nrc1));
                        accg[k][e] = f2fma(dyv, xh, accg[k][e]);
                        if constexpr (LN) accb[k][e] = f2add(accb[k][e], dyv);
                    }
                }
                st_vec(p.dx, row * nv + v, vpack2<T>(o));
            }
        }
    }
    if (t == 0 && *abort_flag) {
        // Copies still landing after an aborted wait: wait for each (bounded)
        // before the CTA may exit.
        int zero = 0;
        for (int j = issued > SG ? issued - SG : 0; j < issued; ++j)
            mbar_wait_bounded(&h.full[grp * SG + j % SG], (uint32_t)((j / SG) & 1),
                              reinterpret_cast<volatile int *>(&zero), nullptr);
    }

    // Epilogue: this CTA's partial row.  With several row groups (same
    // columns), every group writes its partials to the idle ring, then each
    // thread adds, for its columns, the groups' values in group order.
    float *wsg = p.ws + (int64_t)blockIdx.x * p.N;
    float *wsb = p.ws + ((int64_t)gridDim.x + blockIdx.x) * p.N;
    if constexpr (RPP > 1) {
        constexpr int CAP = TPR * VPT * E;
        float *comb = reinterpret_cast<float *>(stages);  // [NS][RPP][CAP]
        __syncthreads();  // every group is done with the ring
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < E / 2; ++e) {
                const int c = (k * TPR + t) * E + 2 * e;
                comb[grp * CAP + c] = accg[k][e].x;
                comb[grp * CAP + c + 1] = accg[k][e].y;
                if constexpr (LN) {
                    comb[(RPP + grp) * CAP + c] = accb[k][e].x;
                    comb[(RPP + grp) * CAP + c + 1] = accb[k][e].y;
                }
            }
        __syncthreads();
        const int64_t ncol = nv * E < CAP ? nv * E : CAP;
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
            const int64_t v = (int64_t)k * TPR + t;
            if (v >= nv) continue;
            float4 *g4 = reinterpret_cast<float4 *>(wsg + v * E);
            float4 *b4 = reinterpret_cast<float4 *>(wsb + v * E);
#pragma unroll
            for (int hh = 0; hh < H; ++hh) {
                g4[hh] = make_float4(accg[k][2 * hh].x, accg[k][2 * hh].y, accg[k][2 * hh + 1].x,
                                     accg[k][2 * hh + 1].y);
                if constexpr (LN)
                    b4[hh] = make_float4(accb[k][2 * hh].x, accb[k][2 * hh].y, accb[k][2 * hh + 1].x,
                                         accb[k][2 * hh + 1].y);
            }
        }
    }
    if constexpr (SK) sk_column_reduce<NT, NS>(p, reinterpret_cast<float *>(stages), &h.abort, kTmaBarAll);
}

}  // namespace gbn
