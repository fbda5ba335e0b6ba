// tma_cluster_kernels.cuh -- RMSNorm / LayerNorm forward and backward for
// wide rows: each row is split across the CL CTAs of a thread-block cluster,
// every CTA streams its contiguous column slice of each row through its own
// shared-memory ring by bulk asynchronous copies, and the row statistics are
// combined through distributed shared memory.
//
// Same arithmetic as norm_kernels.cuh (the definitions on "SOTA normalization
// performance with torch.compile", section "How Did Torch.compile Catch
// Quack?", and "Fused RMSNorm", sections "What it is" / "How it works" /
// "What didn't work"); the torch.compile page's note that wide rows lose
// without distributed shared memory is what this layout answers.
//
// Exchange: each CTA reduces its slice (warp shuffles, then warps through
// shared memory under a named barrier of the 256 consumer threads), writes
// its partial into a slot of every CTA of the cluster (st.shared::cluster)
// and arrives, with release semantics at cluster scope, on that CTA's
// exchange mbarrier; a CTA waits (acquire, bounded) for CL arrivals and adds
// the CL partials in rank order, so every CTA obtains identical bits.  A
// cluster-wide barrier.cluster is not used inside the loop: it would also
// wait for the producer thread, which itself waits for the consumers.
//
// Software pipeline per cluster, in steps of RS rows (rows r_k = cluster id +
// k * clusters): pass 1 of step j+1 (local partials, one CTA reduction for
// its RS rows) overlaps the exchange of step j; then step j's rows are
// finished (pass 2) and step j+1's partials are sent.  Slot and barrier reuse
// are safe: a CTA sends step j+2's partials only after it has received step
// j+1's from every CTA, and each CTA sends step j+1's only after it has read
// all of step j's slots.
//
// LayerNorm forward merges the per-CTA (mean, M2) pairs with the pairwise
// update of Chan, Golub and LeVeque (1979): one exchange per row, and no
// E[x^2] - mean^2 cancellation.
#pragma once

#include "device_common.cuh"
#include "params.h"
#include "tma_kernels.cuh"

namespace gbn {

constexpr int kTmacCW = 8;                 // consumer warps
constexpr int kTmacNT = kTmacCW * 32;      // consumer threads (one row group)
constexpr int kTmacMaxCl = 16;
constexpr int kTmacMaxVals = 8;            // values per exchange: rows per step x 2

struct TmacHeader {
    uint64_t full[kTmaMaxStages];
    uint64_t empty[kTmaMaxStages];
    uint64_t xch[2];                          // exchange barriers, by step parity
    uint64_t pbar;                            // gamma (and beta) slice landed
    int abort;
    int pad;
    float cta_red[2][kTmacMaxVals][kTmacCW];  // [parity][value][warp]
    float slot[2][kTmacMaxCl][kTmacMaxVals];  // [step parity][rank][value]
};
static_assert(sizeof(TmacHeader) <= kTmaHeaderBytes, "cluster header layout");

__device__ __forceinline__ size_t al128(size_t b) { return (b + 127) & ~(size_t)127; }

// Producer of the cluster kernels: one row slice per stage (x, and dy plus a
// 16-byte window of the saved statistics for the backward).
template <bool BWD, bool LN>
__device__ __forceinline__ void tmac_produce(TmacHeader &h, unsigned char *stages, const TileCfg &tc,
                                             int64_t M, size_t row_bytes, int64_t v0, int cnt,
                                             size_t slice_al, const void *t0, const void *t1,
                                             const float *st0, const float *st1) {
    const int S = tc.stages;
    const int64_t cid = cluster_id_x(), ncl = cluster_count_x();
    volatile int *abort_flag = &h.abort;
    const uint32_t bytes = (uint32_t)cnt * 16u;
    int issued = 0;
    for (int64_t row = cid; row < M; row += ncl, ++issued) {
        const int s = issued % S;
        if (issued >= S) mbar_wait_bounded(&h.empty[s], ((issued / S) - 1) & 1, abort_flag, tc.fault);
        if (*abort_flag) break;
        unsigned char *dst = stages + (size_t)s * tc.stride;
        const size_t off = (size_t)row * row_bytes + (size_t)v0 * 16;
        int64_t wa = 0, wb = 0;
        uint32_t tx = bytes;
        if constexpr (BWD) {
            stat_window(row, 1, M, &wa, &wb);
            tx += bytes + (uint32_t)(wb - wa) * 4u * (LN ? 2u : 1u);
        }
        mbar_arrive_expect_tx(&h.full[s], tx);
        bulk_g2s(dst, static_cast<const unsigned char *>(t0) + off, bytes, &h.full[s]);
        if constexpr (BWD) {
            bulk_g2s(dst + slice_al, static_cast<const unsigned char *>(t1) + off, bytes, &h.full[s]);
            if (wb > wa) {
                float *sd = reinterpret_cast<float *>(dst + 2 * slice_al);
                bulk_g2s(sd, st0 + wa, (uint32_t)(wb - wa) * 4u, &h.full[s]);
                if constexpr (LN) bulk_g2s(sd + 4, st1 + wa, (uint32_t)(wb - wa) * 4u, &h.full[s]);
            }
        }
    }
    if (*abort_flag) {
        int zero = 0;
        const int first = issued > S ? issued - S : 0;
        for (int j = first; j < issued; ++j)
            mbar_wait_bounded(&h.full[j % S], (j / S) & 1, reinterpret_cast<volatile int *>(&zero), nullptr);
    }
}

// Sum of NVAL values over the 256 consumer threads (identical bits in all).
template <int NVAL>
__device__ __forceinline__ void tmac_cta_sum(float (&v)[NVAL], TmacHeader &h, int &parity) {
    group_sum<32, NVAL>(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < NVAL; ++i) h.cta_red[parity][i][warp] = v[i];
    }
    named_sync(1, kTmacNT);
#pragma unroll
    for (int i = 0; i < NVAL; ++i) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kTmacCW; ++w) s += h.cta_red[parity][i][w];
        v[i] = s;
    }
    parity ^= 1;
}

// Send this CTA's NVAL-value partial of step parity `par` to every CTA of the
// cluster (threads 0..CL-1, one peer each).
template <int CL, int NVAL>
__device__ __forceinline__ void tmac_send(TmacHeader &h, int par, int rank, const float (&v)[NVAL]) {
    if (threadIdx.x < CL) {
        const uint32_t peer = threadIdx.x;
        const uint32_t slot = map_to_rank(smem_u32(&h.slot[par][rank][0]), peer);
#pragma unroll
        for (int i = 0; i < NVAL; ++i) st_cluster_f32(slot + 4u * i, v[i]);
        mbar_arrive_remote(map_to_rank(smem_u32(&h.xch[par]), peer));
    }
}

// ============================================================================ forward
// Rows of this cluster: k = 0, 1, ... (row = cluster id + k * clusters), in
// steps of RS rows; one CTA reduction and one exchange per step.
template <typename T, bool LN, int VPT, int CL, int RS>
__global__ void __launch_bounds__((kTmacCW + 1) * 32, 1) fwd_tmac(const FwdParams p) {
    constexpr int E = VecTraits<T>::E;
    constexpr int NT = kTmacNT;
    constexpr int NV = 2 * RS;
    static_assert(CL >= 2 && CL <= kTmacMaxCl && NV <= kTmacMaxVals, "cluster shape");
    extern __shared__ __align__(128) unsigned char smem[];
    TmacHeader &h = *reinterpret_cast<TmacHeader *>(smem);
    const int rank = (int)cluster_ctarank();
    const int64_t M = p.M, nv = p.N / E;
    const int64_t slice = (nv + CL - 1) / CL;
    const int64_t v0 = rank * slice;
    const int cnt = (int)(nv - v0 < slice ? nv - v0 : slice);
    const size_t row_bytes = (size_t)p.N * sizeof(T);
    const size_t slice_al = al128((size_t)slice * 16);
    uint4 *gs = reinterpret_cast<uint4 *>(smem + kTmaHeaderBytes);
    uint4 *bs = gs + slice_al / 16;
    unsigned char *stages = smem + kTmaHeaderBytes + slice_al * (LN ? 2 : 1);
    const int S = p.tc.stages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&h.full[s], 1);
            mbar_init(&h.empty[s], kTmacCW);
        }
        mbar_init(&h.xch[0], CL);
        mbar_init(&h.xch[1], CL);
        mbar_init(&h.pbar, 1);
        h.abort = 0;
        fence_mbar_init();
    }
    // Every CTA's barriers exist before any peer arrives on them.
    cluster_sync_all();

    if (warp == kTmacCW) {
        if (lane == 0) {
            load_params(&h.pbar, gs, bs, p.gamma ? static_cast<const uint4 *>(p.gamma) + v0 : nullptr,
                        (LN && p.beta) ? static_cast<const uint4 *>(p.beta) + v0 : nullptr,
                        (uint32_t)cnt * 16u);
            tmac_produce<false, LN>(h, stages, p.tc, M, row_bytes, v0, cnt, slice_al, p.x, nullptr,
                                    nullptr, nullptr);
        }
        return;
    }

    const int t = threadIdx.x;
    mbar_wait_bounded(&h.pbar, 0, &h.abort, p.tc.fault);

    const int64_t cid = cluster_id_x(), ncl = cluster_count_x();
    const int64_t nrows = cid < M ? (M - cid + ncl - 1) / ncl : 0;
    const int64_t nsteps = (nrows + RS - 1) / RS;
    volatile int *abort_flag = &h.abort;
    const float n = (float)p.N;
    int cpar = 0;

    auto stage_of = [&](int64_t k) {
        return reinterpret_cast<const uint4 *>(stages + (size_t)(k % S) * p.tc.stride);
    };
    // Local partials of step j: RMS {sum x^2, 0} per row; LN {slice mean,
    // slice M2} per row.  Rows past the end contribute zeros.
    auto pass1 = [&](int64_t j, float (&out)[NV]) {
        float a[RS];
#pragma unroll
        for (int i = 0; i < RS; ++i) {
            a[i] = 0.f;
            const int64_t k = j * RS + i;
            if (k >= nrows) continue;
            mbar_wait_bounded(&h.full[k % S], (uint32_t)((k / S) & 1), abort_flag, p.tc.fault);
            const uint4 *xs = stage_of(k);
#pragma unroll
            for (int q = 0; q < VPT; ++q) {
                const int lv = q * NT + t;
                if (lv >= cnt) continue;
                const uint4 x = lds128(xs + lv);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float f = vget<T>(x, e);
                    a[i] += LN ? f : f * f;
                }
            }
        }
        tmac_cta_sum<RS>(a, h, cpar);
        if constexpr (LN) {
            float m2[RS];
            const float inv = 1.f / (float)(cnt * E);
#pragma unroll
            for (int i = 0; i < RS; ++i) {
                m2[i] = 0.f;
                a[i] *= inv;  // slice mean
                const int64_t k = j * RS + i;
                if (k >= nrows) continue;
                const uint4 *xs = stage_of(k);
#pragma unroll
                for (int q = 0; q < VPT; ++q) {
                    const int lv = q * NT + t;
                    if (lv >= cnt) continue;
                    const uint4 x = lds128(xs + lv);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float d = vget<T>(x, e) - a[i];
                        m2[i] += d * d;
                    }
                }
            }
            tmac_cta_sum<RS>(m2, h, cpar);
#pragma unroll
            for (int i = 0; i < RS; ++i) {
                out[2 * i] = a[i];
                out[2 * i + 1] = m2[i];
            }
        } else {
#pragma unroll
            for (int i = 0; i < RS; ++i) {
                out[2 * i] = a[i];
                out[2 * i + 1] = 0.f;
            }
        }
    };

    float cur[NV], nxt[NV];
    if (nsteps > 0) {
        pass1(0, cur);
        tmac_send<CL, NV>(h, 0, rank, cur);
    }
    for (int64_t j = 0; j < nsteps; ++j) {
        const bool more = j + 1 < nsteps;
        if (more) pass1(j + 1, nxt);
        const int par = (int)(j & 1);
        mbar_wait_cluster_bounded(&h.xch[par], (uint32_t)((j >> 1) & 1), abort_flag, p.tc.fault);
#pragma unroll
        for (int i = 0; i < RS; ++i) {
            const int64_t k = j * RS + i;
            if (k >= nrows) continue;
            float mean = 0.f, m2 = 0.f;
            if constexpr (LN) {
                // Pairwise merge of the slices' (count, mean, M2), in rank order.
                float tot = 0.f;
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    const int64_t cc = nv - (int64_t)c * slice < slice ? nv - (int64_t)c * slice : slice;
                    tot += (float)(cc * E) * h.slot[par][c][2 * i];
                }
                mean = tot / n;
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    const int64_t cc = nv - (int64_t)c * slice < slice ? nv - (int64_t)c * slice : slice;
                    const float d = h.slot[par][c][2 * i] - mean;
                    m2 += h.slot[par][c][2 * i + 1] + (float)(cc * E) * d * d;
                }
            } else {
#pragma unroll
                for (int c = 0; c < CL; ++c) m2 += h.slot[par][c][2 * i];
            }
            const float rstd = rsqrtf(m2 / n + p.eps);
            const int64_t row = cid + k * ncl;
            if (rank == 0 && t == 0) {
                if (p.rstd) p.rstd[row] = rstd;
                if (LN && p.mean) p.mean[row] = mean;
            }
            const uint4 *xs = stage_of(k);
#pragma unroll
            for (int q = 0; q < VPT; ++q) {
                const int lv = q * NT + t;
                if (lv >= cnt) continue;
                const uint4 x = lds128(xs + lv);
                const uint4 g = p.gamma ? lds128(gs + lv) : ones_vec<T>();
                uint4 bb;
                if constexpr (LN) bb = p.beta ? lds128(bs + lv) : make_uint4(0, 0, 0, 0);
                float o[E];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    o[e] = ((vget<T>(x, e) - mean) * rstd) * vget<T>(g, e);
                    if constexpr (LN) o[e] += vget<T>(bb, e);
                }
                st_vec(p.y, row * nv + v0 + lv, vpack<T>(o));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&h.empty[k % S]);
        }
        if (more) {
#pragma unroll
            for (int i = 0; i < NV; ++i) cur[i] = nxt[i];
            tmac_send<CL, NV>(h, (int)((j + 1) & 1), rank, cur);
        }
    }
    // No CTA leaves while a peer could still write into its shared memory
    // (this matters only after an aborted wait; exited threads do not count).
    cluster_sync_all();
}

// ============================================================================ backward
template <typename T, bool LN, int VPT, int CL, int RS>
__global__ void __launch_bounds__((kTmacCW + 1) * 32, 1) bwd_tmac(const BwdParams p) {
    pdl_launch_dependents();  // the column reduce waits for this grid's completion
    constexpr int E = VecTraits<T>::E;
    constexpr int NT = kTmacNT;
    constexpr int NV = 2 * RS;
    static_assert(CL >= 2 && CL <= kTmacMaxCl && NV <= kTmacMaxVals, "cluster shape");
    extern __shared__ __align__(128) unsigned char smem[];
    TmacHeader &h = *reinterpret_cast<TmacHeader *>(smem);
    const int rank = (int)cluster_ctarank();
    const int64_t M = p.M, nv = p.N / E;
    const int64_t slice = (nv + CL - 1) / CL;
    const int64_t v0 = rank * slice;
    const int cnt = (int)(nv - v0 < slice ? nv - v0 : slice);
    const size_t row_bytes = (size_t)p.N * sizeof(T);
    const size_t slice_al = al128((size_t)slice * 16);
    uint4 *gs = reinterpret_cast<uint4 *>(smem + kTmaHeaderBytes);
    unsigned char *stages = smem + kTmaHeaderBytes + slice_al;
    const int S = p.tc.stages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&h.full[s], 1);
            mbar_init(&h.empty[s], kTmacCW);
        }
        mbar_init(&h.xch[0], CL);
        mbar_init(&h.xch[1], CL);
        mbar_init(&h.pbar, 1);
        h.abort = 0;
        fence_mbar_init();
    }
    cluster_sync_all();

    if (warp == kTmacCW) {
        if (lane == 0) {
            load_params(&h.pbar, gs, nullptr, p.gamma ? static_cast<const uint4 *>(p.gamma) + v0 : nullptr,
                        nullptr, (uint32_t)cnt * 16u);
            tmac_produce<true, LN>(h, stages, p.tc, M, row_bytes, v0, cnt, slice_al, p.x, p.dy, p.rstd,
                                   p.mean);
        }
        return;
    }

    const int t = threadIdx.x;
    mbar_wait_bounded(&h.pbar, 0, &h.abort, p.tc.fault);

    const int64_t cid = cluster_id_x(), ncl = cluster_count_x();
    const int64_t nrows = cid < M ? (M - cid + ncl - 1) / ncl : 0;
    const int64_t nsteps = (nrows + RS - 1) / RS;
    volatile int *abort_flag = &h.abort;
    const float n = (float)p.N;
    int cpar = 0;
    float accg[VPT][E], accb[LN ? VPT : 1][E];
#pragma unroll
    for (int q = 0; q < VPT; ++q)
#pragma unroll
        for (int e = 0; e < E; ++e) {
            accg[q][e] = 0.f;
            if constexpr (LN) accb[q][e] = 0.f;
        }

    auto stage_of = [&](int64_t k) { return stages + (size_t)(k % S) * p.tc.stride; };
    // Saved statistics of row k, from the stage's window or directly.
    auto stats = [&](int64_t k, float &rstd, float &mean) {
        const int64_t row = cid + k * ncl;
        int64_t wa, wb;
        stat_window(row, 1, M, &wa, &wb);
        const float *sd = reinterpret_cast<const float *>(stage_of(k) + 2 * slice_al);
        const bool in = row < wb;
        rstd = in ? sd[row - wa] : __ldg(p.rstd + row);
        mean = 0.f;
        if constexpr (LN) mean = in ? sd[4 + row - wa] : __ldg(p.mean + row);
    };
    // Local partials of step j: {sum g * xhat, sum g} per row.
    auto pass1 = [&](int64_t j, float (&out)[NV]) {
#pragma unroll
        for (int i = 0; i < RS; ++i) {
            out[2 * i] = 0.f;
            out[2 * i + 1] = 0.f;
            const int64_t k = j * RS + i;
            if (k >= nrows) continue;
            mbar_wait_bounded(&h.full[k % S], (uint32_t)((k / S) & 1), abort_flag, p.tc.fault);
            float rstd, mean;
            stats(k, rstd, mean);
            const unsigned char *tb = stage_of(k);
            const uint4 *xs = reinterpret_cast<const uint4 *>(tb);
            const uint4 *ds = reinterpret_cast<const uint4 *>(tb + slice_al);
#pragma unroll
            for (int q = 0; q < VPT; ++q) {
                const int lv = q * NT + t;
                if (lv >= cnt) continue;
                const uint4 x = lds128(xs + lv), d = lds128(ds + lv);
                const uint4 g = p.gamma ? lds128(gs + lv) : ones_vec<T>();
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float xh = (vget<T>(x, e) - mean) * rstd;
                    const float gg = vget<T>(d, e) * vget<T>(g, e);
                    out[2 * i] += gg * xh;
                    if constexpr (LN) out[2 * i + 1] += gg;
                }
            }
        }
        tmac_cta_sum<NV>(out, h, cpar);
    };

    float cur[NV], nxt[NV];
    if (nsteps > 0) {
        pass1(0, cur);
        tmac_send<CL, NV>(h, 0, rank, cur);
    }
    for (int64_t j = 0; j < nsteps; ++j) {
        const bool more = j + 1 < nsteps;
        if (more) pass1(j + 1, nxt);
        const int par = (int)(j & 1);
        mbar_wait_cluster_bounded(&h.xch[par], (uint32_t)((j >> 1) & 1), abort_flag, p.tc.fault);
#pragma unroll
        for (int i = 0; i < RS; ++i) {
            const int64_t k = j * RS + i;
            if (k >= nrows) continue;
            float s2 = 0.f, s1 = 0.f;
#pragma unroll
            for (int c = 0; c < CL; ++c) {
                s2 += h.slot[par][c][2 * i];
                if constexpr (LN) s1 += h.slot[par][c][2 * i + 1];
            }
            const float c2 = s2 / n, c1 = LN ? s1 / n : 0.f;
            float rstd, mean;
            stats(k, rstd, mean);
            const int64_t row = cid + k * ncl;
            const unsigned char *tb = stage_of(k);
            const uint4 *xs = reinterpret_cast<const uint4 *>(tb);
            const uint4 *ds = reinterpret_cast<const uint4 *>(tb + slice_al);
#pragma unroll
            for (int q = 0; q < VPT; ++q) {
                const int lv = q * NT + t;
                if (lv >= cnt) continue;
                const uint4 x = lds128(xs + lv), d = lds128(ds + lv);
                const uint4 g = p.gamma ? lds128(gs + lv) : ones_vec<T>();
                float o[E];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float xh = (vget<T>(x, e) - mean) * rstd;
                    const float dyv = vget<T>(d, e);
                    const float gg = dyv * vget<T>(g, e);
                    o[e] = rstd * (gg - c1 - xh * c2);
                    accg[q][e] += dyv * xh;
                    if constexpr (LN) accb[q][e] += dyv;
                }
                st_vec(p.dx, row * nv + v0 + lv, vpack<T>(o));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&h.empty[k % S]);
        }
        if (more) {
#pragma unroll
            for (int i = 0; i < NV; ++i) cur[i] = nxt[i];
            tmac_send<CL, NV>(h, (int)((j + 1) & 1), rank, cur);
        }
    }
    cluster_sync_all();  // see the forward

    // This CTA's slice of the cluster's partial row (P = clusters).
    float *wsg = p.ws + cid * p.N;
    float *wsb = p.ws + (ncl + cid) * p.N;
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
        const int lv = q * NT + t;
        if (lv >= cnt) continue;
        const int64_t c0 = (v0 + lv) * E;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            wsg[c0 + e] = accg[q][e];
            if constexpr (LN) wsb[c0 + e] = accb[q][e];
        }
    }
}

}  // namespace gbn
