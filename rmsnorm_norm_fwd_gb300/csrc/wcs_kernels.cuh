// wcs_kernels.cuh -- RMSNorm / LayerNorm forward and backward for wide rows
// (16K-128K elements): each row is split across the CL CTAs of a
// thread-block cluster, and every CTA's column slice of each row is brought
// into its shared memory by one bulk asynchronous copy per tensor and read
// from there by both passes.  DRAM sees every element once (x, or x and dy,
// in; y or dx out); the second pass reads shared memory instead of L2, and
// the bytes in flight sit in the ring, not in registers.
//
// Same arithmetic as the other kernels (the definitions on "SOTA
// normalization performance with torch.compile", section "How Did
// Torch.compile Catch Quack?", and "Fused RMSNorm", sections "What it is" /
// "How it works"); the torch.compile page's remark that very wide rows lose
// without distributed shared memory is what the cluster split answers.
//
// Per CTA: NT threads, one CTA per SM; thread t owns vectors t, t + NT, ...
// (at most VPT) of the slice.  gamma (and beta) of the slice are bulk-copied
// once in their storage type.  A ring of S stages holds whole slices of
// consecutive rows of the CTA (row k in stage k % S); thread 0 issues the
// copies: the first S rows up front, then row k + S as soon as every warp
// has arrived on stage k's "empty" barrier after its last read of row k.
//
// Schedule per CTA, rows k = 0, 1, ... of its cluster: pass 1 of row k + 1
// (this thread's partials, then the CTA's, then sent to every CTA of the
// cluster), then the exchange of row k is collected, then pass 2 of row k.
// So row k's exchange has a whole pass 1 to complete, and the copies of rows
// k + 2 ... k + S - 1 are in flight meanwhile.
//
// Exchange (as in wide_kernels.cuh): each CTA writes its partials of row k
// into slot [k % 4][rank] of every CTA (st.shared::cluster) and arrives, with
// release semantics, on that CTA's barrier xch[k % 4]; a CTA waits (acquire,
// bounded) for CL arrivals, then combines the CL partials in rank order, so
// every CTA gets identical bits.  Slot reuse: a CTA sends row k + 4 only
// after it has collected row k + 2, which every peer sends after a CTA
// barrier that follows its own reads of row k's slots.
//
// LayerNorm forward statistics: per thread (count, mean, M2) of its elements
// (two passes over its registers), then the group combine of Chan, Golub and
// LeVeque over the lanes, the warps and the CTAs of the cluster (exact
// algebra; no E[x^2] - mean^2 cancellation).
//
// Every wait is bounded (mbar_wait_bounded / mbar_wait_cluster_bounded): on a
// timeout the CTA raises its abort flag and the device fault word, skips the
// remaining waits and runs to its end; thread 0 then waits (bounded) for the
// copies it issued, and the final cluster barrier keeps every CTA resident
// until its peers are done writing into it.
#pragma once

#include "device_common.cuh"
#include "params.h"
#include "tma_kernels.cuh"
#include "wide_kernels.cuh"

namespace gbn {

constexpr int kWcsMaxStages = 8;
constexpr int kWcsSlots = 4;

// Bytes of one tensor's slice in shared memory.
__host__ __device__ inline size_t wcs_slice_bytes(int64_t slice_vecs) { return ex_al128((size_t)slice_vecs * 16u); }

// Shared state of the wcs kernels (static shared memory).
template <int W, int CL, int NV>
struct WcsShared {
    uint64_t full[kWcsMaxStages];
    uint64_t empty[kWcsMaxStages];
    uint64_t xch[kWcsSlots];
    uint64_t pbar;
    int abort;
    float red[2][3][W];
    float slot[kWcsSlots][CL][NV];
};

// Thread 0: bulk copy of this CTA's slice of row `row` of each tensor into
// stage s, counted on full[s].
__device__ __forceinline__ void wcs_issue(uint64_t *full, unsigned char *stage, size_t slice_b, const void *t0,
                                          const void *t1, int64_t row, int64_t nv, int64_t v0, int cnt) {
    const uint32_t bytes = (uint32_t)cnt * 16u;
    mbar_arrive_expect_tx(full, bytes * (t1 ? 2u : 1u));
    bulk_g2s(stage, static_cast<const uint4 *>(t0) + row * nv + v0, bytes, full);
    if (t1) bulk_g2s(stage + slice_b, static_cast<const uint4 *>(t1) + row * nv + v0, bytes, full);
}

// Sends this CTA's NV partials of row k to every CTA of the cluster (threads
// t < CL, one peer each).
template <int CL, int NV>
__device__ __forceinline__ void wcs_send(float (&slot)[kWcsSlots][CL][NV], uint64_t *xch, int64_t k, int rank,
                                         const float (&v)[NV]) {
    const int t = threadIdx.x;
    if (t < CL) {
        const int sp = (int)(k % kWcsSlots);
        const uint32_t dst = map_to_rank(smem_u32(&slot[sp][rank][0]), (uint32_t)t);
#pragma unroll
        for (int i = 0; i < NV; ++i) st_cluster_f32(dst + 4u * i, v[i]);
        mbar_arrive_remote(map_to_rank(smem_u32(&xch[sp]), (uint32_t)t));
    }
}

// ============================================================================ forward
template <typename T, bool LN, int NT, int VPT, int CL>
__global__ void __launch_bounds__(NT, 1) fwd_wcs(const FwdParams p) {
    constexpr int E = VecTraits<T>::E;
    constexpr int W = NT / 32;
    constexpr int NV = LN ? 3 : 1;  // exchanged: (count, mean, M2) or the sum of squares
    static_assert(NT % 32 == 0 && NT <= 1024 && CL >= 2 && CL <= 16, "shape");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ WcsShared<W, CL, NV> sh;

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int rank = (int)cluster_ctarank();
    const int64_t cid = cluster_id_x(), ncl = cluster_count_x();
    const int64_t M = p.M, nv = p.N / E;
    const int64_t slice = (nv + CL - 1) / CL, v0 = rank * slice;
    const int cnt = (int)(nv - v0 < slice ? nv - v0 : slice);  // > 0 (host geometry)
    const size_t slice_b = wcs_slice_bytes(slice);
    unsigned char *gsm = smem, *bsm = smem + slice_b;  // gamma, beta slices (storage type)
    unsigned char *stages = smem + slice_b * (LN ? 2 : 1);
    const int S = p.tc.stages;
    const size_t stride = p.tc.stride;
    const int64_t nrows = cid < M ? (M - cid + ncl - 1) / ncl : 0;
    auto row_of = [&](int64_t k) { return cid + k * ncl; };
    const float n = (float)p.N;
    volatile int *abort_flag = &sh.abort;
    int issued = 0;

    if (t == 0) {
        sh.abort = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], W);
        }
        for (int j = 0; j < kWcsSlots; ++j) mbar_init(&sh.xch[j], CL);
        mbar_init(&sh.pbar, 1);
        fence_mbar_init();
    }
    cluster_sync_all();  // every CTA's barriers exist before any peer arrives on them
    if (t == 0) {
        const uint4 *g = static_cast<const uint4 *>(p.gamma), *b = static_cast<const uint4 *>(p.beta);
        load_params(&sh.pbar, gsm, bsm, g ? g + v0 : nullptr, (LN && b) ? b + v0 : nullptr, (uint32_t)cnt * 16u);
        for (int64_t k = 0; k < nrows && k < S; ++k, ++issued)
            wcs_issue(&sh.full[k], stages + k * stride, slice_b, p.x, nullptr, row_of(k), nv, v0, cnt);
    }
    mbar_wait_bounded(&sh.pbar, 0, abort_flag, p.tc.fault);
    const bool has_g = p.gamma != nullptr, has_b = LN && p.beta != nullptr;

    // pass 1 of row k: this CTA's partials, combined over the CTA, sent out
    auto pass1 = [&](int64_t k) {
        const int s = (int)(k % S);
        mbar_wait_bounded(&sh.full[s], (uint32_t)((k / S) & 1), abort_flag, p.tc.fault);
        const uint4 *xs = reinterpret_cast<const uint4 *>(stages + s * stride);
        float v[NV];
        float (*buf)[3][W] = sh.red;
        const int par = (int)(k & 1);
        if constexpr (!LN) {
            float2 a = f2s(0.f);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int lv = j * NT + t;
                if (lv < cnt) {
                    const uint4 q = lds128(xs + lv);
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) {
                        const float2 f = vpair<T>(q, e);
                        a = f2fma(f, f, a);
                    }
                }
            }
            float acc = a.x + a.y;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) buf[par][0][warp] = acc;
            __syncthreads();
            acc = 0.f;
#pragma unroll 4
            for (int w = 0; w < W; ++w) acc += buf[par][0][w];
            v[0] = acc;
        } else {
            // this thread's (count, mean, M2), two passes over its elements
            float2 a = f2s(0.f);
            int nb = 0;
            uint4 q[VPT];
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int lv = j * NT + t;
                q[j] = lv < cnt ? lds128(xs + lv) : make_uint4(0, 0, 0, 0);
                if (lv < cnt) {
                    nb += E;
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) a = f2add(a, vpair<T>(q[j], e));
                }
            }
            float cnt_t = (float)nb;
            float mean = nb > 0 ? __fdiv_rn(a.x + a.y, cnt_t) : 0.f;
            const float2 nm = f2s(-mean);
            float2 m2 = f2s(0.f);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                if (j * NT + t < cnt) {
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) {
                        const float2 d = f2add(vpair<T>(q[j], e), nm);
                        m2 = f2fma(d, d, m2);
                    }
                }
            }
            float acc = m2.x + m2.y;
            warp_combine(cnt_t, mean, acc);
            if (lane == 0) {
                buf[par][0][warp] = cnt_t;
                buf[par][1][warp] = mean;
                buf[par][2][warp] = acc;
            }
            __syncthreads();
            // the same group combine over the warps, in warp order
            float tn = 0.f, ts = 0.f;
#pragma unroll 4
            for (int w = 0; w < W; ++w) {
                tn += buf[par][0][w];
                ts += buf[par][0][w] * buf[par][1][w];
            }
            const float mu = ts / tn;  // tn > 0: every CTA has columns
            float a2 = 0.f;
#pragma unroll 4
            for (int w = 0; w < W; ++w) {
                const float d = buf[par][1][w] - mu;
                a2 += buf[par][2][w] + buf[par][0][w] * (d * d);
            }
            v[0] = tn;
            v[1] = mu;
            v[2] = a2;
        }
        wcs_send<CL, NV>(sh.slot, sh.xch, k, rank, v);
    };
    // the exchange of row k: (mean, rstd), identical bits in every CTA
    auto recv = [&](int64_t k, float &mean, float &rstd) {
        const int sp = (int)(k % kWcsSlots);
        mbar_wait_cluster_bounded(&sh.xch[sp], (uint32_t)((k / kWcsSlots) & 1), abort_flag, p.tc.fault);
        if constexpr (!LN) {
            float s = 0.f;
#pragma unroll
            for (int c = 0; c < CL; ++c) s += sh.slot[sp][c][0];
            mean = 0.f;
            rstd = rsqrtf(s / n + p.eps);
        } else {
            float tn = 0.f, ts = 0.f;
#pragma unroll
            for (int c = 0; c < CL; ++c) {
                tn += sh.slot[sp][c][0];
                ts += sh.slot[sp][c][0] * sh.slot[sp][c][1];
            }
            const float mu = ts / tn;
            float a2 = 0.f;
#pragma unroll
            for (int c = 0; c < CL; ++c) {
                const float d = sh.slot[sp][c][1] - mu;
                a2 += sh.slot[sp][c][2] + sh.slot[sp][c][0] * (d * d);
            }
            mean = mu;
            rstd = rsqrtf(a2 / n + p.eps);
        }
    };

    if (nrows > 0) pass1(0);
    for (int64_t k = 0; k < nrows; ++k) {
        if (k + 1 < nrows) pass1(k + 1);
        float mean, rstd;
        recv(k, mean, rstd);
        const int64_t row = row_of(k);
        if (rank == 0 && t == 0) {
            if (p.rstd) p.rstd[row] = rstd;
            if (LN && p.mean) p.mean[row] = mean;
        }
        // pass 2: y = (x - mean) rstd gamma (+ beta) from the staged slice
        const int s = (int)(k % S);
        const uint4 *xs = reinterpret_cast<const uint4 *>(stages + s * stride);
        uint4 *yr = static_cast<uint4 *>(p.y) + row * nv + v0;
        const float2 nm = f2s(-mean), rs = f2s(rstd);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int lv = j * NT + t;
            if (lv >= cnt) continue;
            const uint4 q = lds128(xs + lv);
            const uint4 g = has_g ? lds128(reinterpret_cast<const uint4 *>(gsm) + lv) : ones_vec<T>();
            uint4 b = make_uint4(0, 0, 0, 0);
            if (has_b) b = lds128(reinterpret_cast<const uint4 *>(bsm) + lv);
            float2 o[E / 2];
#pragma unroll
            for (int e = 0; e < E / 2; ++e) {
                o[e] = f2mul(f2mul(f2add(vpair<T>(q, e), nm), rs), vpair<T>(g, e));
                if constexpr (LN) o[e] = f2add(o[e], vpair<T>(b, e));
            }
            st_vec(yr, lv, vpack2<T>(o));
        }
        // stage s is free once every warp is past its reads: refill it
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[s]);
        if (t == 0 && k + S < nrows) {
            mbar_wait_bounded(&sh.empty[s], (uint32_t)((k / S) & 1), abort_flag, p.tc.fault);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (!*abort_flag) {
                wcs_issue(&sh.full[s], stages + s * stride, slice_b, p.x, nullptr, row_of(k + S), nv, v0, cnt);
                ++issued;
            }
        }
    }
    if (t == 0 && *abort_flag) {
        // copies still landing after an aborted wait: wait for each (bounded)
        int zero = 0;
        for (int j = issued > S ? issued - S : 0; j < issued; ++j)
            mbar_wait_bounded(&sh.full[j % S], (uint32_t)((j / S) & 1), reinterpret_cast<volatile int *>(&zero),
                              nullptr);
    }
    // no CTA leaves while a peer could still write into its shared memory
    cluster_sync_all();
}

// ============================================================================ backward
template <typename T, bool LN, int NT, int VPT, int CL>
__global__ void __launch_bounds__(NT, 1) bwd_wcs(const BwdParams p) {
    pdl_launch_dependents();  // the column reduce waits for this grid's completion
    constexpr int E = VecTraits<T>::E;
    constexpr int W = NT / 32;
    constexpr int NV = LN ? 2 : 1;  // exchanged: sum g xhat (and sum g)
    static_assert(NT % 32 == 0 && NT <= 1024 && CL >= 2 && CL <= 16, "shape");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ WcsShared<W, CL, NV> sh;

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int rank = (int)cluster_ctarank();
    const int64_t cid = cluster_id_x(), ncl = cluster_count_x();
    const int64_t M = p.M, nv = p.N / E;
    const int64_t slice = (nv + CL - 1) / CL, v0 = rank * slice;
    const int cnt = (int)(nv - v0 < slice ? nv - v0 : slice);  // > 0 (host geometry)
    const size_t slice_b = wcs_slice_bytes(slice);
    unsigned char *gsm = smem;  // gamma slice (storage type)
    unsigned char *stages = smem + slice_b;  // stage: x slice, then dy slice
    const int S = p.tc.stages;
    const size_t stride = p.tc.stride;
    const int64_t nrows = cid < M ? (M - cid + ncl - 1) / ncl : 0;
    auto row_of = [&](int64_t k) { return cid + k * ncl; };
    const float n = (float)p.N;
    volatile int *abort_flag = &sh.abort;
    int issued = 0;

    if (t == 0) {
        sh.abort = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], W);
        }
        for (int j = 0; j < kWcsSlots; ++j) mbar_init(&sh.xch[j], CL);
        mbar_init(&sh.pbar, 1);
        fence_mbar_init();
    }
    cluster_sync_all();
    if (t == 0) {
        const uint4 *g = static_cast<const uint4 *>(p.gamma);
        load_params(&sh.pbar, gsm, nullptr, g ? g + v0 : nullptr, nullptr, (uint32_t)cnt * 16u);
        for (int64_t k = 0; k < nrows && k < S; ++k, ++issued)
            wcs_issue(&sh.full[k], stages + k * stride, slice_b, p.x, p.dy, row_of(k), nv, v0, cnt);
    }
    mbar_wait_bounded(&sh.pbar, 0, abort_flag, p.tc.fault);
    const bool has_g = p.gamma != nullptr;
    auto gam = [&](int lv) {
        return has_g ? lds128(reinterpret_cast<const uint4 *>(gsm) + lv) : ones_vec<T>();
    };

    // dgamma (and dbeta) sums of this thread's columns, as pairs
    float2 accg[VPT][E / 2], accb[LN ? VPT : 1][E / 2];
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
        for (int e = 0; e < E / 2; ++e) {
            accg[j][e] = f2s(0.f);
            if constexpr (LN) accb[j][e] = f2s(0.f);
        }

    // pass 1 of row k: rstd sum g (x - mean) (and sum g), g = dy gamma, over
    // the CTA, sent out
    auto pass1 = [&](int64_t k) {
        const int s = (int)(k % S);
        const int64_t row = row_of(k);
        const float rstd = __ldg(p.rstd + row);
        const float2 nm = f2s(LN ? -__ldg(p.mean + row) : 0.f);
        mbar_wait_bounded(&sh.full[s], (uint32_t)((k / S) & 1), abort_flag, p.tc.fault);
        const uint4 *xs = reinterpret_cast<const uint4 *>(stages + s * stride);
        const uint4 *ds = reinterpret_cast<const uint4 *>(stages + s * stride + slice_b);
        float2 a2 = f2s(0.f), a1 = f2s(0.f);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int lv = j * NT + t;
            if (lv >= cnt) continue;
            const uint4 q = lds128(xs + lv), d = lds128(ds + lv), g = gam(lv);
#pragma unroll
            for (int e = 0; e < E / 2; ++e) {
                const float2 gg = f2mul(vpair<T>(d, e), vpair<T>(g, e));
                a2 = f2fma(gg, f2add(vpair<T>(q, e), nm), a2);
                if constexpr (LN) a1 = f2add(a1, gg);
            }
        }
        float v[NV];
        v[0] = (a2.x + a2.y) * rstd;
        if constexpr (LN) v[NV - 1] = a1.x + a1.y;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1)
#pragma unroll
            for (int i = 0; i < NV; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
        const int par = (int)(k & 1);
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < NV; ++i) sh.red[par][i][warp] = v[i];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            float s2 = 0.f;
#pragma unroll 4
            for (int w = 0; w < W; ++w) s2 += sh.red[par][i][w];
            v[i] = s2;
        }
        wcs_send<CL, NV>(sh.slot, sh.xch, k, rank, v);
    };

    if (nrows > 0) pass1(0);
    for (int64_t k = 0; k < nrows; ++k) {
        if (k + 1 < nrows) pass1(k + 1);
        // the exchange of row k
        const int sp = (int)(k % kWcsSlots);
        mbar_wait_cluster_bounded(&sh.xch[sp], (uint32_t)((k / kWcsSlots) & 1), abort_flag, p.tc.fault);
        float tot[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            tot[i] = 0.f;
#pragma unroll
            for (int c = 0; c < CL; ++c) tot[i] += sh.slot[sp][c][i];
        }
        const int64_t row = row_of(k);
        const float rstd = __ldg(p.rstd + row);
        const float mean = LN ? __ldg(p.mean + row) : 0.f;
        // dx = rstd g - rstd c1 - (rstd c2) xhat, c1 = sum g / n, c2 = sum g xhat / n
        const float rc1 = LN ? rstd * (tot[NV - 1] / n) : 0.f, rc2 = rstd * (tot[0] / n);
        const float2 nm = f2s(-mean), r2 = f2s(rstd), nrc1 = f2s(-rc1), nrc2 = f2s(-rc2);
        const int s = (int)(k % S);
        const uint4 *xs = reinterpret_cast<const uint4 *>(stages + s * stride);
        const uint4 *ds = reinterpret_cast<const uint4 *>(stages + s * stride + slice_b);
        uint4 *dxr = static_cast<uint4 *>(p.dx) + row * nv + v0;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int lv = j * NT + t;
            if (lv >= cnt) continue;
            const uint4 q = lds128(xs + lv), d = lds128(ds + lv), g = gam(lv);
            float2 o[E / 2];
#pragma unroll
            for (int e = 0; e < E / 2; ++e) {
                const float2 xh = f2mul(f2add(vpair<T>(q, e), nm), r2);
                const float2 dyv = vpair<T>(d, e);
                o[e] = f2fma(nrc2, xh, f2fma(r2, f2mul(dyv, vpair<T>(g, e)), nrc1));
                accg[j][e] = f2fma(dyv, xh, accg[j][e]);
                if constexpr (LN) accb[j][e] = f2add(accb[j][e], dyv);
            }
            st_vec(dxr, lv, vpack2<T>(o));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[s]);
        if (t == 0 && k + S < nrows) {
            mbar_wait_bounded(&sh.empty[s], (uint32_t)((k / S) & 1), abort_flag, p.tc.fault);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (!*abort_flag) {
                wcs_issue(&sh.full[s], stages + s * stride, slice_b, p.x, p.dy, row_of(k + S), nv, v0, cnt);
                ++issued;
            }
        }
    }
    if (t == 0 && *abort_flag) {
        int zero = 0;
        for (int j = issued > S ? issued - S : 0; j < issued; ++j)
            mbar_wait_bounded(&sh.full[j % S], (uint32_t)((j / S) & 1), reinterpret_cast<volatile int *>(&zero),
                              nullptr);
    }
    cluster_sync_all();

    // this CTA's slice of the cluster's partial row (P = clusters)
    float *wsg = p.ws + cid * p.N + v0 * E;
    float *wsb = p.ws + (ncl + cid) * p.N + v0 * E;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int lv = j * NT + t;
        if (lv >= cnt) continue;
#pragma unroll
        for (int h = 0; h < E / 4; ++h) {
            reinterpret_cast<float4 *>(wsg + (int64_t)lv * E)[h] =
                make_float4(accg[j][2 * h].x, accg[j][2 * h].y, accg[j][2 * h + 1].x, accg[j][2 * h + 1].y);
            if constexpr (LN)
                reinterpret_cast<float4 *>(wsb + (int64_t)lv * E)[h] =
                    make_float4(accb[j][2 * h].x, accb[j][2 * h].y, accb[j][2 * h + 1].x, accb[j][2 * h + 1].y);
        }
    }
}

}  // namespace gbn
