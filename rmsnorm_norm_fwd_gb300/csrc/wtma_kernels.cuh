// wtma_kernels.cuh -- RMSNorm / LayerNorm forward for wide rows: one CTA per
// row at a time, the row streamed twice through a shared-memory ring by bulk
// asynchronous copies.
//
// Same arithmetic as norm_kernels.cuh (the definitions on "SOTA normalization
// performance with torch.compile", section "How Did Torch.compile Catch
// Quack?", and "Fused RMSNorm", sections "What it is" / "How it works").  The
// torch.compile page reports the large-N regression of kernels that cannot
// keep a wide row on chip; here a row of any length is read from DRAM once
// for its statistics (pass 1, copies marked L2 evict_last) and a second time
// from L2 for the output (pass 2, evict_first), and the TMA engine keeps up to
// kTmaMaxStages stages of either pass in flight, so neither pass waits on
// memory latency the way register-held loads do.
//
// The row is cut into chunks of CV = NT * U 16-byte vectors (thread t of the
// NT consumers handles vectors t + u * NT of every chunk: conflict-free
// shared-memory reads and 512-byte runs per warp for the stores).  Every
// stage holds NP + 1 chunks (NP = 1 for RMSNorm, 2 for LayerNorm): a pass-1
// job copies NP + 1 consecutive chunks of x; a pass-2 job copies one chunk of
// x with the same chunk of gamma (and beta), which every row needs again and
// which stay in L2.  One producer warp issues the jobs in order (pass 1 of row
// r, pass 2 of row r, pass 1 of the next row, ...) as stages free up, so the
// copies of pass 2 and of the next row are already landing while the
// consumers reduce a row's statistics.
//
// LayerNorm statistics: per job each thread forms the exact (count, mean,
// M2) of its elements, folds it into a running triple with the pairwise
// update of Chan, Golub and LeVeque, and the consumers combine their triples
// with the same update at the end of pass 1.
//
// Waits are bounded (mbar_wait_bounded): on a timeout the CTA raises its
// abort flag and the device fault word, skips later waits and ends; the
// producer waits (bounded) for its copies in flight before it exits.
#pragma once

#include "device_common.cuh"
#include "params.h"
#include "tma_kernels.cuh"
#include "wide_kernels.cuh"

namespace gbn {

// Bulk copy global -> shared with an L2 eviction policy (createpolicy).
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

struct WtmaHeader {
    uint64_t full[kTmaMaxStages];
    uint64_t empty[kTmaMaxStages];
    int abort;
    int pad;
    float red[2][3][32];  // [parity][value][consumer warp]
};
static_assert(sizeof(WtmaHeader) <= kTmaHeaderBytes, "header layout");

template <typename T, bool LN, int CW, int U>
__global__ void __launch_bounds__((CW + 1) * 32, 1) fwd_wtma(const FwdParams p) {
    constexpr int E = VecTraits<T>::E;
    constexpr int NT = CW * 32;
    constexpr int CV = NT * U;           // vectors per chunk
    constexpr int NP = LN ? 2 : 1;       // parameter rows
    constexpr int CPJ = NP + 1;          // chunks per stage
    static_assert(CW >= 1 && CW <= 32, "consumer warps");
    extern __shared__ __align__(128) unsigned char smem[];
    WtmaHeader &h = *reinterpret_cast<WtmaHeader *>(smem);
    unsigned char *ring = smem + kTmaHeaderBytes;
    const int S = p.tc.stages;
    const int64_t M = p.M, nv = p.N / E;
    const int64_t nch = (nv + CV - 1) / CV;     // chunks per row
    const int64_t nj1 = (nch + CPJ - 1) / CPJ;  // pass-1 jobs per row
    const int64_t jobs_per_row = nj1 + nch;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &h.abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&h.full[s], 1);
            mbar_init(&h.empty[s], CW);
        }
        h.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const int64_t my_rows = blockIdx.x < M ? (M - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int64_t njobs = my_rows * jobs_per_row;
    constexpr uint32_t kChunkBytes = CV * 16;
    const uint32_t stage_bytes = p.tc.stride;

    if (warp == CW) {
        // ---- producer
        if (lane == 0) {
            const uint64_t keep = l2_policy_keep(), drop = l2_policy_drop();
            const unsigned char *x = static_cast<const unsigned char *>(p.x);
            int64_t issued = 0;
            for (int64_t j = 0; j < njobs; ++j, ++issued) {
                const int s = (int)(j % S);
                if (j >= S) mbar_wait_bounded(&h.empty[s], (uint32_t)(((j / S) - 1) & 1), abort_flag, p.tc.fault);
                if (*abort_flag) break;
                const int64_t row = blockIdx.x + (j / jobs_per_row) * (int64_t)gridDim.x;
                const int64_t q = j % jobs_per_row;
                unsigned char *dst = ring + (size_t)s * stage_bytes;
                const unsigned char *xr = x + (size_t)row * (size_t)nv * 16;
                if (q < nj1) {
                    // pass 1: chunks q * CPJ .. of x
                    const int64_t v0 = q * CPJ * CV;
                    const int64_t vn = nv - v0 < (int64_t)CPJ * CV ? nv - v0 : (int64_t)CPJ * CV;
                    const uint32_t bytes = (uint32_t)vn * 16u;
                    mbar_arrive_expect_tx(&h.full[s], bytes);
                    bulk_g2s_hint(dst, xr + v0 * 16, bytes, &h.full[s], keep);
                } else {
                    // pass 2: chunk c of x, gamma (and beta)
                    const int64_t c = q - nj1;
                    const int64_t v0 = c * CV;
                    const int64_t vn = nv - v0 < (int64_t)CV ? nv - v0 : (int64_t)CV;
                    const uint32_t bytes = (uint32_t)vn * 16u;
                    const int npar = (p.gamma ? 1 : 0) + ((LN && p.beta) ? 1 : 0);
                    mbar_arrive_expect_tx(&h.full[s], bytes * (1u + (uint32_t)npar));
                    bulk_g2s_hint(dst, xr + v0 * 16, bytes, &h.full[s], drop);
                    if (p.gamma)
                        bulk_g2s_hint(dst + kChunkBytes, static_cast<const unsigned char *>(p.gamma) + v0 * 16,
                                      bytes, &h.full[s], keep);
                    if (LN && p.beta)
                        bulk_g2s_hint(dst + 2 * kChunkBytes, static_cast<const unsigned char *>(p.beta) + v0 * 16,
                                      bytes, &h.full[s], keep);
                }
            }
            if (*abort_flag) {
                // copies issued may still be landing: wait for each (bounded) before exiting
                int zero = 0;
                for (int64_t j = issued > S ? issued - S : 0; j < issued; ++j)
                    mbar_wait_bounded(&h.full[j % S], (uint32_t)((j / S) & 1),
                                      reinterpret_cast<volatile int *>(&zero), nullptr);
            }
        }
        return;
    }

    // ---- consumers
    const int t = threadIdx.x;
    const float n = (float)p.N;
    int parity = 0;
    int64_t j = 0;  // job index, in the producer's order
    for (int64_t k = 0; k < my_rows; ++k) {
        const int64_t row = blockIdx.x + k * (int64_t)gridDim.x;
        // pass 1: statistics
        float acc[4] = {0.f, 0.f, 0.f, 0.f};   // RMS: sum of squares chains
        float cnt = 0.f, mean = 0.f, m2 = 0.f;  // LN: running (count, mean, M2)
        for (int64_t q = 0; q < nj1; ++q, ++j) {
            const int s = (int)(j % S);
            mbar_wait_bounded(&h.full[s], (uint32_t)((j / S) & 1), abort_flag, p.tc.fault);
            const uint4 *xs = reinterpret_cast<const uint4 *>(ring + (size_t)s * stage_bytes);
            const int64_t v0 = q * CPJ * CV;
            float ps = 0.f;
            int nb = 0;
            uint4 xv[CPJ * U];
#pragma unroll
            for (int i = 0; i < CPJ * U; ++i) {
                const int lv = i * NT + t;
                const bool ok = v0 + lv < nv;
                xv[i] = ok ? lds128(xs + lv) : make_uint4(0, 0, 0, 0);
                if (ok) nb += E;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float f = vget<T>(xv[i], e);
                    if constexpr (LN) ps += f;
                    else acc[(i * E + e) & 3] += f * f;
                }
            }
            if constexpr (LN) {
                if (nb > 0) {
                    const float fb = (float)nb;
                    const float mb = __fdiv_rn(ps, fb);
                    float pm = 0.f;
#pragma unroll
                    for (int i = 0; i < CPJ * U; ++i) {
                        if (v0 + i * NT + t >= nv) continue;
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            const float d = vget<T>(xv[i], e) - mb;
                            pm += d * d;
                        }
                    }
                    if (cnt == 0.f) {
                        cnt = fb;
                        mean = mb;
                        m2 = pm;
                    } else {
                        const float tot = cnt + fb;
                        const float d = mb - mean;
                        const float rr = __fdiv_rn(fb, tot);
                        mean += d * rr;
                        m2 += pm + d * d * cnt * rr;
                        cnt = tot;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&h.empty[s]);
        }
        // CTA reduction over the NT consumers (identical bits in all)
        float rstd;
        if constexpr (!LN) {
            float a = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (lane == 0) h.red[parity][0][warp] = a;
            named_sync(1, NT);
            float s2 = 0.f;
#pragma unroll 4
            for (int w = 0; w < CW; ++w) s2 += h.red[parity][0][w];
            rstd = rsqrtf(s2 / n + p.eps);
            mean = 0.f;
        } else {
            warp_combine(cnt, mean, m2);
            if (lane == 0) {
                h.red[parity][0][warp] = cnt;
                h.red[parity][1][warp] = mean;
                h.red[parity][2][warp] = m2;
            }
            named_sync(1, NT);
            float tn = 0.f, ts = 0.f;
#pragma unroll 4
            for (int w = 0; w < CW; ++w) {
                tn += h.red[parity][0][w];
                ts += h.red[parity][0][w] * h.red[parity][1][w];
            }
            mean = ts / tn;  // tn = N > 0
            float a2 = 0.f;
#pragma unroll 4
            for (int w = 0; w < CW; ++w) {
                const float d = h.red[parity][1][w] - mean;
                a2 += h.red[parity][2][w] + h.red[parity][0][w] * (d * d);
            }
            rstd = rsqrtf(a2 / n + p.eps);
        }
        parity ^= 1;
        if (t == 0) {
            if (p.rstd) p.rstd[row] = rstd;
            if (LN && p.mean) p.mean[row] = mean;
        }
        // pass 2: y = ((x - mean) * rstd) * gamma (+ beta), x from L2
        const uint64_t drop = l2_policy_drop();
        uint4 *yr = static_cast<uint4 *>(p.y) + row * nv;
        for (int64_t c = 0; c < nch; ++c, ++j) {
            const int s = (int)(j % S);
            mbar_wait_bounded(&h.full[s], (uint32_t)((j / S) & 1), abort_flag, p.tc.fault);
            const uint4 *xs = reinterpret_cast<const uint4 *>(ring + (size_t)s * stage_bytes);
            const uint4 *gs = xs + CV;
            const uint4 *bs = xs + 2 * CV;
            const int64_t v0 = c * CV;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int lv = u * NT + t;
                if (v0 + lv >= nv) continue;
                const uint4 q = lds128(xs + lv);
                const uint4 g = p.gamma ? lds128(gs + lv) : ones_vec<T>();
                uint4 b = make_uint4(0, 0, 0, 0);
                if constexpr (LN) b = p.beta ? lds128(bs + lv) : make_uint4(0, 0, 0, 0);
                float o[E];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    o[e] = ((vget<T>(q, e) - mean) * rstd) * vget<T>(g, e);
                    if constexpr (LN) o[e] += vget<T>(b, e);
                }
                st_l2hint(yr + v0 + lv, vpack<T>(o), drop);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&h.empty[s]);
        }
    }
}

}  // namespace gbn

namespace gbn {

// ============================================================================ backward
// Wide rows, backward: a cluster of CL CTAs shares each row, CTA `rank`
// owning a column slice of SL = ceil(nv / CL) 16-byte vectors, cut into K
// chunks of NT vectors; consumer thread t owns vector k * NT + t of every
// chunk, for every row the cluster visits, so its dgamma/dbeta sums (K * E
// floats each) stay in registers (gamma of the slice sits in shared memory,
// read by each thread at its own vectors: registers are the limit here).  The
// slice of each row is streamed twice through the bulk-copy ring (x and dy
// chunks per stage): pass 1 from DRAM (evict_last) for the partial sums
// sum g (x - mean) and sum g, which the CTA reduces and sends to every CTA
// of the cluster through distributed shared memory; pass 2 from L2
// (evict_first) for dx and the sums.  The order of the passes, the same for
// producer and consumers, is P1(0), then for i = 1..n: P1(i) (if any) and
// P2(i - 1), so each row's exchange has a whole pass of the next row to
// complete.  Exchange slots and barriers are reused every fourth row, as in
// bwd_wide (a peer sends row k + 4 only after receiving row k + 2 from this
// CTA, which this CTA sends after a CTA barrier that follows its reads of
// row k's slots).
template <typename T, bool LN, int CL, int K>
__global__ void __launch_bounds__(17 * 32, 1) bwd_wtma(const BwdParams p) {
    pdl_launch_dependents();  // the column reduce waits for this grid's completion
    constexpr int E = VecTraits<T>::E;
    constexpr int CW = 16;
    constexpr int NT = CW * 32;
    constexpr int NVAL = LN ? 2 : 1;
    constexpr int NS = 4;  // exchange slots
    static_assert(CL >= 1 && CL <= 16, "cluster size");
    extern __shared__ __align__(128) unsigned char smem[];
    WtmaHeader &h = *reinterpret_cast<WtmaHeader *>(smem);
    uint4 *gs = reinterpret_cast<uint4 *>(smem + kTmaHeaderBytes);  // gamma of the slice, [K * NT]
    unsigned char *ring = smem + kTmaHeaderBytes + (size_t)K * NT * 16;
    __shared__ float slot[NS][CL][NVAL];
    __shared__ __align__(8) uint64_t xch[NS];
    const int S = p.tc.stages;
    const uint32_t stage_bytes = p.tc.stride;  // 2 * NT * 16: a chunk of x, then of dy
    const int rank = CL > 1 ? (int)cluster_ctarank() : 0;
    const int64_t cid = CL > 1 ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
    const int64_t ncl = CL > 1 ? (int64_t)cluster_count_x() : (int64_t)gridDim.x;
    const int64_t M = p.M, nv = p.N / E;
    const int64_t SL = (nv + CL - 1) / CL;
    const int64_t v0 = rank * SL;
    const int64_t cnt = nv - v0 < SL ? (nv - v0 > 0 ? nv - v0 : 0) : SL;  // this CTA's vectors
    const int64_t nrows = cid < M ? (M - cid + ncl - 1) / ncl : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &h.abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&h.full[s], 1);
            mbar_init(&h.empty[s], CW);
        }
        if (CL > 1)
            for (int j = 0; j < NS; ++j) mbar_init(&xch[j], CL);
        h.abort = 0;
        fence_mbar_init();
    }
    // every CTA's barriers exist before any peer arrives on them
    if constexpr (CL > 1) cluster_sync_all();
    else __syncthreads();

    // jobs: step i < nrows: pass 1 of row i (K jobs); step i >= 1: pass 2 of row i - 1 (K jobs)
    const int64_t njobs = nrows > 0 ? 2 * nrows * K : 0;
    auto job = [&](int64_t j, int64_t &row, int &pass, int &k) {
        // jobs of step 0: K (pass 1 only); of steps 1..nrows-1: 2K; of step nrows: K
        if (j < K) {
            row = 0, pass = 1, k = (int)j;
            return;
        }
        const int64_t q = j - K;
        const int64_t step = 1 + q / (2 * K);
        const int r = (int)(q % (2 * K));
        if (step < nrows && r < K) {
            row = step, pass = 1, k = r;
        } else {
            row = step - 1, pass = 2, k = step < nrows ? r - K : r;
        }
    };

    if (warp == CW) {
        // ---- producer
        if (lane == 0) {
            const uint64_t keep = l2_policy_keep(), drop = l2_policy_drop();
            int64_t issued = 0;
            for (int64_t j = 0; j < njobs; ++j, ++issued) {
                const int s = (int)(j % S);
                if (j >= S) mbar_wait_bounded(&h.empty[s], (uint32_t)(((j / S) - 1) & 1), abort_flag, p.tc.fault);
                if (*abort_flag) break;
                int64_t i;
                int pass, k;
                job(j, i, pass, k);
                const int64_t row = cid + i * ncl;
                const int64_t c0 = (int64_t)k * NT;  // first vector of the chunk within the slice
                const int64_t vn = cnt - c0 < NT ? (cnt - c0 > 0 ? cnt - c0 : 0) : NT;
                const uint32_t bytes = (uint32_t)vn * 16u;
                unsigned char *dst = ring + (size_t)s * stage_bytes;
                mbar_arrive_expect_tx(&h.full[s], 2 * bytes);
                if (bytes > 0) {
                    const size_t off = ((size_t)row * (size_t)nv + (size_t)(v0 + c0)) * 16;
                    const uint64_t pol = pass == 1 ? keep : drop;
                    bulk_g2s_hint(dst, static_cast<const unsigned char *>(p.x) + off, bytes, &h.full[s], pol);
                    bulk_g2s_hint(dst + NT * 16, static_cast<const unsigned char *>(p.dy) + off, bytes, &h.full[s],
                                  pol);
                }
            }
            if (*abort_flag) {
                int zero = 0;
                for (int64_t j = issued > S ? issued - S : 0; j < issued; ++j)
                    mbar_wait_bounded(&h.full[j % S], (uint32_t)((j / S) & 1),
                                      reinterpret_cast<volatile int *>(&zero), nullptr);
            }
        }
        return;
    }

    // ---- consumers
    const int t = threadIdx.x;
    const float n = (float)p.N;
    float accg[K][E], accb[LN ? K : 1][E];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int64_t lv = (int64_t)k * NT + t;
        gs[lv] = lv < cnt ? param_vec<T>(p.gamma, v0 + lv, true) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            accg[k][e] = 0.f;
            if constexpr (LN) accb[k][e] = 0.f;
        }
    }
    named_sync(1, NT);
    const uint64_t drop = l2_policy_drop();
    int parity = 0;
    int64_t j = 0;
    float c1s[NS], c2s[NS];  // (c1, c2) of the rows in the exchange slots (single-CTA clusters)

    auto pass1 = [&](int64_t i) {
        const int64_t row = cid + i * ncl;
        const float rstd = __ldg(p.rstd + row);
        const float mean = LN ? __ldg(p.mean + row) : 0.f;
        float v[NVAL];
#pragma unroll
        for (int q = 0; q < NVAL; ++q) v[q] = 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k, ++j) {
            const int s = (int)(j % S);
            mbar_wait_bounded(&h.full[s], (uint32_t)((j / S) & 1), abort_flag, p.tc.fault);
            const uint4 *st = reinterpret_cast<const uint4 *>(ring + (size_t)s * stage_bytes);
            const int64_t lv = (int64_t)k * NT + t;
            if (lv < cnt) {
                const uint4 xq = lds128(st + t), dq = lds128(st + NT + t), gq = lds128(gs + lv);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float gg = vget<T>(dq, e) * vget<T>(gq, e);
                    v[0] += gg * (vget<T>(xq, e) - mean);
                    if constexpr (LN) v[NVAL - 1] += gg;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&h.empty[s]);
        }
        v[0] *= rstd;  // sum g xhat = rstd sum g (x - mean)
        // CTA reduction over the NT consumers (identical bits in all)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1)
#pragma unroll
            for (int q = 0; q < NVAL; ++q) v[q] += __shfl_xor_sync(0xffffffffu, v[q], o);
        if (lane == 0) {
#pragma unroll
            for (int q = 0; q < NVAL; ++q) h.red[parity][q][warp] = v[q];
        }
        named_sync(1, NT);
#pragma unroll
        for (int q = 0; q < NVAL; ++q) {
            float sum = 0.f;
#pragma unroll 4
            for (int w = 0; w < CW; ++w) sum += h.red[parity][q][w];
            v[q] = sum;
        }
        parity ^= 1;
        const int sp = (int)(i % NS);
        if constexpr (CL > 1) {
            if (t < CL) {
                const uint32_t dst = map_to_rank(smem_u32(&slot[sp][rank][0]), (uint32_t)t);
#pragma unroll
                for (int q = 0; q < NVAL; ++q) st_cluster_f32(dst + 4u * q, v[q]);
                mbar_arrive_remote(map_to_rank(smem_u32(&xch[sp]), (uint32_t)t));
            }
        } else {
            c2s[sp] = v[0] / n;
            c1s[sp] = LN ? v[NVAL - 1] / n : 0.f;
        }
    };

    auto pass2 = [&](int64_t i) {
        const int64_t row = cid + i * ncl;
        const float rstd = __ldg(p.rstd + row);
        const float mean = LN ? __ldg(p.mean + row) : 0.f;
        const int sp = (int)(i % NS);
        float c1 = 0.f, c2 = 0.f;
        if constexpr (CL > 1) {
            mbar_wait_cluster_bounded(&xch[sp], (uint32_t)((i / NS) & 1), abort_flag, p.tc.fault);
            float s2 = 0.f, s1 = 0.f;
#pragma unroll
            for (int c = 0; c < CL; ++c) {
                s2 += slot[sp][c][0];
                if constexpr (LN) s1 += slot[sp][c][NVAL - 1];
            }
            c2 = s2 / n;
            c1 = LN ? s1 / n : 0.f;
        } else {
            c2 = c2s[sp];
            c1 = c1s[sp];
        }
        const float rc1 = rstd * c1, rc2 = rstd * c2;
        uint4 *dxr = static_cast<uint4 *>(p.dx) + row * nv + v0;
#pragma unroll
        for (int k = 0; k < K; ++k, ++j) {
            const int s = (int)(j % S);
            mbar_wait_bounded(&h.full[s], (uint32_t)((j / S) & 1), abort_flag, p.tc.fault);
            const uint4 *st = reinterpret_cast<const uint4 *>(ring + (size_t)s * stage_bytes);
            const int64_t lv = (int64_t)k * NT + t;
            if (lv < cnt) {
                const uint4 xq = lds128(st + t), dq = lds128(st + NT + t), gq = lds128(gs + lv);
                float o[E];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float xh = (vget<T>(xq, e) - mean) * rstd;
                    const float dyv = vget<T>(dq, e);
                    o[e] = fmaf(-rc2, xh, fmaf(rstd, dyv * vget<T>(gq, e), -rc1));
                    accg[k][e] += dyv * xh;
                    if constexpr (LN) accb[k][e] += dyv;
                }
                st_l2hint(dxr + lv, vpack<T>(o), drop);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&h.empty[s]);
        }
    };

    for (int64_t i = 0; i <= nrows; ++i) {
        if (i < nrows) pass1(i);
        if (i >= 1) pass2(i - 1);
    }
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
        for (int hh = 0; hh < E / 4; ++hh) {
            reinterpret_cast<float4 *>(wsg + lv * E)[hh] =
                make_float4(accg[k][4 * hh], accg[k][4 * hh + 1], accg[k][4 * hh + 2], accg[k][4 * hh + 3]);
            if constexpr (LN)
                reinterpret_cast<float4 *>(wsb + lv * E)[hh] =
                    make_float4(accb[k][4 * hh], accb[k][4 * hh + 1], accb[k][4 * hh + 2], accb[k][4 * hh + 3]);
        }
    }
}

}  // namespace gbn
