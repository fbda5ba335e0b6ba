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
