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
__device__ __forceinline__ void warp_combine(float &n, float &mean, float &m2) {
    float tn = n, ts = n * mean;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        tn += __shfl_xor_sync(0xffffffffu, tn, o);
        ts += __shfl_xor_sync(0xffffffffu, ts, o);
    }
    const float mu = tn > 0.f ? ts / tn : 0.f;
    const float d = mean - mu;
    float tm = m2 + n * (d * d);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) tm += __shfl_xor_sync(0xffffffffu, tm, o);
    n = tn;
    mean = mu;
    m2 = tm;
}

// PF (prefetch): 0 none; 1 each row is bulk-prefetched into L2 as its pass 1
// starts; 2 as 1 for the first row, then the CTA's next row is prefetched as
// the current row's pass 2 starts (two rows per CTA resident in L2).
template <typename T, bool LN, int NT, int UV, int MINB, int PF>
__global__ void __launch_bounds__(NT, MINB) fwd_wide(const FwdParams p) {
    constexpr int E = VecTraits<T>::E;
    constexpr int W = NT / 32;
    constexpr bool kRoomy = 65536 / (NT * MINB) >= 128;  // registers per thread >= 128
    // The LayerNorm batch is read twice from registers (sum, then M2): with
    // fewer than 128 registers per thread it holds at most 4 vectors.
    constexpr int U = (LN && !kRoomy && UV > 4) ? 4 : UV;
    // Pass 2 loads x, gamma (and beta) per vector: fewer vectors per batch
    // unless the register budget is roomy.
    constexpr int U2r = LN ? U / 2 : (kRoomy ? U : U / 2);
    constexpr int U2 = U2r > 0 ? U2r : 1;
    // Independent partial sums per thread in pass 1 (two for the LayerNorm
    // batch sum and M2 when registers are short).
    constexpr int A0 = (LN && !kRoomy) ? 2 : 4;
    constexpr int A = U < A0 ? U : A0;
    static_assert(NT % 32 == 0 && NT <= 1024, "CTA shape");
    __shared__ float red[2][3][W];

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int64_t nv = p.N / E;
    const float n = (float)p.N;
    const size_t row_bytes = (size_t)nv * 16;
    const uint64_t keep = l2_policy_keep(), drop = l2_policy_drop();
    const uint4 *gam = static_cast<const uint4 *>(p.gamma);
    const uint4 *bet = static_cast<const uint4 *>(p.beta);
    int parity = 0;

    if (PF == 2 && warp == 0 && blockIdx.x < p.M)
        prefetch_row(static_cast<const uint4 *>(p.x) + (int64_t)blockIdx.x * nv, row_bytes, lane, keep);

    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
        const uint4 *xr = static_cast<const uint4 *>(p.x) + row * nv;
        uint4 *yr = static_cast<uint4 *>(p.y) + row * nv;
        if (PF == 1 && warp == 0) prefetch_row(xr, row_bytes, lane, keep);

        // ---- pass 1: statistics (row from DRAM, kept in L2)
        float cnt = 0.f, mean = 0.f, acc = 0.f;  // acc: sum x^2 (RMS) or M2 (LN)
        float pa[A];
#pragma unroll
        for (int a = 0; a < A; ++a) pa[a] = 0.f;
        for (int64_t b = t; b < nv; b += (int64_t)NT * U) {
            uint4 q[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = b + (int64_t)u * NT;
                q[u] = v < nv ? ld_l2hint(xr + v, keep) : make_uint4(0, 0, 0, 0);
            }
            if constexpr (!LN) {
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float f = vget<T>(q[u], e);
                        pa[u % A] += f * f;
                    }
            } else {
                float ps[A], pm[A];
                int nb = 0;
#pragma unroll
                for (int a = 0; a < A; ++a) ps[a] = pm[a] = 0.f;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (b + (int64_t)u * NT < nv) {
                        nb += E;
#pragma unroll
                        for (int e = 0; e < E; ++e) ps[u % A] += vget<T>(q[u], e);
                    }
                }
                float s = ps[0];
#pragma unroll
                for (int a = 1; a < A; ++a) s += ps[a];
                const float fb = (float)nb;
                const float mb = __fdiv_rn(s, fb);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (b + (int64_t)u * NT < nv) {
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            const float d = vget<T>(q[u], e) - mb;
                            pm[u % A] += d * d;
                        }
                    }
                }
                float m2b = pm[0];
#pragma unroll
                for (int a = 1; a < A; ++a) m2b += pm[a];
                if (cnt == 0.f) {
                    cnt = fb;
                    mean = mb;
                    acc = m2b;
                } else {
                    // running += batch (one division per batch of U vectors)
                    const float tot = cnt + fb;
                    const float d = mb - mean;
                    const float r = __fdiv_rn(fb, tot);
                    mean += d * r;
                    acc += m2b + d * d * cnt * r;
                    cnt = tot;
                }
            }
        }
        if constexpr (!LN) {
            acc = pa[0];
#pragma unroll
            for (int a = 1; a < A; ++a) acc += pa[a];
        }

        // ---- CTA reduction (identical bits in every thread)
        float *buf = &red[parity][0][0];
        parity ^= 1;
        if constexpr (!LN) {
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) buf[warp] = acc;
            __syncthreads();
            acc = 0.f;
#pragma unroll 4
            for (int w = 0; w < W; ++w) acc += buf[w];
        } else {
            warp_combine(cnt, mean, acc);
            if (lane == 0) {
                buf[warp] = cnt;
                buf[W + warp] = mean;
                buf[2 * W + warp] = acc;
            }
            __syncthreads();
            // the same group combine over the W warps, in warp order
            float tn = 0.f, ts = 0.f;
#pragma unroll 4
            for (int w = 0; w < W; ++w) {
                tn += buf[w];
                ts += buf[w] * buf[W + w];
            }
            mean = ts / tn;  // tn = N > 0
            acc = 0.f;
#pragma unroll 4
            for (int w = 0; w < W; ++w) {
                const float d = buf[W + w] - mean;
                acc += buf[2 * W + w] + buf[w] * (d * d);
            }
        }
        const float rstd = rsqrtf(acc / n + p.eps);
        if (!LN) mean = 0.f;
        if (t == 0) {
            if (p.rstd) p.rstd[row] = rstd;
            if (LN && p.mean) p.mean[row] = mean;
        }

        if (PF == 2 && warp == 0 && row + gridDim.x < p.M)
            prefetch_row(xr + (int64_t)gridDim.x * nv, row_bytes, lane, keep);

        // ---- pass 2: y = (x - mean) * rstd * gamma (+ beta), x from L2
        for (int64_t b = t; b < nv; b += (int64_t)NT * U2) {
            uint4 q[U2], g[U2], bb[LN ? U2 : 1];
#pragma unroll
            for (int u = 0; u < U2; ++u) {
                const int64_t v = b + (int64_t)u * NT;
                if (v < nv) {
                    q[u] = ld_l2hint(xr + v, drop);
                    g[u] = ld_l2hint(gam + v, keep);
                    if constexpr (LN) bb[u] = ld_l2hint(bet + v, keep);
                }
            }
#pragma unroll
            for (int u = 0; u < U2; ++u) {
                const int64_t v = b + (int64_t)u * NT;
                if (v < nv) {
                    float o[E];
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        o[e] = ((vget<T>(q[u], e) - mean) * rstd) * vget<T>(g[u], e);
                        if constexpr (LN) o[e] += vget<T>(bb[u], e);
                    }
                    st_l2hint(yr + v, vpack<T>(o), drop);
                }
            }
        }
    }
}

}  // namespace gbn
