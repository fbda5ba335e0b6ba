// device_common.cuh -- device-side building blocks shared by the norm kernels:
// 128-bit vector packing for bf16/fp16/fp32, row reductions at warp, CTA and
// thread-block-cluster level (the last through distributed shared memory),
// and the few PTX wrappers the cluster path needs.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gbn {

// Elements of T carried by one 16-byte vector.
template <typename T> struct VecTraits;
template <> struct VecTraits<float> { static constexpr int E = 4; };
template <> struct VecTraits<__half> { static constexpr int E = 8; };
template <> struct VecTraits<__nv_bfloat16> { static constexpr int E = 8; };

// ---------------------------------------------------------------- 16-byte vectors
__device__ __forceinline__ uint32_t word(const uint4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Element e of a 16-byte vector, widened to float (exact for all three types).
template <typename T> __device__ __forceinline__ float vget(const uint4 &v, int e);

template <> __device__ __forceinline__ float vget<float>(const uint4 &v, int e) {
    return __uint_as_float(word(v, e));
}
template <> __device__ __forceinline__ float vget<__nv_bfloat16>(const uint4 &v, int e) {
    const uint32_t w = word(v, e >> 1);
    return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
}
template <> __device__ __forceinline__ float vget<__half>(const uint4 &v, int e) {
    const uint32_t w = word(v, e >> 1);
    __half2 h = *reinterpret_cast<const __half2 *>(&w);
    return (e & 1) ? __high2float(h) : __low2float(h);
}

// Pack E floats into one 16-byte vector of T, each rounded to nearest even.
template <typename T> __device__ __forceinline__ uint4 vpack(const float *f);

template <> __device__ __forceinline__ uint4 vpack<float>(const float *f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
}
template <> __device__ __forceinline__ uint4 vpack<__nv_bfloat16>(const float *f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}
template <> __device__ __forceinline__ uint4 vpack<__half>(const float *f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------- fp32 pairs
// Blackwell issues two fp32 lanes as one instruction (__fadd2_rn, __fmul2_rn,
// __ffma2_rn on float2).  Each lane is rounded exactly like the scalar
// operation, so a computation on pairs gives the bits of the two scalar
// computations in the same order, for half the issue slots.
__device__ __forceinline__ float2 f2s(float s) { return make_float2(s, s); }
__device__ __forceinline__ float2 f2add(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 f2mul(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 f2fma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// Elements 2i and 2i + 1 of a 16-byte vector, widened to float (exact).
template <typename T> __device__ __forceinline__ float2 vpair(const uint4 &v, int i);
template <> __device__ __forceinline__ float2 vpair<float>(const uint4 &v, int i) {
    return make_float2(__uint_as_float(word(v, 2 * i)), __uint_as_float(word(v, 2 * i + 1)));
}
template <> __device__ __forceinline__ float2 vpair<__nv_bfloat16>(const uint4 &v, int i) {
    const uint32_t w = word(v, i);
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <> __device__ __forceinline__ float2 vpair<__half>(const uint4 &v, int i) {
    const uint32_t w = word(v, i);
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}
// Pack E / 2 pairs into one 16-byte vector of T, each element rounded to
// nearest even.
template <typename T> __device__ __forceinline__ uint4 vpack2(const float2 *f) {
    float o[VecTraits<T>::E];
#pragma unroll
    for (int i = 0; i < VecTraits<T>::E / 2; ++i) {
        o[2 * i] = f[i].x;
        o[2 * i + 1] = f[i].y;
    }
    return vpack<T>(o);
}

// Scalar element conversions for the element-wise (any-alignment) path.
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Read-only 16-byte load through the non-coherent path; p must be 16-byte aligned.
__device__ __forceinline__ uint4 ld_vec(const void *base, int64_t idx) {
    return __ldg(reinterpret_cast<const uint4 *>(base) + idx);
}
__device__ __forceinline__ void st_vec(void *base, int64_t idx, const uint4 &v) {
    reinterpret_cast<uint4 *>(base)[idx] = v;
}

// A 16-byte vector of ones of T (the value of an absent gamma).
template <typename T> __device__ __forceinline__ uint4 ones_vec();
template <> __device__ __forceinline__ uint4 ones_vec<float>() {
    return make_uint4(0x3F800000u, 0x3F800000u, 0x3F800000u, 0x3F800000u);
}
template <> __device__ __forceinline__ uint4 ones_vec<__half>() {
    return make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
}
template <> __device__ __forceinline__ uint4 ones_vec<__nv_bfloat16>() {
    return make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
}
// Vector v of a parameter row; a null row stands for the constant row of
// ones (gamma, one = true) or zeros (beta).
template <typename T>
__device__ __forceinline__ uint4 param_vec(const void *row, int64_t v, bool one) {
    return row ? ld_vec(row, v) : (one ? ones_vec<T>() : make_uint4(0, 0, 0, 0));
}

// ---------------------------------------------------------------- cluster PTX
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// Full cluster barrier: every thread of every CTA arrives (release) and waits
// (acquire), so shared::cluster stores issued before it are visible after it.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// ---------------------------------------------------------------- mbarrier + bulk async copy
// A wait gives up after this many SM clock cycles (about two seconds at the
// GB300's top clock); real waits last microseconds.
constexpr long long kWaitLimitCycles = 4000000000LL;

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
// Makes barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// global to this CTA's shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Waits for phase `parity` of `bar` to complete, at most kWaitLimitCycles.
// Returns false without waiting once the CTA has aborted (*abort != 0); on a
// timeout it sets *abort and the device fault word, then returns false.  The
// caller carries on either way, so that every barrier of the CTA stays
// matched and the kernel ends in bounded time.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  volatile int *abort, int *fault) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (*abort) return false;
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort = 1;
            if (fault) atomicExch(fault, 1);
            return false;
        }
    }
}

// 16-byte shared-memory load the compiler may not merge with other loads of
// the same address: staged rows are re-read on every pass instead of being
// kept live in registers across the row reductions.
__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

// Programmatic dependent launch.  launch_dependents lets the next kernel of the
// stream (launched with programmatic stream serialization) start its CTAs
// early; wait_primary, in that next kernel, blocks until the previous grid
// has completed and its memory writes are visible.  Both are hardware
// operations (no polling loop).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Arrive (release, cluster scope) on an mbarrier in another CTA of the
// cluster; `remote` comes from map_to_rank.  Orders this thread's earlier
// st.shared::cluster stores before the arrival.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote)
                 : "memory");
}
// try_wait with cluster-scope acquire: after it succeeds, stores that peers
// made before their release-arrive on this barrier are visible.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait on a cluster-exchange barrier; same abort protocol as
// mbar_wait_bounded.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t *bar, uint32_t parity,
                                                          volatile int *abort, int *fault) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (*abort) return false;
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort = 1;
            if (fault) atomicExch(fault, 1);
            return false;
        }
    }
}

// Release store / acquire load of a 32-bit word in global memory at GPU scope.
__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Named barrier over `count` threads (a multiple of 32); id 0 is __syncthreads.
__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------- reductions
// Butterfly sum over aligned groups of G lanes (G a power of two <= 32).  Every
// lane of a group ends with the same bits: each step adds the same two
// operands on both partner lanes, and float addition is commutative.
template <int G, int R>
__device__ __forceinline__ void group_sum(float (&v)[R]) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) {
#pragma unroll
        for (int r = 0; r < R; ++r) v[r] += __shfl_xor_sync(0xffffffffu, v[r], o);
    }
}

// Shared-memory scratch of one row reducer (two parity copies, so that one
// barrier per reduction suffices: the barrier of call k+1 proves every thread
// has finished reading the copy that call k+2 overwrites).
template <int TPR, int RPC, int CL, int R> struct RowReduceSmem {
    static constexpr int WPR = TPR > 32 ? TPR / 32 : 1;
    float warp_part[TPR > 32 ? 2 * RPC * R * WPR : 1];
    float cta_part[CL > 1 ? 2 * R * CL : 1];
};

// All-reduce R independent sums over the TPR threads of a row group, and over
// the CL CTAs of the cluster when CL > 1.  Every thread of the row (in every
// CTA of the cluster) receives identical bits: partials are combined in a
// fixed order (lane butterfly, then warps in index order, then CTAs in rank
// order).  All threads of the CTA must call it together.
template <int TPR, int RPC, int CL, int R>
__device__ __forceinline__ void row_allreduce(float (&v)[R], RowReduceSmem<TPR, RPC, CL, R> &sm,
                                              int &parity) {
    group_sum<(TPR < 32 ? TPR : 32), R>(v);
    if constexpr (TPR > 32) {
        constexpr int WPR = TPR / 32;
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int grp = threadIdx.x / TPR, wig = warp % WPR;
        float *buf = sm.warp_part + parity * (RPC * R * WPR);
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r) buf[(grp * R + r) * WPR + wig] = v[r];
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < WPR; ++w) s += buf[(grp * R + r) * WPR + w];
            v[r] = s;
        }
    }
    if constexpr (CL > 1) {
        float *buf = sm.cta_part + parity * (R * CL);
        const uint32_t me = cluster_ctarank();
        if (threadIdx.x < CL) {
            const uint32_t remote = map_to_rank(smem_u32(buf), threadIdx.x);
#pragma unroll
            for (int r = 0; r < R; ++r) st_cluster_f32(remote + 4u * (r * CL + me), v[r]);
        }
        cluster_sync_all();
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float s = 0.f;
#pragma unroll
            for (int c = 0; c < CL; ++c) s += buf[r * CL + c];
            v[r] = s;
        }
    }
    parity ^= 1;
}

// Sum over all threads of a CTA of NT threads (NT a multiple of 32), same
// determinism guarantees; used by the element-wise path.
template <int NT, int R>
__device__ __forceinline__ void cta_allreduce(float (&v)[R], float *buf2 /* [2][R][NT/32] */,
                                              int &parity) {
    constexpr int W = NT / 32;
    group_sum<32, R>(v);
    float *buf = buf2 + parity * (R * W);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) buf[r * W + warp] = v[r];
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < R; ++r) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) s += buf[r * W + w];
        v[r] = s;
    }
    parity ^= 1;
}

}  // namespace gbn

namespace gbn {

// All-reduce R sums over a row group of TPR consecutive threads that does not
// span the whole CTA.  TPR <= 32: lane butterfly only.  TPR > 32: butterfly,
// then warp partials through shared memory `scratch` ([2][R][TPR/32] floats,
// private to this group) under named barrier `bar_id` (TPR threads).  Same
// determinism guarantees as row_allreduce.
template <int TPR, int R>
__device__ __forceinline__ void group_allreduce(float (&v)[R], float *scratch, int &parity,
                                                int bar_id) {
    group_sum<(TPR < 32 ? TPR : 32), R>(v);
    if constexpr (TPR > 32) {
        constexpr int WPR = TPR / 32;
        const int wig = (threadIdx.x % TPR) >> 5, lane = threadIdx.x & 31;
        float *buf = scratch + parity * (R * WPR);
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r) buf[r * WPR + wig] = v[r];
        }
        named_sync(bar_id, TPR);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < WPR; ++w) s += buf[r * WPR + w];
            v[r] = s;
        }
    }
    parity ^= 1;
}

// ---------------------------------------------------------------- equal-count group combine
// (mean, M2) of a row from the threads' (mean_t, M2_t) when every thread holds
// the same count c: the union of groups of equal size k has mean
// M = (1/G) sum m_g and M2 = sum (M2_g + k (m_g - M)^2) (the group form of the
// update of Chan, Golub and LeVeque; exact algebra, centred on the union's
// mean).  Applied twice: over the lanes of a warp (butterfly sums, every lane
// identical bits), then over the warps of the row group through shared
// memory (every thread adds the warps in index order).  About half the
// instructions of merging pairs level by level.
template <int TPR, int RPC, int R>
__device__ __forceinline__ void row_meanvar_equal(float (&mean)[R], float (&m2)[R], float c,
                                                  RowReduceSmem<TPR, RPC, 1, 2 * R> &sm, int &parity) {
    constexpr int L = TPR < 32 ? TPR : 32;  // lanes per warp in the group
    float s[R], q[R];
#pragma unroll
    for (int r = 0; r < R; ++r) s[r] = mean[r];
#pragma unroll
    for (int o = 1; o < L; o <<= 1)
#pragma unroll
        for (int r = 0; r < R; ++r) s[r] += __shfl_xor_sync(0xffffffffu, s[r], o);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float mw = s[r] * (1.f / L);
        const float d = mean[r] - mw;
        q[r] = m2[r] + c * (d * d);
        mean[r] = mw;
    }
#pragma unroll
    for (int o = 1; o < L; o <<= 1)
#pragma unroll
        for (int r = 0; r < R; ++r) q[r] += __shfl_xor_sync(0xffffffffu, q[r], o);
#pragma unroll
    for (int r = 0; r < R; ++r) m2[r] = q[r];
    if constexpr (TPR > 32) {
        constexpr int WPR = TPR / 32;
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int grp = threadIdx.x / TPR, wig = warp % WPR;
        float2 *buf = reinterpret_cast<float2 *>(sm.warp_part + parity * (RPC * 2 * R * WPR)) + grp * R * WPR;
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r) buf[r * WPR + wig] = make_float2(mean[r], m2[r]);
        }
        __syncthreads();
        const float cw = c * 32.f;  // count per warp
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float ms = 0.f;
#pragma unroll
            for (int w = 0; w < WPR; ++w) ms += buf[r * WPR + w].x;
            const float M = ms * (1.f / WPR);
            float t2 = 0.f;
#pragma unroll
            for (int w = 0; w < WPR; ++w) {
                const float2 b = buf[r * WPR + w];
                const float dd = b.x - M;
                t2 += b.y + cw * (dd * dd);
            }
            mean[r] = M;
            m2[r] = t2;
        }
    }
    parity ^= 1;
}

// The same combine over a row group of TPR consecutive threads that does not
// span the whole CTA (TPR > 32: warps through `scratch`, this group's
// [2][WPR] float2, under named barrier bar_id).
template <int TPR>
__device__ __forceinline__ void group_meanvar_equal(float &mean, float &m2, float c, float *scratch,
                                                    int &parity, int bar_id) {
    constexpr int L = TPR < 32 ? TPR : 32;
    float s = mean;
#pragma unroll
    for (int o = 1; o < L; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float mw = s * (1.f / L);
    const float d = mean - mw;
    float q = m2 + c * (d * d);
#pragma unroll
    for (int o = 1; o < L; o <<= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    mean = mw;
    m2 = q;
    if constexpr (TPR > 32) {
        constexpr int WPR = TPR / 32;
        const int wig = (threadIdx.x % TPR) >> 5, lane = threadIdx.x & 31;
        float2 *buf = reinterpret_cast<float2 *>(scratch) + parity * WPR;
        if (lane == 0) buf[wig] = make_float2(mw, q);
        named_sync(bar_id, TPR);
        const float cw = c * 32.f;
        float ms = 0.f;
#pragma unroll
        for (int w = 0; w < WPR; ++w) ms += buf[w].x;
        const float M = ms * (1.f / WPR);
        float t2 = 0.f;
#pragma unroll
        for (int w = 0; w < WPR; ++w) {
            const float2 b = buf[w];
            const float dd = b.x - M;
            t2 += b.y + cw * (dd * dd);
        }
        mean = M;
        m2 = t2;
    }
    parity ^= 1;
}

}  // namespace gbn
