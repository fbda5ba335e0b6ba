// api.cu -- the C ABI declared in include/gbnorm.h: argument checks, dispatch
// to a kernel variant, launch geometry from the device's SM count, shared
// memory and measured occupancy, launches.
//
// Nothing here allocates device memory or synchronises (except the diagnostic
// gbnorm_read_fault); every launch goes on the caller's stream.  The only
// shared state is a per-device cache (SM count, shared-memory limit, fault
// word address, occupancy per variant), filled once, read lock-free.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/gbnorm.h"
#include "params.h"

namespace gbn {

// Set to nonzero by a kernel whose bounded wait gave up (see gbnorm_read_fault).
__device__ int g_fault_word;

namespace {

constexpr int kMaxDev = 64;
// Bound on the variants of one (op, direction, dtype) table: the per-variant
// caches below are indexed by variant.  tables_fit() checks it once.
constexpr int kMaxVariants = 160;

struct DispatchRow {
    int is_ln, dir, dtype;
    int64_t m_max;  // rows: the row applies to calls with M <= m_max (-1: any M)
    int64_t nv_max;
    const char *variant;
};
const DispatchRow kDispatch[] = {
#include "dispatch_table.inc"
};

// [is_ln][dir][dtype]
const VariantTable *const kTables[2][2][3] = {
    {{&kFwdRms_f32, &kFwdRms_f16, &kFwdRms_bf16}, {&kBwdRms_f32, &kBwdRms_f16, &kBwdRms_bf16}},
    {{&kFwdLn_f32, &kFwdLn_f16, &kFwdLn_bf16}, {&kBwdLn_f32, &kBwdLn_f16, &kBwdLn_bf16}},
};

int elem_size(int dtype) { return dtype == GBNORM_F32 ? 4 : 2; }

// ------------------------------------------------------------------ device cache
struct DevInfo {
    std::atomic<int> state{0};  // 0 unknown, 1 usable, 2 unusable
    int sms = 0;
    int smem_optin = 0;         // max dynamic shared memory per block (opt-in)
    int *fault = nullptr;       // device address of g_fault_word
};
DevInfo g_dev[kMaxDev];
std::mutex g_dev_mu;
// Per (device, table, variant): occupancy (blocks per SM, or active clusters
// on the whole GPU for cluster variants), 0 = not yet measured; and whether
// the kernel's dynamic shared-memory limit has been raised.
std::atomic<int> g_occ[kMaxDev][2][2][3][kMaxVariants];
std::atomic<int> g_smem_set[kMaxDev][2][2][3][kMaxVariants];
// TMA variants: the last (dynamic shared memory, occupancy) pair asked for,
// packed as (bytes << 16) | blocks; their footprint depends on the shape.
std::atomic<uint64_t> g_occ_tma[kMaxDev][2][2][3][kMaxVariants];

// Forced variant per (is_ln, dir, dtype): index + 1, 0 = none.
std::atomic<int> g_force[2][2][3];
// Cap on the persistent grid (CTAs), 0 = none (tests and tuning only).
std::atomic<int> g_grid_limit{0};
// Call counter of the single-kernel backward variants (their flag epochs).
std::atomic<uint32_t> g_epoch{0};
uint32_t next_epoch() {
    uint32_t e;
    do {
        e = g_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
    } while (e == 0);
    return e;
}

// Every compiled table within the caches' bound (else no call is served).
bool tables_fit() {
    static const bool ok = [] {
        for (int ln = 0; ln < 2; ++ln)
            for (int dir = 0; dir < 2; ++dir)
                for (int dt = 0; dt < 3; ++dt)
                    if (kTables[ln][dir][dt]->count > kMaxVariants) return false;
        return true;
    }();
    return ok;
}

int current_device(int *dev) {
    if (!tables_fit()) return GBNORM_ERR_UNSUPPORTED;
    if (cudaGetDevice(dev) != cudaSuccess) return GBNORM_ERR_CUDA;
    if (*dev < 0 || *dev >= kMaxDev) return GBNORM_ERR_UNSUPPORTED;
    DevInfo &d = g_dev[*dev];
    int st = d.state.load(std::memory_order_acquire);
    if (st == 0) {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        st = d.state.load(std::memory_order_relaxed);
        if (st == 0) {
            int major = 0, minor = 0, sms = 0, smem = 0;
            void *fault = nullptr;
            bool ok = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) == cudaSuccess &&
                      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) == cudaSuccess &&
                      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, *dev) == cudaSuccess &&
                      cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, *dev) ==
                          cudaSuccess;
            if (!ok) return GBNORM_ERR_CUDA;
            // The kernels are compiled for sm_103a only.
            st = (major == 10 && minor == 3 && sms > 0) ? 1 : 2;
            if (st == 1) {
                if (cudaGetSymbolAddress(&fault, g_fault_word) != cudaSuccess) return GBNORM_ERR_CUDA;
            }
            d.sms = sms;
            d.smem_optin = smem;
            d.fault = static_cast<int *>(fault);
            d.state.store(st, std::memory_order_release);
        }
    }
    return st == 1 ? GBNORM_OK : GBNORM_ERR_UNSUPPORTED;
}

// What a call allows: 16-byte vectors for the row tensors and gamma/beta
// (vec), and 16-byte-aligned saved statistics (stats; backward TMA kernels
// copy them in bulk).
struct CallShape {
    int is_ln, dir, dtype;
    int64_t M, N;
    bool vec, stats;
};

// Pipeline geometry of a TMA variant for a row of N elements; false if two
// stages of at least one row do not fit.
bool tma_geometry(const Variant &v, const CallShape &c, int dev, TileCfg *tc, size_t *dyn_smem) {
    const size_t row_bytes = (size_t)c.N * elem_size(c.dtype);
    const int ntens = c.dir == 0 ? 1 : 2;
    auto al = [](size_t b) { return (b + 127) & ~(size_t)127; };
    // Header, then gamma (and beta for the LayerNorm forward), then the ring.
    // The backward kernels and the kernels without a producer warp keep them
    // widened to fp32.
    const size_t pbytes = (c.dir == 1 || v.kind == kTmaP) ? (size_t)c.N * 4 : row_bytes;
    const size_t params = al(pbytes) * ((c.dir == 0 && c.is_ln) ? 2 : 1);
    const size_t budget_all = (size_t)g_dev[dev].smem_optin / (size_t)v.ctas_per_sm;
    if (budget_all <= (size_t)kTmaHeaderBytes + params + 1024) return false;
    const size_t budget = budget_all - kTmaHeaderBytes - params;
    // Statistics window per stage (backward): the tile's rows widened to
    // 16-byte multiples, (RT + 7) & ~3 floats per statistic.
    auto stride_of = [&](int64_t rt) {
        size_t s = ntens * al((size_t)rt * row_bytes);
        if (c.dir == 1) s += al((size_t)((rt + 7) & ~(int64_t)3) * 4 * (c.is_ln ? 2 : 1));
        return s;
    };
    // Row groups of the CTA; without a producer warp each keeps its own part
    // of the ring (at least two stages each, the same number for all).
    const int rpp = v.consumers() / v.tpr;
    const int min_stages = v.kind == kTmaP ? 2 * rpp : 2;
    if (min_stages > kTmaMaxStages) return false;
    int64_t rt = (int64_t)(v.stage_target / (ntens * row_bytes));
    if (rt < 1) rt = 1;
    if (rt > c.M) rt = c.M > 0 ? c.M : 1;  // never more rows per tile than the problem has
    while (rt > 1 && (size_t)min_stages * stride_of(rt) > budget) rt /= 2;
    const size_t stride = stride_of(rt);
    if ((size_t)min_stages * stride > budget) return false;
    int stages = (int)(budget / stride);
    if (stages > kTmaMaxStages) stages = kTmaMaxStages;
    if (v.kind == kTmaP) stages -= stages % rpp;
    size_t ring = (size_t)stages * stride;
    // The backward combines its row groups' partials in the idle ring: every
    // group's row of partials side by side ([NS][groups][TPR * VPT * E]).
    if (c.dir == 1 && rpp > 1) {
        const size_t comb = (size_t)v.consumers() * v.vpt * v.elems_per_vec * 4 * (c.is_ln ? 2 : 1);
        if (comb > ring) ring = comb;
    }
    // Single-kernel variants sum the partial rows through 16 x 128 floats of
    // the idle ring.
    if (v.fused && ring < kSkPartBytes) ring = kSkPartBytes;
    if (ring > budget) return false;
    tc->rows = (int)rt;
    tc->stages = stages;
    tc->stride = (uint32_t)stride;
    tc->fault = g_dev[dev].fault;
    *dyn_smem = kTmaHeaderBytes + params + ring;
    return true;
}

// Geometry of a cluster TMA variant: each of the CL CTAs stages one column
// slice of one row per stage.  False if a slice exceeds the variant's
// per-thread capacity, a CTA would get no columns, or two stages do not fit.
bool tmac_geometry(const Variant &v, const CallShape &c, int dev, TileCfg *tc, size_t *dyn_smem) {
    auto al = [](size_t b) { return (b + 127) & ~(size_t)127; };
    const int64_t nv = c.N / (16 / elem_size(c.dtype));
    const int64_t slice = (nv + v.cl - 1) / v.cl;
    if (slice > (int64_t)v.tpr * v.vpt || (int64_t)(v.cl - 1) * slice >= nv) return false;
    const size_t slice_al = al((size_t)slice * 16);
    const size_t params = slice_al * ((c.dir == 0 && c.is_ln) ? 2 : 1);
    const size_t stride = (c.dir == 0 ? 1 : 2) * slice_al + (c.dir == 1 ? 128 : 0);
    const size_t optin = (size_t)g_dev[dev].smem_optin;
    if (optin <= (size_t)kTmaHeaderBytes + params + 2 * stride) return false;
    int stages = (int)((optin - kTmaHeaderBytes - params) / stride);
    if (stages > kTmaMaxStages) stages = kTmaMaxStages;
    // The consumers hold the rows of two exchange steps (2 * RS stages) at
    // once; a shallower ring could never refill.
    if (stages < 2 * v.rows) return false;
    tc->rows = 1;
    tc->stages = stages;
    tc->stride = (uint32_t)stride;
    tc->fault = g_dev[dev].fault;
    *dyn_smem = kTmaHeaderBytes + params + (size_t)stages * stride;
    return true;
}

// Ring of a bulk-copy wide-row forward: stages of (params + 1) chunks of
// tpr * vpt 16-byte vectors, as many as fit (at most kTmaMaxStages, at least 2).
bool wtma_geometry(const Variant &v, const CallShape &c, int dev, TileCfg *tc, size_t *dyn_smem) {
    if (c.dir != 0) return false;
    const size_t stage = (size_t)(c.is_ln ? 3 : 2) * (size_t)v.tpr * v.vpt * 16u;
    const size_t budget = (size_t)g_dev[dev].smem_optin - kTmaHeaderBytes;
    int stages = (int)(budget / stage);
    if (stages > kTmaMaxStages) stages = kTmaMaxStages;
    if (stages < 2) return false;
    tc->rows = 1;
    tc->stages = stages;
    tc->stride = (uint32_t)stage;
    tc->fault = g_dev[dev].fault;
    *dyn_smem = kTmaHeaderBytes + (size_t)stages * stage;
    return true;
}

// Ring of a bulk-copy wide-row backward: stages of one chunk of x and one of dy
// (tpr vectors each); false unless each CTA's column slice fits in vpt chunks.
bool wtmac_geometry(const Variant &v, const CallShape &c, int dev, TileCfg *tc, size_t *dyn_smem) {
    if (c.dir != 1) return false;
    const int64_t nv = c.N / v.elems_per_vec;
    const int64_t slice = (nv + v.cl - 1) / v.cl;
    if (slice > (int64_t)v.tpr * v.vpt) return false;
    const size_t stage = 2u * (size_t)v.tpr * 16u;
    const size_t gam = (size_t)v.tpr * v.vpt * 16u;  // gamma of the slice
    // the kernel's static shared memory (exchange slots, barriers) stays below 1 KB
    const size_t budget = (size_t)g_dev[dev].smem_optin - kTmaHeaderBytes - gam - 1024;
    int stages = (int)(budget / stage);
    if (stages > kTmaMaxStages) stages = kTmaMaxStages;
    if (stages < 2) return false;
    tc->rows = 1;
    tc->stages = stages;
    tc->stride = (uint32_t)stage;
    tc->fault = g_dev[dev].fault;
    *dyn_smem = kTmaHeaderBytes + gam + (size_t)stages * stage;
    return true;
}

// Shared memory of a register-sum wide backward: gamma of the slice as fp32
// (E / 4 planes of tpr * vpt float4); false if a CTA's slice exceeds vpt
// vectors per thread.
bool wider_geometry(const Variant &v, const CallShape &c, int dev, size_t *dyn_smem) {
    if (c.dir != 1) return false;
    const int64_t nv = c.N / v.elems_per_vec;
    const int64_t slice = (nv + v.cl - 1) / v.cl;
    if (slice > (int64_t)v.tpr * v.vpt) return false;
    // gamma as fp32 planes; with db 1, gamma in its storage type and the
    // dbeta sums as fp32 planes; with db 2, the dbeta sums only
    const size_t planes = (size_t)(v.elems_per_vec / 4) * (size_t)v.tpr * v.vpt * 16u;
    const size_t bytes = v.db == 1 ? (size_t)v.tpr * v.vpt * 16u + planes : planes;
    if (bytes + 4096 > (size_t)g_dev[dev].smem_optin) return false;
    *dyn_smem = bytes;
    return true;
}

// Shared-memory ring of a wcs variant (cluster slices resident in shared
// memory): gamma (and beta, forward LayerNorm) slices in their storage type,
// then S stages of one row's slice of x (and dy), S between 2 and 8 as room
// allows.  False if a CTA of the cluster would get no columns, a slice
// exceeds the per-thread capacity, or two stages do not fit.
bool wcs_geometry(const Variant &v, const CallShape &c, int dev, TileCfg *tc, size_t *dyn_smem) {
    const int64_t nv = c.N / v.elems_per_vec;
    const int64_t slice = (nv + v.cl - 1) / v.cl;
    if (slice > (int64_t)v.tpr * v.vpt || (int64_t)(v.cl - 1) * slice >= nv) return false;
    const size_t sb = ex_al128((size_t)slice * 16u);
    const size_t params = sb * ((c.dir == 0 && c.is_ln) ? 2u : 1u);
    const size_t stage = sb * (c.dir == 1 ? 2u : 1u);
    // room for the kernel's static shared memory (barriers, reductions, slots)
    const size_t avail = (size_t)g_dev[dev].smem_optin - 4096;
    if (avail < params + 2 * stage) return false;
    int stages = (int)((avail - params) / stage);
    if (stages > 8) stages = 8;
    tc->rows = 1;
    tc->stages = stages;
    tc->stride = (uint32_t)stage;
    tc->fault = g_dev[dev].fault;
    *dyn_smem = params + (size_t)stages * stage;
    return true;
}

// Shared memory of a cluster-slice forward variant: gamma (and beta) of a
// slice in their storage type.  False if the slice exceeds the per-thread
// capacity or does not fit.
bool fwider_geometry(const Variant &v, const CallShape &c, int dev, size_t *dyn_smem) {
    if (c.dir != 0) return false;
    const int64_t nv = c.N / v.elems_per_vec;
    const int64_t slice = (nv + v.cl - 1) / v.cl;
    if (slice > (int64_t)v.tpr * v.vpt) return false;
    const size_t bytes = (size_t)v.tpr * v.vpt * 16u * (c.is_ln ? 2u : 1u);
    if (bytes + 4096 > (size_t)g_dev[dev].smem_optin) return false;
    *dyn_smem = bytes;
    return true;
}

// Shared memory of a wide-row variant: none for the forward; for the
// backward each CTA's column slice of dgamma (and dbeta) sums in fp32.  False
// if a CTA of the cluster would get no columns or the sums do not fit.
bool wide_geometry(const Variant &v, const CallShape &c, int dev, size_t *dyn_smem) {
    *dyn_smem = 0;
    if (c.dir == 0) return true;
    const int64_t nv = c.N / v.elems_per_vec;
    const int64_t slice = (nv + v.cl - 1) / v.cl;
    if ((int64_t)(v.cl - 1) * slice >= nv) return false;
    const size_t bytes = (size_t)slice * v.elems_per_vec * 4u * (c.is_ln ? 2u : 1u);
    // room for the kernel's static shared memory (reductions, exchange slots)
    if (bytes + 4096 > (size_t)g_dev[dev].smem_optin) return false;
    *dyn_smem = bytes;
    return true;
}

// Shared memory of a row-resident variant with gamma (and beta) staged as
// fp32 ([N] floats each) or, raw, in their storage type ([N / E] 16-byte
// vectors each); false if it does not fit.
bool rows_s_geometry(const Variant &v, const CallShape &c, int dev, size_t *dyn_smem) {
    const size_t per = v.raw ? (size_t)(c.N / v.elems_per_vec) * 16u : (size_t)c.N * 4u;
    const size_t bytes = per * (c.is_ln ? 2u : 1u);
    if (bytes + 4096 > (size_t)g_dev[dev].smem_optin) return false;
    *dyn_smem = bytes;
    return true;
}

bool can_serve(const Variant &v, const CallShape &c, int dev) {
    if (v.kind == kElem) return true;
    if (!c.vec || c.N > v.max_n()) return false;
    if (v.kind == kWide) {
        size_t dyn;
        return wide_geometry(v, c, dev, &dyn);
    }
    if (v.kind == kWtma) {
        TileCfg tc;
        size_t dyn;
        return wtma_geometry(v, c, dev, &tc, &dyn);
    }
    if (v.kind == kWtmaC) {
        TileCfg tc;
        size_t dyn;
        return wtmac_geometry(v, c, dev, &tc, &dyn);
    }
    if (v.kind == kWideR) {
        size_t dyn;
        return wider_geometry(v, c, dev, &dyn);
    }
    if (v.kind == kWcs) {
        TileCfg tc;
        size_t dyn;
        return wcs_geometry(v, c, dev, &tc, &dyn);
    }
    if (v.kind == kWideF) {
        size_t dyn;
        return fwider_geometry(v, c, dev, &dyn);
    }
    if (v.kind == kRowsS) {
        size_t dyn;
        return rows_s_geometry(v, c, dev, &dyn);
    }
    if (v.staged_rows() || v.kind == kTmaCl) {
        if (c.dir == 1 && !c.stats) return false;
        TileCfg tc;
        size_t dyn;
        return v.staged_rows() ? tma_geometry(v, c, dev, &tc, &dyn) : tmac_geometry(v, c, dev, &tc, &dyn);
    }
    return true;
}

int find_variant(const VariantTable &t, const char *name) {
    for (int i = 0; i < t.count; ++i)
        if (std::strcmp(t.v[i].name, name) == 0) return i;
    return -1;
}

// The dispatch table resolved once to variant indices, per (is_ln, dir, dtype):
// the rows that apply, in table order, and the element-wise fallback.
constexpr int kMaxRows = sizeof(kDispatch) / sizeof(kDispatch[0]);
struct Resolved {
    int n = 0;
    int64_t m_max[kMaxRows];
    int64_t nv_max[kMaxRows];
    int idx[kMaxRows];
    int elem = -1;
};
struct ResolvedAll {
    Resolved r[2][2][3];
    ResolvedAll() {
        for (int ln = 0; ln < 2; ++ln)
            for (int dir = 0; dir < 2; ++dir)
                for (int dt = 0; dt < 3; ++dt) {
                    Resolved &o = r[ln][dir][dt];
                    const VariantTable &t = *kTables[ln][dir][dt];
                    o.elem = find_variant(t, "elem");
                    for (const DispatchRow &row : kDispatch) {
                        if ((row.is_ln >= 0 && row.is_ln != ln) || row.dir != dir ||
                            (row.dtype >= 0 && row.dtype != dt))
                            continue;
                        const int i = find_variant(t, row.variant);
                        if (i < 0) continue;
                        o.m_max[o.n] = row.m_max;
                        o.nv_max[o.n] = row.nv_max;
                        o.idx[o.n] = i;
                        ++o.n;
                    }
                }
    }
};
const Resolved &resolved(int ln, int dir, int dt) {
    static const ResolvedAll all;  // built on first use (thread-safe)
    return all.r[ln][dir][dt];
}

// Index of the variant that serves this call.
int select_variant(const CallShape &c, int dev) {
    const VariantTable &t = *kTables[c.is_ln][c.dir][c.dtype];
    const int forced = g_force[c.is_ln][c.dir][c.dtype].load(std::memory_order_relaxed) - 1;
    if (forced >= 0 && forced < t.count && can_serve(t.v[forced], c, dev)) return forced;
    const Resolved &r = resolved(c.is_ln, c.dir, c.dtype);
    if (!c.vec) return r.elem;
    const int64_t nv = c.N / (16 / elem_size(c.dtype));
    for (int k = 0; k < r.n; ++k) {
        if (nv > r.nv_max[k] || (r.m_max[k] >= 0 && c.M > r.m_max[k])) continue;
        if (can_serve(t.v[r.idx[k]], c, dev)) return r.idx[k];
    }
    return r.elem;
}

struct Plan {
    int idx;
    int64_t grid;      // CTAs
    int64_t P;         // partial rows the backward writes (CTAs, or clusters)
    size_t dyn_smem;
    TileCfg tc;
};

// Occupancy of a variant on device dev (cached, except for TMA variants whose
// shared-memory footprint depends on the shape).
int occupancy(const CallShape &c, int idx, int dev, size_t dyn_smem, int *out) {
    std::atomic<int> &slot = g_occ[dev][c.is_ln][c.dir][c.dtype][idx];
    int o = slot.load(std::memory_order_relaxed);
    const Variant &v = kTables[c.is_ln][c.dir][c.dtype]->v[idx];
    // Kinds whose shared memory (and so occupancy) depends on the shape.
    const bool per_shape = v.staged_rows() || v.kind == kRowsS || v.kind == kWtma || v.kind == kWtmaC ||
                           v.kind == kWideR || v.kind == kWcs || v.kind == kWideF ||
                           (v.kind == kWide && dyn_smem > 0);
    if (o > 0 && !per_shape) {
        *out = o;
        return GBNORM_OK;
    }
    if (v.staged_rows() || v.kind == kTmaCl || v.kind == kRowsS || v.kind == kWtma || v.kind == kWtmaC ||
        v.kind == kWideR || v.kind == kWcs || v.kind == kWideF || (v.kind == kWide && dyn_smem > 0)) {
        std::atomic<uint64_t> &cache = g_occ_tma[dev][c.is_ln][c.dir][c.dtype][idx];
        const uint64_t hit = cache.load(std::memory_order_relaxed);
        if (hit != 0 && (hit >> 16) == (uint64_t)dyn_smem) {
            *out = (int)(hit & 0xffff);
            return GBNORM_OK;
        }
        std::atomic<int> &set = g_smem_set[dev][c.is_ln][c.dir][c.dtype][idx];
        if (!set.load(std::memory_order_acquire)) {
            // Dynamic limit: the per-SM share, less the kernel's static shared memory.
            cudaFuncAttributes fa;
            if (cudaFuncGetAttributes(&fa, v.kernel) != cudaSuccess) return GBNORM_ERR_CUDA;
            // (kTma splits the SM between ctas_per_sm CTAs; for the other kinds it
            // is only a launch bound and occupancy follows from the footprint.)
            const int share = v.kind == kTma ? v.ctas_per_sm : 1;
            const int lim = g_dev[dev].smem_optin / share - (int)fa.sharedSizeBytes;
            if (cudaFuncSetAttribute(v.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lim) !=
                cudaSuccess)
                return GBNORM_ERR_CUDA;
            if (v.cl > 8 &&
                cudaFuncSetAttribute(v.kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                    cudaSuccess)
                return GBNORM_ERR_CUDA;
            set.store(1, std::memory_order_release);
        }
        if (v.cl == 1) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, v.kernel, v.cta, dyn_smem) != cudaSuccess)
                return GBNORM_ERR_CUDA;
        } else {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = v.cl;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(v.cl * g_dev[dev].sms);
            cfg.blockDim = dim3(v.cta);
            cfg.dynamicSmemBytes = dyn_smem;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&o, v.kernel, &cfg) != cudaSuccess) return GBNORM_ERR_CUDA;
        }
        if (o > 0 && o < 0xffff) cache.store(((uint64_t)dyn_smem << 16) | (uint64_t)o, std::memory_order_relaxed);
    } else if (v.cl == 1) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, v.kernel, v.cta, 0) != cudaSuccess)
            return GBNORM_ERR_CUDA;
    } else {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = v.cl;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(v.cl * g_dev[dev].sms);
        cfg.blockDim = dim3(v.cta);
        cfg.dynamicSmemBytes = 0;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&o, v.kernel, &cfg) != cudaSuccess) return GBNORM_ERR_CUDA;
    }
    if (o <= 0) return GBNORM_ERR_UNSUPPORTED;
    if (!per_shape) slot.store(o, std::memory_order_relaxed);
    *out = o;
    return GBNORM_OK;
}

// Launch geometry for variant idx.
int make_plan(const CallShape &c, int idx, int dev, Plan *pl) {
    const Variant &v = kTables[c.is_ln][c.dir][c.dtype]->v[idx];
    const int sms = g_dev[dev].sms;
    pl->idx = idx;
    pl->grid = 0;
    pl->P = 0;
    pl->dyn_smem = 0;
    pl->tc = TileCfg{0, 0, 0, g_dev[dev].fault};
    if (c.M <= 0) return GBNORM_OK;
    if (v.staged_rows() && !tma_geometry(v, c, dev, &pl->tc, &pl->dyn_smem)) return GBNORM_ERR_UNSUPPORTED;
    if (v.kind == kTmaCl && !tmac_geometry(v, c, dev, &pl->tc, &pl->dyn_smem)) return GBNORM_ERR_UNSUPPORTED;
    if (v.kind == kWide && !wide_geometry(v, c, dev, &pl->dyn_smem)) return GBNORM_ERR_UNSUPPORTED;
    if (v.kind == kRowsS && !rows_s_geometry(v, c, dev, &pl->dyn_smem)) return GBNORM_ERR_UNSUPPORTED;
    if (v.kind == kWtma && !wtma_geometry(v, c, dev, &pl->tc, &pl->dyn_smem)) return GBNORM_ERR_UNSUPPORTED;
    if (v.kind == kWtmaC && !wtmac_geometry(v, c, dev, &pl->tc, &pl->dyn_smem)) return GBNORM_ERR_UNSUPPORTED;
    if (v.kind == kWideR && !wider_geometry(v, c, dev, &pl->dyn_smem)) return GBNORM_ERR_UNSUPPORTED;
    if (v.kind == kWcs && !wcs_geometry(v, c, dev, &pl->tc, &pl->dyn_smem)) return GBNORM_ERR_UNSUPPORTED;
    if (v.kind == kWideF && !fwider_geometry(v, c, dev, &pl->dyn_smem)) return GBNORM_ERR_UNSUPPORTED;
    int occ = 0;
    int st = occupancy(c, idx, dev, pl->dyn_smem, &occ);
    if (st != GBNORM_OK) return st;
    const int64_t limit = g_grid_limit.load(std::memory_order_relaxed);
    if (v.kind == kElem) {
        // Element-wise kernels: one CTA per row at a time.  The backward keeps
        // one partial row per CTA, so it is held to one CTA per SM.
        int64_t cap = c.dir == 0 ? (int64_t)occ * sms : (int64_t)sms;
        if (limit > 0 && limit < cap) cap = limit;
        pl->grid = c.M < cap ? c.M : cap;
        pl->P = pl->grid;
        return GBNORM_OK;
    }
    if (v.kind == kWtmaC) {
        // occ = clusters that fit on the GPU at once; one row per cluster at a time
        int64_t cap = occ;
        if (limit > 0) {
            const int64_t lc = limit / v.cl > 0 ? limit / v.cl : 1;
            if (lc < cap) cap = lc;
        }
        const int64_t ncl = c.M < cap ? c.M : cap;
        pl->grid = ncl * v.cl;
        pl->P = ncl;
        return GBNORM_OK;
    }
    if (v.kind == kWtma) {
        // one row per CTA at a time
        int64_t cap = (int64_t)occ * sms;
        if (limit > 0 && limit < cap) cap = limit;
        pl->grid = c.M < cap ? c.M : cap;
        pl->P = pl->grid;
        return GBNORM_OK;
    }
    if (v.kind == kTmaCl) {
        // occ = clusters that fit on the GPU at once; one row per cluster at a time.
        int64_t cap = occ;
        if (limit > 0) {
            const int64_t lc = limit / v.cl > 0 ? limit / v.cl : 1;
            if (lc < cap) cap = lc;
        }
        const int64_t ncl = c.M < cap ? c.M : cap;
        pl->grid = ncl * v.cl;
        pl->P = ncl;
        return GBNORM_OK;
    }
    if (v.staged_rows()) {
        const int64_t ntiles = (c.M + pl->tc.rows - 1) / pl->tc.rows;
        int64_t cap = (int64_t)occ * sms;
        if (limit > 0 && limit < cap) cap = limit;
        pl->grid = ntiles < cap ? ntiles : cap;
        pl->P = pl->grid;
        return GBNORM_OK;
    }
    const int64_t rows_per_unit = v.cl > 1 ? v.rows : v.rows_per_cta_iter();
    const int64_t units = (c.M + rows_per_unit - 1) / rows_per_unit;
    int64_t cap = v.cl > 1 ? (int64_t)occ : (int64_t)occ * sms;
    if (limit > 0) {
        const int64_t lu = limit / v.cl > 0 ? limit / v.cl : 1;
        if (lu < cap) cap = lu;
    }
    const int64_t n_units = units < cap ? units : cap;
    pl->grid = n_units * v.cl;
    pl->P = n_units;
    return GBNORM_OK;
}

// Selected variant and its plan; if the GPU cannot host the selected variant
// (e.g. no cluster of its size fits), the element-wise variant, which always
// can.
int plan_call(const CallShape &c, int dev, Plan *pl) {
    const int idx = select_variant(c, dev);
    int st = make_plan(c, idx, dev, pl);
    const int elem = resolved(c.is_ln, c.dir, c.dtype).elem;
    if (st == GBNORM_ERR_UNSUPPORTED && idx != elem) st = make_plan(c, elem, dev, pl);
    return st;
}

int launch_kernel(const Variant &v, const Plan &pl, void *params, cudaStream_t s) {
    void *args[1] = {params};
    cudaError_t e;
    if (v.fused) {
        // Single-kernel variants wait for every CTA's partial row: a cooperative
        // launch guarantees that all CTAs are resident together (the grid is
        // capped at the measured occupancy), or fails instead of starting.
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.gridDim = dim3((unsigned)pl.grid);
        cfg.blockDim = dim3(v.cta);
        cfg.dynamicSmemBytes = pl.dyn_smem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelExC(&cfg, v.kernel, args);
    } else if (v.cl == 1) {
        e = cudaLaunchKernel(v.kernel, dim3((unsigned)pl.grid), dim3(v.cta), args, pl.dyn_smem, s);
    } else {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = v.cl;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3((unsigned)pl.grid);
        cfg.blockDim = dim3(v.cta);
        cfg.dynamicSmemBytes = pl.dyn_smem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelExC(&cfg, v.kernel, args);
    }
    if (e != cudaSuccess) return GBNORM_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? GBNORM_OK : GBNORM_ERR_CUDA;
}

// ------------------------------------------------------------------ argument checks

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

bool valid_shape(int64_t M, int64_t N, int dtype) {
    if (dtype != GBNORM_F32 && dtype != GBNORM_F16 && dtype != GBNORM_BF16) return false;
    if (M < 0 || N < 1 || N > GBNORM_MAX_N) return false;
    // Byte offsets must fit comfortably in int64.
    if (M > 0 && M > (INT64_MAX / 16) / N) return false;
    return true;
}

struct Buf {
    const void *p;
    size_t bytes;
};

// Any output overlapping any input, or another output, is rejected; an
// output may coincide exactly with the one input named as its in-place pair.
bool bad_aliasing(const Buf *outs, int no, const Buf *ins, int ni, const void *inplace_out,
                  const void *inplace_in) {
    for (int i = 0; i < no; ++i) {
        for (int j = 0; j < ni; ++j) {
            if (outs[i].p == inplace_out && ins[j].p == inplace_in && inplace_out == inplace_in &&
                outs[i].bytes == ins[j].bytes)
                continue;
            if (overlap(outs[i].p, outs[i].bytes, ins[j].p, ins[j].bytes)) return true;
        }
        for (int j = i + 1; j < no; ++j)
            if (overlap(outs[i].p, outs[i].bytes, outs[j].p, outs[j].bytes)) return true;
    }
    return false;
}

int do_fwd(int is_ln, const void *x, const void *gamma, const void *beta, void *y, float *mean,
           float *rstd, int64_t M, int64_t N, int dtype, float eps, cudaStream_t stream) {
    if (!valid_shape(M, N, dtype)) return GBNORM_ERR_INVALID_ARG;
    if (M > 0 && (!x || !y)) return GBNORM_ERR_INVALID_ARG;
    if (!std::isfinite(eps) || eps < 0.f) return GBNORM_ERR_INVALID_ARG;
    // A NULL gamma / beta is passed through: the kernels use gamma = 1, beta = 0.
    const size_t b = (size_t)elem_size(dtype);
    const size_t mat = (size_t)M * (size_t)N * b, vec = (size_t)N * b, st = (size_t)M * 4;
    const Buf outs[3] = {{y, mat}, {rstd, st}, {is_ln ? mean : nullptr, st}};
    const Buf ins[3] = {{x, mat}, {gamma, vec}, {is_ln ? beta : nullptr, vec}};
    if (bad_aliasing(outs, 3, ins, 3, y, x)) return GBNORM_ERR_INVALID_ARG;
    int dev;
    int s = current_device(&dev);
    if (s != GBNORM_OK) return s;
    if (M == 0) return GBNORM_OK;
    CallShape c{is_ln, 0, dtype, M, N, false, true};
    c.vec = (vec % 16) == 0 && aligned16(x) && aligned16(y) && aligned16(gamma) &&
            (!is_ln || aligned16(beta));
    Plan pl;
    s = plan_call(c, dev, &pl);
    if (s != GBNORM_OK) return s;
    FwdParams p{x, gamma, is_ln ? beta : nullptr, y, is_ln ? mean : nullptr, rstd, M, N, eps, pl.tc};
    return launch_kernel(kTables[is_ln][0][dtype]->v[pl.idx], pl, &p, stream);
}

// Workspace bytes the backward of this shape needs.  The call may take the
// TMA, the register or the element-wise path (that depends on pointer
// alignment), so this sizes for the largest of the three.
size_t ws_bytes_for(int is_ln, int64_t M, int64_t N, int dtype, int dev, int *status) {
    const int E = 16 / elem_size(dtype);
    size_t best = 0;
    const bool flags[3][2] = {{false, false}, {true, false}, {true, true}};  // (vec, stats)
    for (const auto &f : flags) {
        if (f[0] && (N % E) != 0) continue;
        CallShape c{is_ln, 1, dtype, M, N, f[0], f[1]};
        Plan pl;
        *status = plan_call(c, dev, &pl);
        if (*status != GBNORM_OK) return 0;
        // [2][P][N] partial rows (one block for RMSNorm), then P flag words of
        // the single-kernel variants
        const size_t need = (size_t)pl.P * (size_t)N * 4u * (is_ln ? 2u : 1u) + (size_t)pl.P * 4u;
        if (need > best) best = need;
    }
    return (best + 255u) & ~(size_t)255u;
}

int launch_colreduce(int is_ln, const float *wsc, int64_t P, int64_t N, float *dgamma, float *dbeta, bool pdl,
                     cudaStream_t stream);

int do_bwd(int is_ln, const void *dy, const void *x, const void *gamma, const float *mean,
           const float *rstd, void *dx, float *dgamma, float *dbeta, void *ws, size_t ws_bytes,
           int64_t M, int64_t N, int dtype, cudaStream_t stream) {
    if (!valid_shape(M, N, dtype)) return GBNORM_ERR_INVALID_ARG;
    if (M > 0 && (!dy || !x || !rstd || !dx || (is_ln && !mean))) return GBNORM_ERR_INVALID_ARG;
    // A NULL gamma is passed through (the kernels use gamma = 1); a NULL
    // dgamma / dbeta is not produced.
    if (!is_ln) dbeta = nullptr;
    const size_t b = (size_t)elem_size(dtype);
    const size_t mat = (size_t)M * (size_t)N * b, vec = (size_t)N * b, st = (size_t)M * 4,
                 pv = (size_t)N * 4;
    const Buf outs[4] = {{dx, mat}, {dgamma, pv}, {is_ln ? dbeta : nullptr, pv}, {nullptr, 0}};
    const Buf ins[5] = {{dy, mat}, {x, mat}, {gamma, vec}, {rstd, st}, {is_ln ? mean : nullptr, st}};
    if (bad_aliasing(outs, 3, ins, 5, dx, dy)) return GBNORM_ERR_INVALID_ARG;
    int dev;
    int s = current_device(&dev);
    if (s != GBNORM_OK) return s;
    const size_t need = ws_bytes_for(is_ln, M, N, dtype, dev, &s);
    if (s != GBNORM_OK) return s;
    if (M > 0) {
        if (!ws || ws_bytes < need || !aligned16(ws)) return GBNORM_ERR_WORKSPACE;
        const Buf all_out[4] = {outs[0], outs[1], outs[2], {ws, need}};
        if (bad_aliasing(all_out, 4, ins, 5, dx, dy)) return GBNORM_ERR_INVALID_ARG;
    }
    int64_t P = 0;
    if (M > 0) {
        CallShape c{is_ln, 1, dtype, M, N, false, false};
        c.vec = (vec % 16) == 0 && aligned16(dy) && aligned16(x) && aligned16(dx) && aligned16(gamma);
        c.stats = aligned16(rstd) && (!is_ln || aligned16(mean));
        Plan pl;
        s = plan_call(c, dev, &pl);
        if (s != GBNORM_OK) return s;
        const Variant &v = kTables[is_ln][1][dtype]->v[pl.idx];
        BwdParams p{dy, x, gamma, is_ln ? mean : nullptr, rstd, dx, static_cast<float *>(ws), M, N, pl.tc,
                    nullptr, nullptr, 0u};
        if (v.fused) {
            // The kernel sums the partial rows itself; its flag words follow
            // the partial rows in the workspace.
            p.dgamma = dgamma;
            p.dbeta = dbeta;
            p.epoch = next_epoch();
            return launch_kernel(v, pl, &p, stream);
        }
        s = launch_kernel(v, pl, &p, stream);
        if (s != GBNORM_OK) return s;
        P = pl.P;
    }
    return launch_colreduce(is_ln, static_cast<const float *>(ws), P, N, dgamma, dbeta, M > 0, stream);
}

// ------------------------------------------------------------------ general form
// Rows with their own strides, a storage type per tensor, a fused residual
// add (norm_fwd_ex / norm_bwd_ex in include/gbnorm.h).

// Bytes an [M, N] matrix with row stride ld spans.
size_t span(int64_t M, int64_t N, int64_t ld, int dtype) {
    return M > 0 ? ((size_t)(M - 1) * (size_t)ld + (size_t)N) * (size_t)elem_size(dtype) : 0;
}

bool valid_dtype(int d) { return d == GBNORM_F32 || d == GBNORM_F16 || d == GBNORM_BF16; }

// A strided row tensor as the aliasing check sees it.
struct Mat {
    const void *p;
    int64_t ld;
    int dtype;
    size_t bytes;
};

// Outputs may not overlap inputs or each other, except that an output may be
// exactly an input (same base, row stride and element size): every element is
// then read before it is written, by the thread that writes it.
bool bad_aliasing_ex(const Mat *outs, int no, const Mat *ins, int ni) {
    for (int i = 0; i < no; ++i) {
        for (int j = 0; j < ni; ++j) {
            if (outs[i].p && outs[i].p == ins[j].p && outs[i].ld == ins[j].ld &&
                elem_size(outs[i].dtype) == elem_size(ins[j].dtype) && outs[i].bytes == ins[j].bytes)
                continue;
            if (overlap(outs[i].p, outs[i].bytes, ins[j].p, ins[j].bytes)) return true;
        }
        for (int j = i + 1; j < no; ++j)
            if (overlap(outs[i].p, outs[i].bytes, outs[j].p, outs[j].bytes)) return true;
    }
    return false;
}

// 16-byte vectors for a row tensor: aligned base and row stride.
bool vec_rows(const void *p, int64_t ld, int dtype) {
    return !p || (aligned16(p) && ((size_t)ld * (size_t)elem_size(dtype)) % 16 == 0);
}

struct ExPlan {
    const void *kernel;
    int64_t grid;
    size_t dyn;
    int cta;
    TileCfg tc;        // ring kernels
    const char *name;
    int planes = 0;    // ring kernels: parameters as fp32 planes
};

// A general-form call as the planner sees it.
struct ExCall {
    int is_ln, dir;
    int64_t M, N;
    int xdt, ydt, pdt;
    bool extra;    // residual rows (forward) or dres rows (backward)
    bool vec;      // every row tensor allows 16-byte vectors, gamma (and beta) 16-byte aligned
    bool stats16;  // backward: rstd (and mean) 16-byte aligned
    bool no_ring;  // plan as if the ring kernels did not exist (workspace bound)
};

// Slots per (device, is_ln, dir): one per table entry, the last one for the
// element-wise kernel.
constexpr int kExSlots = kExMaxVariants + 1;
// Per slot: the dynamic shared-memory limit raised, and the last (shared
// memory, occupancy) pair.
std::atomic<int> g_ex_smem_set[kMaxDev][2][2][kExSlots];
std::atomic<uint64_t> g_ex_occ[kMaxDev][2][2][kExSlots];
// Forced general-form kernel per (is_ln, dir): table index + 1 (count + 1:
// the element-wise kernel), 0 for none.
std::atomic<int> g_ex_force[2][2];
// Name of the kernel the calling thread's last general-form call launched.
thread_local const char *g_ex_last[2] = {"", ""};

int ex_occupancy(int dev, int is_ln, int dir, int slot, const void *k, int cta, size_t dyn, int *occ) {
    std::atomic<uint64_t> &cache = g_ex_occ[dev][is_ln][dir][slot];
    const uint64_t hit = cache.load(std::memory_order_relaxed);
    if (hit != 0 && (hit >> 16) == (uint64_t)dyn) {
        *occ = (int)(hit & 0xffff);
        return GBNORM_OK;
    }
    std::atomic<int> &set = g_ex_smem_set[dev][is_ln][dir][slot];
    if (dyn > 0 && !set.load(std::memory_order_acquire)) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, k) != cudaSuccess) return GBNORM_ERR_CUDA;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 g_dev[dev].smem_optin - (int)fa.sharedSizeBytes) != cudaSuccess)
            return GBNORM_ERR_CUDA;
        set.store(1, std::memory_order_release);
    }
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, k, cta, dyn) != cudaSuccess) return GBNORM_ERR_CUDA;
    if (o <= 0) return GBNORM_ERR_UNSUPPORTED;
    if (o < 0xffff) cache.store(((uint64_t)dyn << 16) | (uint64_t)o, std::memory_order_relaxed);
    *occ = o;
    return GBNORM_OK;
}

// Ring layout of a ring variant for this call: shared memory holds the
// header, gamma (and beta, forward LayerNorm) widened to fp32 planes (planes)
// or in their storage type, then the stages.  A stage is a tile of RT rows: x (then the residual rows), or x, dy
// (then dres) and the statistics windows.  About 16 KB of rows per stage, at
// least two stages per row group, at most kExRingMaxStages in all.  False if
// that does not fit.
bool exr_geometry(const ExVariant &v, const ExCall &c, int dev, bool planes, TileCfg *tc, size_t *dyn) {
    const int rpp = v.cta / v.tpr;
    const int min_stages = 2 * rpp;
    if (min_stages > kExRingMaxStages) return false;
    const size_t params = exr_param_bytes(c.N, c.pdt, c.dir == 0 && c.is_ln, planes);
    const size_t optin = (size_t)g_dev[dev].smem_optin;
    if (optin <= (size_t)kTmaHeaderBytes + params + 1024) return false;
    const size_t budget = optin - kTmaHeaderBytes - params;
    const size_t xrow = (size_t)c.N * elem_size(c.xdt), yrow = (size_t)c.N * elem_size(c.ydt);
    auto stride_of = [&](int64_t rt) {
        size_t st = exr_section((int)rt, c.N, c.xdt) * (c.extra ? 2 : 1);
        if (c.dir == 1)
            st += exr_section((int)rt, c.N, c.ydt) + ex_al128((size_t)exr_stat_floats((int)rt) * 4u * (c.is_ln ? 2u : 1u));
        return st;
    };
    const size_t per_row = xrow * (c.extra ? 2 : 1) + (c.dir == 1 ? yrow : 0);
    int64_t rt = (int64_t)((16u << 10) / per_row);
    if (rt < 1) rt = 1;
    if (rt > 64) rt = 64;
    if (rt > c.M) rt = c.M > 0 ? c.M : 1;
    while (rt > 1 && (size_t)min_stages * stride_of(rt) > budget) rt /= 2;
    const size_t stride = stride_of(rt);
    if ((size_t)min_stages * stride > budget) return false;
    int stages = (int)(budget / stride);
    if (stages > kExRingMaxStages) stages = kExRingMaxStages;
    stages -= stages % rpp;
    size_t ring = (size_t)stages * stride;
    // the backward combines its row groups' partials in the idle ring
    if (c.dir == 1 && rpp > 1) {
        const size_t comb = (size_t)v.cta * v.vpt * 8u * 4u * (c.is_ln ? 2u : 1u);
        if (comb > ring) ring = comb;
    }
    if (ring > budget) return false;
    tc->rows = (int)rt;
    tc->stages = stages;
    tc->stride = (uint32_t)stride;
    tc->fault = g_dev[dev].fault;
    *dyn = kTmaHeaderBytes + params + ring;
    return true;
}

// Plans variant i of the table for this call: false if it cannot serve it.
int ex_try(const ExCall &c, int i, int dev, ExPlan *pl, bool *ok) {
    *ok = false;
    const ExTable &t = ex_table(c.is_ln, c.dir);
    const ExVariant &v = t.v[i];
    if ((int64_t)v.tpr * v.vpt * 8 < c.N) return GBNORM_OK;
    const int64_t limit = g_grid_limit.load(std::memory_order_relaxed);
    const int sms = g_dev[dev].sms;
    int occ = 0;
    if (v.ring) {
        if (c.no_ring || (c.dir == 1 && !c.stats16)) return GBNORM_OK;
        if (v.xt >= 0 && (v.xt != c.xdt || c.ydt != c.xdt)) return GBNORM_OK;
        // gamma (beta) widened into fp32 planes (conflict-free 16-byte reads,
        // nothing to convert) where the ring still fits beside them, except
        // 16-bit gamma and beta of the LayerNorm forward, which measured
        // faster read in their storage type (one 16-byte read per 8
        // elements of each)
        TileCfg tc;
        size_t dyn;
        int planes = (c.dir == 0 && c.is_ln && c.pdt != GBNORM_F32) ? 0 : 1;
        if (!planes || !exr_geometry(v, c, dev, true, &tc, &dyn)) {
            planes = 0;
            if (!exr_geometry(v, c, dev, false, &tc, &dyn)) return GBNORM_OK;
        }
        const int st = ex_occupancy(dev, c.is_ln, c.dir, i, v.kernel, v.cta, dyn, &occ);
        if (st != GBNORM_OK) return st;
        // persistent: at most one CTA per SM
        const int64_t ntiles = (c.M + tc.rows - 1) / tc.rows;
        int64_t cap = sms;
        if (limit > 0 && limit < cap) cap = limit;
        *pl = ExPlan{v.kernel, ntiles < cap ? ntiles : cap, dyn, v.cta, tc, v.name, planes};
        *ok = true;
        return GBNORM_OK;
    }
    // fp32 parameters (forward: gamma and beta; backward: gamma, then the row
    // groups' partials of dgamma and dbeta)
    const size_t dyn = (size_t)c.N * 4u * (c.is_ln ? 2u : 1u);
    if (dyn + 4096 > (size_t)g_dev[dev].smem_optin) return GBNORM_OK;
    const int st = ex_occupancy(dev, c.is_ln, c.dir, i, v.kernel, v.cta, dyn, &occ);
    if (st != GBNORM_OK) return st;
    const int64_t rows_per_cta = v.cta / v.tpr;
    const int64_t units = (c.M + rows_per_cta - 1) / rows_per_cta;
    int64_t cap = (int64_t)occ * sms;
    if (limit > 0 && limit < cap) cap = limit;
    *pl = ExPlan{v.kernel, units < cap ? units : cap, dyn, v.cta, TileCfg{0, 0, 0, nullptr}, v.name};
    *ok = true;
    return GBNORM_OK;
}

// The first table entry that serves the call (ring kernels come first; a
// forced entry is tried before all others), else the element-wise kernel.
int ex_plan(const ExCall &c, int dev, ExPlan *pl) {
    const ExTable &t = ex_table(c.is_ln, c.dir);
    const int forced = g_ex_force[c.is_ln][c.dir].load(std::memory_order_relaxed) - 1;
    if (c.vec && c.N % 8 == 0) {
        bool ok = false;
        if (forced >= 0 && forced < t.count) {
            const int st = ex_try(c, forced, dev, pl, &ok);
            if (st != GBNORM_OK || ok) return st;
        }
        if (forced != t.count) {
            for (int i = 0; i < t.count; ++i) {
                const int st = ex_try(c, i, dev, pl, &ok);
                if (st != GBNORM_OK || ok) return st;
            }
        }
    }
    const void *k = t.elem;
    int occ = 0;
    const int st = ex_occupancy(dev, c.is_ln, c.dir, kExSlots - 1, k, kElemCTA, 0, &occ);
    if (st != GBNORM_OK) return st;
    // one partial row per CTA in the backward: at most one CTA per SM
    int64_t cap = c.dir == 0 ? (int64_t)occ * g_dev[dev].sms : (int64_t)g_dev[dev].sms;
    const int64_t limit = g_grid_limit.load(std::memory_order_relaxed);
    if (limit > 0 && limit < cap) cap = limit;
    *pl = ExPlan{k, c.M < cap ? c.M : cap, 0, kElemCTA, TileCfg{0, 0, 0, nullptr}, "exe"};
    return GBNORM_OK;
}

int launch_ex(const ExPlan &pl, void *params, cudaStream_t s) {
    void *args[1] = {params};
    if (cudaLaunchKernel(pl.kernel, dim3((unsigned)pl.grid), dim3(pl.cta), args, pl.dyn, s) != cudaSuccess)
        return GBNORM_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? GBNORM_OK : GBNORM_ERR_CUDA;
}

int do_fwd_ex(int is_ln, int64_t M, int64_t N, float eps, const void *x, int64_t ldx, int xdt,
              const void *res, int64_t ldr, void *h, int64_t ldh, const void *gamma, const void *beta,
              int pdt, void *y, int64_t ldy, int ydt, float *mean, float *rstd, cudaStream_t stream) {
    if ((is_ln != 0 && is_ln != 1) || !valid_dtype(xdt) || !valid_dtype(pdt) || !valid_dtype(ydt))
        return GBNORM_ERR_INVALID_ARG;
    if (!valid_shape(M, N, xdt) || !std::isfinite(eps) || eps < 0.f) return GBNORM_ERR_INVALID_ARG;
    if (!is_ln) {
        beta = nullptr;
        mean = nullptr;
    }
    if (!res && h) return GBNORM_ERR_INVALID_ARG;  // h is the residual sum: only with a residual
    if (!res) ldr = N;
    if (!h) ldh = N;
    if (M > 0) {
        if (!x || !y) return GBNORM_ERR_INVALID_ARG;
        for (int64_t ld : {ldx, ldr, ldh, ldy})
            if (ld < N || ld > (INT64_MAX / 16) / M) return GBNORM_ERR_INVALID_ARG;
    }
    const Mat outs[4] = {{y, ldy, ydt, span(M, N, ldy, ydt)}, {h, ldh, xdt, span(M, N, ldh, xdt)},
                         {rstd, 1, GBNORM_F32, (size_t)M * 4}, {mean, 1, GBNORM_F32, (size_t)M * 4}};
    const Mat ins[4] = {{x, ldx, xdt, span(M, N, ldx, xdt)}, {res, ldr, xdt, span(M, N, ldr, xdt)},
                        {gamma, N, pdt, (size_t)N * elem_size(pdt)}, {beta, N, pdt, (size_t)N * elem_size(pdt)}};
    if (bad_aliasing_ex(outs, 4, ins, 4)) return GBNORM_ERR_INVALID_ARG;
    int dev;
    int s = current_device(&dev);
    if (s != GBNORM_OK) return s;
    g_ex_last[0] = "";
    if (M == 0) return GBNORM_OK;
    const bool vec = vec_rows(x, ldx, xdt) && vec_rows(res, ldr, xdt) && vec_rows(h, ldh, xdt) &&
                     vec_rows(y, ldy, ydt) && aligned16(gamma) && aligned16(beta);
    ExPlan pl;
    s = ex_plan(ExCall{is_ln, 0, M, N, xdt, ydt, pdt, res != nullptr, vec, true, false}, dev, &pl);
    if (s != GBNORM_OK) return s;
    g_ex_last[0] = pl.name;
    ExFwdParams p{x, res, h, gamma, beta, y, mean, rstd, ldx, ldr, ldh, ldy, M, N, eps, xdt, pdt, ydt, pl.tc,
                  pl.planes};
    return launch_ex(pl, &p, stream);
}

// Workspace of the general backward: the largest partial-row count any plan
// of (is_ln, M, N) may use -- the element-wise and register plans, and the
// ring plans' one CTA per SM (capped by the rows).  Independent of storage
// types and extras.
size_t ex_ws_bytes(int is_ln, int64_t M, int64_t N, int dev, int *status) {
    int64_t P = M < g_dev[dev].sms ? M : g_dev[dev].sms;
    const int64_t limit = g_grid_limit.load(std::memory_order_relaxed);
    if (limit > 0 && limit < P) P = limit;
    for (bool vec : {false, true}) {
        ExPlan pl;
        *status = ex_plan(ExCall{is_ln, 1, M, N, GBNORM_F32, GBNORM_F32, GBNORM_F32, false, vec, true, true}, dev, &pl);
        if (*status != GBNORM_OK) return 0;
        if (pl.grid > P) P = pl.grid;
    }
    const size_t need = (size_t)P * (size_t)N * 4u * (is_ln ? 2u : 1u);
    return (need + 255u) & ~(size_t)255u;
}

int do_bwd_ex(int is_ln, int64_t M, int64_t N, const void *dy, int64_t lddy, int ydt, const void *x,
              int64_t ldx, int xdt, const void *dres, int64_t lddres, const void *gamma, int pdt,
              const float *mean, const float *rstd, void *dx, int64_t lddx, float *dgamma, float *dbeta,
              void *ws, size_t ws_bytes, cudaStream_t stream) {
    if ((is_ln != 0 && is_ln != 1) || !valid_dtype(xdt) || !valid_dtype(pdt) || !valid_dtype(ydt))
        return GBNORM_ERR_INVALID_ARG;
    if (!valid_shape(M, N, xdt)) return GBNORM_ERR_INVALID_ARG;
    if (!is_ln) {
        dbeta = nullptr;
        mean = nullptr;
    }
    if (!dres) lddres = N;
    if (M > 0) {
        if (!dy || !x || !rstd || !dx || (is_ln && !mean)) return GBNORM_ERR_INVALID_ARG;
        for (int64_t ld : {lddy, ldx, lddres, lddx})
            if (ld < N || ld > (INT64_MAX / 16) / M) return GBNORM_ERR_INVALID_ARG;
    }
    const Mat outs[3] = {{dx, lddx, xdt, span(M, N, lddx, xdt)}, {dgamma, N, GBNORM_F32, (size_t)N * 4},
                         {dbeta, N, GBNORM_F32, (size_t)N * 4}};
    const Mat ins[6] = {{dy, lddy, ydt, span(M, N, lddy, ydt)}, {x, ldx, xdt, span(M, N, ldx, xdt)},
                        {dres, lddres, xdt, span(M, N, lddres, xdt)},
                        {gamma, N, pdt, (size_t)N * elem_size(pdt)},
                        {rstd, 1, GBNORM_F32, (size_t)M * 4}, {mean, 1, GBNORM_F32, (size_t)M * 4}};
    if (bad_aliasing_ex(outs, 3, ins, 6)) return GBNORM_ERR_INVALID_ARG;
    // only dx may coincide with an input, and only with dy or dres
    if (dx && (dx == x || dx == static_cast<const void *>(rstd) || dx == static_cast<const void *>(mean) ||
               dx == gamma))
        return GBNORM_ERR_INVALID_ARG;
    int dev;
    int s = current_device(&dev);
    if (s != GBNORM_OK) return s;
    const size_t need = ex_ws_bytes(is_ln, M, N, dev, &s);
    if (s != GBNORM_OK) return s;
    g_ex_last[1] = "";
    int64_t P = 0;
    if (M > 0) {
        if (!ws || ws_bytes < need || !aligned16(ws)) return GBNORM_ERR_WORKSPACE;
        const Mat all_out[4] = {outs[0], outs[1], outs[2], {ws, 1, GBNORM_F32, need}};
        if (bad_aliasing_ex(all_out, 4, ins, 6)) return GBNORM_ERR_INVALID_ARG;
        const bool vec = vec_rows(dy, lddy, ydt) && vec_rows(x, ldx, xdt) && vec_rows(dres, lddres, xdt) &&
                         vec_rows(dx, lddx, xdt) && aligned16(gamma);
        const bool stats16 = aligned16(rstd) && (!is_ln || aligned16(mean));
        ExPlan pl;
        s = ex_plan(ExCall{is_ln, 1, M, N, xdt, ydt, pdt, dres != nullptr, vec, stats16, false}, dev, &pl);
        if (s != GBNORM_OK) return s;
        g_ex_last[1] = pl.name;
        ExBwdParams p{dy, x, dres, gamma, mean, rstd, dx, static_cast<float *>(ws), lddy, ldx, lddres, lddx,
                      M, N, xdt, pdt, ydt, pl.tc, pl.planes};
        s = launch_ex(pl, &p, stream);
        if (s != GBNORM_OK) return s;
        P = pl.grid;
    }
    return launch_colreduce(is_ln, static_cast<const float *>(ws), P, N, dgamma, dbeta, M > 0, stream);
}

// Stage two of every backward: column sums of the P partial rows of ws
// (P = 0 writes zeros); a NULL output's blocks return at once.  After a row
// kernel (pdl) it is launched with programmatic stream serialization.
int launch_colreduce(int is_ln, const float *wsc, int64_t P, int64_t N, float *dgamma, float *dbeta, bool pdl,
                     cudaStream_t stream) {
    if (!dgamma && !dbeta) return GBNORM_OK;
    const bool v4 = (N % 4) == 0;
    const int64_t cols_per_cta = 32 * (v4 ? 4 : 1);
    const dim3 grid2((unsigned)((N + cols_per_cta - 1) / cols_per_cta), is_ln ? 2u : 1u);
    void *args[5] = {&wsc, &P, &N, &dgamma, &dbeta};
    // Programmatic stream serialization: the column reduce may be scheduled
    // while the row kernel drains; it waits (griddepcontrol.wait) for that
    // grid's completion before reading the workspace.
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid2;
    cfg.blockDim = dim3(kColCTA);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (cudaLaunchKernelExC(&cfg, v4 ? kColReduceVec4 : kColReduceScalar, args) != cudaSuccess)
        return GBNORM_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? GBNORM_OK : GBNORM_ERR_CUDA;
}

}  // namespace
}  // namespace gbn

using namespace gbn;

extern "C" {

int rmsnorm_fwd(const void *x, const void *gamma, void *y, float *rstd, int64_t M, int64_t N,
                int dtype, float eps, gbnorm_stream_t stream) {
    return do_fwd(0, x, gamma, nullptr, y, nullptr, rstd, M, N, dtype, eps,
                  reinterpret_cast<cudaStream_t>(stream));
}

int layernorm_fwd(const void *x, const void *gamma, const void *beta, void *y, float *mean,
                  float *rstd, int64_t M, int64_t N, int dtype, float eps,
                  gbnorm_stream_t stream) {
    return do_fwd(1, x, gamma, beta, y, mean, rstd, M, N, dtype, eps,
                  reinterpret_cast<cudaStream_t>(stream));
}

size_t norm_bwd_workspace_size(int is_layernorm, int64_t M, int64_t N, int dtype) {
    if (!valid_shape(M, N, dtype)) return 0;
    int dev;
    if (current_device(&dev) != GBNORM_OK) return 0;
    int st = GBNORM_OK;
    const size_t b = ws_bytes_for(is_layernorm ? 1 : 0, M, N, dtype, dev, &st);
    if (st != GBNORM_OK) return 0;
    return b > 256 ? b : 256;
}

int rmsnorm_bwd(const void *dy, const void *x, const void *gamma, const float *rstd, void *dx,
                float *dgamma, void *workspace, size_t workspace_bytes, int64_t M, int64_t N,
                int dtype, gbnorm_stream_t stream) {
    return do_bwd(0, dy, x, gamma, nullptr, rstd, dx, dgamma, nullptr, workspace, workspace_bytes,
                  M, N, dtype, reinterpret_cast<cudaStream_t>(stream));
}

int layernorm_bwd(const void *dy, const void *x, const void *gamma, const float *mean,
                  const float *rstd, void *dx, float *dgamma, float *dbeta, void *workspace,
                  size_t workspace_bytes, int64_t M, int64_t N, int dtype,
                  gbnorm_stream_t stream) {
    return do_bwd(1, dy, x, gamma, mean, rstd, dx, dgamma, dbeta, workspace, workspace_bytes, M, N,
                  dtype, reinterpret_cast<cudaStream_t>(stream));
}

int norm_fwd_ex(int is_layernorm, int64_t M, int64_t N, float eps, const void *x, int64_t ldx, int x_dtype,
                const void *residual, int64_t ldr, void *h, int64_t ldh, const void *gamma, const void *beta,
                int param_dtype, void *y, int64_t ldy, int y_dtype, float *mean, float *rstd,
                gbnorm_stream_t stream) {
    return do_fwd_ex(is_layernorm, M, N, eps, x, ldx, x_dtype, residual, ldr, h, ldh, gamma, beta, param_dtype,
                     y, ldy, y_dtype, mean, rstd, reinterpret_cast<cudaStream_t>(stream));
}

size_t norm_bwd_ex_workspace_size(int is_layernorm, int64_t M, int64_t N) {
    if ((is_layernorm != 0 && is_layernorm != 1) || !valid_shape(M, N, GBNORM_F32)) return 0;
    int dev;
    if (current_device(&dev) != GBNORM_OK) return 0;
    int st = GBNORM_OK;
    const size_t b = ex_ws_bytes(is_layernorm, M, N, dev, &st);
    if (st != GBNORM_OK) return 0;
    return b > 256 ? b : 256;
}

int norm_bwd_ex(int is_layernorm, int64_t M, int64_t N, const void *dy, int64_t lddy, int y_dtype,
                const void *x, int64_t ldx, int x_dtype, const void *dres, int64_t lddres, const void *gamma,
                int param_dtype, const float *mean, const float *rstd, void *dx, int64_t lddx, float *dgamma,
                float *dbeta, void *workspace, size_t workspace_bytes, gbnorm_stream_t stream) {
    return do_bwd_ex(is_layernorm, M, N, dy, lddy, y_dtype, x, ldx, x_dtype, dres, lddres, gamma, param_dtype,
                     mean, rstd, dx, lddx, dgamma, dbeta, workspace, workspace_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

const char *gbnorm_status_string(int status) {
    switch (status) {
    case GBNORM_OK: return "ok";
    case GBNORM_ERR_INVALID_ARG: return "invalid argument";
    case GBNORM_ERR_UNSUPPORTED: return "unsupported (needs an sm_103a device)";
    case GBNORM_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case GBNORM_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
    }
}

int gbnorm_variant_name(int is_layernorm, int dir, int64_t M, int64_t N, int dtype, int aligned,
                        char *buf, size_t len) {
    if (!valid_shape(M, N, dtype) || (dir != 0 && dir != 1) || !buf || len == 0)
        return GBNORM_ERR_INVALID_ARG;
    int dev;
    const int s = current_device(&dev);
    if (s != GBNORM_OK) return s;
    const int E = 16 / elem_size(dtype);
    CallShape c{is_layernorm ? 1 : 0, dir, dtype, M, N, aligned && (N % E) == 0, aligned != 0};
    Plan pl;
    const int st = plan_call(c, dev, &pl);
    if (st != GBNORM_OK) return st;
    std::snprintf(buf, len, "%s", kTables[c.is_ln][dir][dtype]->v[pl.idx].name);
    return GBNORM_OK;
}

int gbnorm_force_variant(int is_layernorm, int dir, int dtype, const char *name) {
    if ((dir != 0 && dir != 1) || dtype < 0 || dtype > 2) return GBNORM_ERR_INVALID_ARG;
    const int ln = is_layernorm ? 1 : 0;
    if (!name || !name[0]) {
        g_force[ln][dir][dtype].store(0);
        return GBNORM_OK;
    }
    const int i = find_variant(*kTables[ln][dir][dtype], name);
    if (i < 0) return GBNORM_ERR_INVALID_ARG;
    g_force[ln][dir][dtype].store(i + 1);
    return GBNORM_OK;
}

int gbnorm_variant_count(int is_layernorm, int dir, int dtype) {
    if ((dir != 0 && dir != 1) || dtype < 0 || dtype > 2) return 0;
    return kTables[is_layernorm ? 1 : 0][dir][dtype]->count;
}

const char *gbnorm_variant_at(int is_layernorm, int dir, int dtype, int index) {
    if ((dir != 0 && dir != 1) || dtype < 0 || dtype > 2) return nullptr;
    const VariantTable &t = *kTables[is_layernorm ? 1 : 0][dir][dtype];
    return (index >= 0 && index < t.count) ? t.v[index].name : nullptr;
}

int gbnorm_ex_variant_count(int is_layernorm, int dir) {
    if (dir != 0 && dir != 1) return 0;
    return ex_table(is_layernorm ? 1 : 0, dir).count + 1;
}

const char *gbnorm_ex_variant_at(int is_layernorm, int dir, int index) {
    if (dir != 0 && dir != 1) return nullptr;
    const ExTable &t = ex_table(is_layernorm ? 1 : 0, dir);
    if (index == t.count) return "exe";
    return (index >= 0 && index < t.count) ? t.v[index].name : nullptr;
}

int gbnorm_ex_force_variant(int is_layernorm, int dir, const char *name) {
    if (dir != 0 && dir != 1) return GBNORM_ERR_INVALID_ARG;
    const int ln = is_layernorm ? 1 : 0;
    if (!name || !name[0]) {
        g_ex_force[ln][dir].store(0);
        return GBNORM_OK;
    }
    const ExTable &t = ex_table(ln, dir);
    for (int i = 0; i <= t.count; ++i) {
        if (std::strcmp(gbnorm_ex_variant_at(ln, dir, i), name) == 0) {
            g_ex_force[ln][dir].store(i + 1);
            return GBNORM_OK;
        }
    }
    return GBNORM_ERR_INVALID_ARG;
}

int gbnorm_ex_last_variant(int dir, char *buf, size_t len) {
    if ((dir != 0 && dir != 1) || !buf || len == 0) return GBNORM_ERR_INVALID_ARG;
    std::snprintf(buf, len, "%s", g_ex_last[dir]);
    return GBNORM_OK;
}

int gbnorm_set_grid_limit(int max_ctas) {
    if (max_ctas < 0) return GBNORM_ERR_INVALID_ARG;
    g_grid_limit.store(max_ctas);
    return GBNORM_OK;
}

int gbnorm_read_fault(int reset, int *value) {
    if (!value) return GBNORM_ERR_INVALID_ARG;
    int dev;
    const int s = current_device(&dev);
    if (s != GBNORM_OK) return s;
    if (cudaMemcpyFromSymbol(value, g_fault_word, sizeof(int)) != cudaSuccess) return GBNORM_ERR_CUDA;
    if (reset) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(int)) != cudaSuccess) return GBNORM_ERR_CUDA;
    }
    return GBNORM_OK;
}

}  // extern "C"
