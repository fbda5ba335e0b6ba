// params.h -- kernel argument blocks and the variant descriptor shared by the
// kernel instantiation units and the host API.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace gbn {

constexpr int kElemCTA = 256;  // threads per CTA of the element-wise kernels
constexpr int kColCTA = 512;   // threads per CTA of the column-reduce kernel
constexpr int kTmaHeaderBytes = 2048;  // TMA kernels: barriers, abort flag, reduction scratch
constexpr int kTmaMaxStages = 8;       // TMA kernels: deepest shared-memory ring
constexpr int kExRingMaxStages = 16;   // general-form ring kernels: deepest ring (2 per row group)
constexpr int kSkPartBytes = 16 * 128 * 4;  // single-kernel column reduce: band sums in shared memory

// Pipeline geometry of the TMA-staged kernels, chosen by the host per call.
struct TileCfg {
    int rows;          // rows per tile (one bulk copy per tensor per tile)
    int stages;        // tiles in flight (shared-memory ring depth)
    uint32_t stride;   // bytes between consecutive stages in shared memory
    int *fault;        // device word set to nonzero if a bounded wait gives up
};

struct FwdParams {
    const void *x;      // [M, N] T
    const void *gamma;  // [N] T
    const void *beta;   // [N] T (LayerNorm only)
    void *y;            // [M, N] T
    float *mean;        // [M] or null (LayerNorm only)
    float *rstd;        // [M] or null
    int64_t M, N;
    float eps;
    TileCfg tc;         // used by the TMA-staged kernels only
};

struct BwdParams {
    const void *dy;     // [M, N] T
    const void *x;      // [M, N] T
    const void *gamma;  // [N] T
    const float *mean;  // [M] (LayerNorm only)
    const float *rstd;  // [M]
    void *dx;           // [M, N] T
    float *ws;          // [2][P][N] float partial rows (second block: dbeta), then P flag words
    int64_t M, N;
    TileCfg tc;         // used by the TMA-staged kernels only
    // Single-kernel variants only (they reduce the partial rows themselves):
    float *dgamma;      // [N] or null
    float *dbeta;       // [N] or null
    uint32_t epoch;     // nonzero, different for every call of the process
};

// General form (strided rows, a storage type per tensor, fused residual
// add).  Strides (ld*) are in elements; dtypes are gbnorm_dtype_t codes.
// Shared-memory layout of the general-form ring kernels (host and device
// agree on it): after the header, gamma (and beta) in their storage type
// (dt 0: fp32, else 16-bit), then the stages; a stage holds one section per
// row tensor of its tile of rt rows (x, then the residual rows; or x, dy,
// dres), each 128-byte aligned.  With `planes`, gamma (and beta) are held
// widened to fp32 whatever their storage type.
__host__ __device__ inline size_t ex_al128(size_t b) { return (b + 127) & ~(size_t)127; }
__host__ __device__ inline size_t exr_param_bytes(int64_t N, int pdt, bool two, bool planes = false) {
    return ex_al128((size_t)N * (planes || pdt == 0 ? 4 : 2)) * (two ? 2 : 1);
}
__host__ __device__ inline size_t exr_section(int rt, int64_t N, int dt) {
    return ex_al128((size_t)rt * (size_t)N * (dt == 0 ? 4 : 2));
}
// Floats reserved per saved statistic per backward stage: the widest
// 16-byte-aligned window of rt rows.
__host__ __device__ constexpr int exr_stat_floats(int rt) { return (rt + 7) & ~3; }

struct ExFwdParams {
    const void *x;      // [M, ldx] xdt
    const void *res;    // [M, ldr] xdt, or null (no residual add)
    void *h;            // [M, ldh] xdt: x + res as normalised, or null (not stored)
    const void *gamma;  // [N] pdt, or null (1)
    const void *beta;   // [N] pdt, or null (0; LayerNorm only)
    void *y;            // [M, ldy] ydt
    float *mean;        // [M] or null (LayerNorm only)
    float *rstd;        // [M] or null
    int64_t ldx, ldr, ldh, ldy;
    int64_t M, N;
    float eps;
    int xdt, pdt, ydt;
    TileCfg tc;  // ring kernels: rows per tile, stages, stage stride, fault word
    int planes;  // ring kernels: gamma (beta) widened to fp32 planes in shared memory, else kept raw
};

struct ExBwdParams {
    const void *dy;     // [M, lddy] ydt
    const void *x;      // [M, ldx] xdt: the normalised rows (h with a residual add)
    const void *dres;   // [M, lddres] xdt: gradient reaching x from elsewhere, or null
    const void *gamma;  // [N] pdt, or null (1)
    const float *mean;  // [M] (LayerNorm only)
    const float *rstd;  // [M]
    void *dx;           // [M, lddx] xdt
    float *ws;          // [2][P][N] float partial rows (second block: dbeta)
    int64_t lddy, ldx, lddres, lddx;
    int64_t M, N;
    int xdt, pdt, ydt;
    TileCfg tc;  // ring kernels: rows per tile, stages, stage stride, fault word
    int planes;  // ring kernels: gamma widened to fp32 planes in shared memory, else kept raw
};

enum VariantKind : int {
    kRows = 0,  // row-resident registers, plain 16-byte loads
    kElem = 1,  // element-wise, any N and alignment
    kTma = 2,   // rows staged through a shared-memory ring by bulk async copies
    kTmaCl = 3, // as kTma, each row split across a thread-block cluster (column slices)
    kWide = 4,  // one CTA per row, the row streamed twice (DRAM, then L2); any row length
    kRowsS = 5, // as kRows (no cluster), gamma/beta in shared memory as fp32
    kTmaP = 6,  // as kTma without a producer warp (one thread of the CTA refills the ring)
    kWtma = 7,  // one CTA per row, the row streamed twice through a bulk-copy ring (forward)
    kWtmaC = 8, // column slices of a cluster streamed twice through a bulk-copy ring (backward)
    kWideR = 9, // as kWide (backward), the dgamma/dbeta sums in registers, gamma in shared memory
    kWcs = 10,  // cluster column slices of each row resident in shared memory (bulk-copy ring)
    kWideF = 11, // forward on kWideR's layout: cluster column slices, gamma/beta slices in shared memory
};

// One compiled kernel and the geometry the host needs to launch it.
struct Variant {
    const char *name;
    const void *kernel;  // __global__ entry (takes FwdParams or BwdParams by value)
    int kind;            // VariantKind
    int tpr;             // threads per row group (within one CTA)
    int vpt;             // 16-byte vectors per thread per row (max); kWide: vectors per batch
    int rows;            // rows per row group per iteration (kRows, kWide); rows per exchange step (kTmaCl)
    int cl;              // CTAs per row (thread-block cluster size)
    int cta;             // threads per CTA
    int elems_per_vec;   // E (16 bytes / sizeof(T)); 1 for element-wise kernels
    int ctas_per_sm;     // kTma: CTAs meant to share an SM (shared-memory budget split); kWide: launch bound
    int stage_target;    // kTma: bytes of one stage the host aims for
    int fused = 0;       // 1: the kernel also sums the partial rows (cooperative launch, no column reduce)
    int db = 0;          // kWideR: 1 the dbeta sums (and gamma, in its storage type) in shared memory; 2 the sums only
    int raw = 0;         // kRowsS: 1 gamma (and beta) staged in their storage type, not as fp32

    // Longest row (elements) this variant can hold.
    int64_t max_n() const {
        return (kind == kElem || kind == kWide || kind == kWtma) ? INT64_MAX
                                                                 : (int64_t)tpr * vpt * cl * elems_per_vec;
        // (kWtmaC: tpr = consumer threads, vpt = chunks per slice)
    }
    // Threads of a CTA that work on rows (TMA kinds add one producer warp).
    int consumers() const {
        return (kind == kTma || kind == kTmaCl || kind == kWtma || kind == kWtmaC) ? cta - 32 : cta;
    }
    bool staged_rows() const { return kind == kTma || kind == kTmaP; }
    int rows_per_cta_iter() const {
        return (kind == kRows || kind == kRowsS) ? (cta / tpr) * rows
                                                 : ((kind == kWide || kind == kWideR || kind == kWideF) && cl == 1)
                                                       ? rows
                                                       : 1;
    }
};

struct VariantTable {
    const Variant *v;
    int count;
};

// Tables defined by the instantiation units (one unit per dtype and direction).
extern const VariantTable kFwdRms_f32, kFwdLn_f32, kBwdRms_f32, kBwdLn_f32;
extern const VariantTable kFwdRms_f16, kFwdLn_f16, kBwdRms_f16, kBwdLn_f16;
extern const VariantTable kFwdRms_bf16, kFwdLn_bf16, kBwdRms_bf16, kBwdLn_bf16;
extern const void *const kColReduceVec4;
extern const void *const kColReduceScalar;

// General-form kernels (ex_kernels.cuh): row-resident geometries in order of
// row capacity, and the element-wise kernel; [is_ln][dir].
struct ExVariant {
    const char *name;
    const void *kernel;
    int tpr, vpt, cta;  // capacity tpr * vpt * 8 elements
    int ring = 0;       // rows staged through a bulk-copy ring (else read into registers)
    int xt = -1;        // ring: storage type of the rows fixed at compile time (x = y, dy), -1 any
};
struct ExTable {
    const ExVariant *v;
    int count;
    const void *elem;
};
constexpr int kExMaxVariants = 48;  // entries per table (the planner keeps one slot each, and one for exe)
extern const ExTable kExFwdTables[2], kExBwdTables[2];  // [is_ln]
inline const ExTable &ex_table(int is_ln, int dir) { return dir ? kExBwdTables[is_ln] : kExFwdTables[is_ln]; }

}  // namespace gbn
