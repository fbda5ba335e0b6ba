// params.h -- kernel argument blocks and the variant descriptor shared by the
// kernel instantiation units and the host API.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace gbn {

constexpr int kElemCTA = 256;  // threads per CTA of the element-wise kernels
constexpr int kColCTA = 512;   // threads per CTA of the column-reduce kernel

struct FwdParams {
    const void *x;      // [M, N] T
    const void *gamma;  // [N] T
    const void *beta;   // [N] T (LayerNorm only)
    void *y;            // [M, N] T
    float *mean;        // [M] or null (LayerNorm only)
    float *rstd;        // [M] or null
    int64_t M, N;
    float eps;
};

struct BwdParams {
    const void *dy;     // [M, N] T
    const void *x;      // [M, N] T
    const void *gamma;  // [N] T
    const float *mean;  // [M] (LayerNorm only)
    const float *rstd;  // [M]
    void *dx;           // [M, N] T
    float *ws;          // [2][P][N] float partial rows (second block: dbeta)
    int64_t M, N;
};

// One compiled kernel and the geometry the host needs to launch it.
struct Variant {
    const char *name;
    const void *kernel;  // __global__ entry (takes FwdParams or BwdParams by value)
    int tpr;             // threads per row group (within one CTA)
    int vpt;             // 16-byte vectors per thread per row (0: element-wise kernel)
    int rows;            // rows each row group handles per iteration
    int cl;              // CTAs per row (thread-block cluster size)
    int cta;             // threads per CTA
    int elems_per_vec;   // E (16 bytes / sizeof(T)); 1 for element-wise kernels

    // Longest row (elements) this variant can hold.
    int64_t max_n() const {
        return vpt == 0 ? INT64_MAX : (int64_t)tpr * vpt * cl * elems_per_vec;
    }
    int rows_per_cta_iter() const { return vpt == 0 ? 1 : (cta / tpr) * rows; }
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

}  // namespace gbn
