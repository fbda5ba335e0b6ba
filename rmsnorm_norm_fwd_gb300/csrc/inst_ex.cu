// General-form kernel instantiations (strided rows, a storage type per
// tensor, fused residual add): one kernel per geometry serves every
// combination of storage types.
#include "ex_kernels.cuh"

namespace gbn {

// (TPR, VPT, CTA): capacity TPR * VPT * 8 elements per row.
#define GBN_EX_GEOMS(X) \
    X(32, 1, 256)       \
    X(32, 2, 256)       \
    X(64, 2, 256)       \
    X(128, 2, 256)      \
    X(128, 4, 256)      \
    X(256, 4, 256)      \
    X(512, 4, 512)

#define GBN_EX(LN, TPR, VPT, CTA)                                                                     \
    ExVariant{"ex" #TPR "x" #VPT "b" #CTA, (const void *)&fwd_ex<LN, TPR, VPT, CTA>,                 \
              (const void *)&bwd_ex<LN, TPR, VPT, CTA>, TPR, VPT, CTA},
#define GBN_EX_RMS(TPR, VPT, CTA) GBN_EX(false, TPR, VPT, CTA)
#define GBN_EX_LN(TPR, VPT, CTA) GBN_EX(true, TPR, VPT, CTA)

static const ExVariant ex_rms[] = {GBN_EX_GEOMS(GBN_EX_RMS)};
static const ExVariant ex_ln[] = {GBN_EX_GEOMS(GBN_EX_LN)};

const ExTable kExTables[2] = {
    {ex_rms, (int)(sizeof(ex_rms) / sizeof(ExVariant)), (const void *)&fwd_exe<false>,
     (const void *)&bwd_exe<false>},
    {ex_ln, (int)(sizeof(ex_ln) / sizeof(ExVariant)), (const void *)&fwd_exe<true>,
     (const void *)&bwd_exe<true>},
};

}  // namespace gbn
