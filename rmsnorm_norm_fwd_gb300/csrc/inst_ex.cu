// General-form kernel instantiations (strided rows, a storage type per
// tensor, fused residual add): one kernel per geometry serves every
// combination of storage types.
#include "ex_kernels.cuh"

namespace gbn {

// (TPR, VPT, CTA, MINB): capacity TPR * VPT * 8 elements, MINB CTAs per SM of
// the launch bound.  The backward holds four arrays of VPT * 8 floats per
// thread (x - mean, dy, dgamma and dbeta sums): more threads per row, fewer
// chunks each.
#define GBN_EXF_GEOMS(X) \
    X(32, 1, 256, 4)     \
    X(32, 2, 256, 4)     \
    X(64, 2, 256, 4)     \
    X(128, 2, 256, 4)    \
    X(128, 4, 256, 2)    \
    X(256, 4, 256, 2)    \
    X(512, 4, 512, 1)

#define GBN_EXB_GEOMS(X) \
    X(32, 1, 256, 4)     \
    X(64, 1, 256, 4)     \
    X(128, 1, 256, 4)    \
    X(256, 1, 256, 4)    \
    X(512, 1, 512, 2)    \
    X(512, 2, 512, 1)    \
    X(512, 4, 512, 1)

// Ring kernels (TPR, VPT, NT): one CTA of NT threads per SM, NT / TPR row
// groups; capacity TPR * VPT * 8 elements.  Tried before the register
// kernels, in this order (512 x 2 after 256 x 4: the same capacity, measured
// slower, but one row group needs only two stages where two groups' four do
// not fit).
#define GBN_EXR_GEOMS(X) \
    X(64, 1, 512)        \
    X(64, 2, 512)        \
    X(128, 2, 512)       \
    X(128, 4, 512)       \
    X(256, 4, 512)       \
    X(512, 2, 512)       \
    X(512, 4, 512)

#define GBN_EXRF(LN, TPR, VPT, NT) \
    ExVariant{"exrf" #TPR "x" #VPT "b" #NT, (const void *)&fwd_exr<LN, TPR, VPT, NT>, TPR, VPT, NT, 1},
#define GBN_EXRB(LN, TPR, VPT, NT) \
    ExVariant{"exrb" #TPR "x" #VPT "b" #NT, (const void *)&bwd_exr<LN, TPR, VPT, NT>, TPR, VPT, NT, 1},
#define GBN_EXRF_RMS(TPR, VPT, NT) GBN_EXRF(false, TPR, VPT, NT)
#define GBN_EXRF_LN(TPR, VPT, NT) GBN_EXRF(true, TPR, VPT, NT)
#define GBN_EXRB_RMS(TPR, VPT, NT) GBN_EXRB(false, TPR, VPT, NT)
#define GBN_EXRB_LN(TPR, VPT, NT) GBN_EXRB(true, TPR, VPT, NT)

#define GBN_EXF(LN, TPR, VPT, CTA, MINB) \
    ExVariant{"exf" #TPR "x" #VPT "b" #CTA, (const void *)&fwd_ex<LN, TPR, VPT, CTA, MINB>, TPR, VPT, CTA},
#define GBN_EXB(LN, TPR, VPT, CTA, MINB) \
    ExVariant{"exb" #TPR "x" #VPT "b" #CTA, (const void *)&bwd_ex<LN, TPR, VPT, CTA, MINB>, TPR, VPT, CTA},
#define GBN_EXF_RMS(TPR, VPT, CTA, MINB) GBN_EXF(false, TPR, VPT, CTA, MINB)
#define GBN_EXF_LN(TPR, VPT, CTA, MINB) GBN_EXF(true, TPR, VPT, CTA, MINB)
#define GBN_EXB_RMS(TPR, VPT, CTA, MINB) GBN_EXB(false, TPR, VPT, CTA, MINB)
#define GBN_EXB_LN(TPR, VPT, CTA, MINB) GBN_EXB(true, TPR, VPT, CTA, MINB)

static const ExVariant exf_rms[] = {GBN_EXR_GEOMS(GBN_EXRF_RMS) GBN_EXF_GEOMS(GBN_EXF_RMS)};
static const ExVariant exf_ln[] = {GBN_EXR_GEOMS(GBN_EXRF_LN) GBN_EXF_GEOMS(GBN_EXF_LN)};
static const ExVariant exb_rms[] = {GBN_EXR_GEOMS(GBN_EXRB_RMS) GBN_EXB_GEOMS(GBN_EXB_RMS)};
static const ExVariant exb_ln[] = {GBN_EXR_GEOMS(GBN_EXRB_LN) GBN_EXB_GEOMS(GBN_EXB_LN)};

#define GBN_N(a) (int)(sizeof(a) / sizeof(ExVariant))
static_assert(GBN_N(exf_rms) < 33 && GBN_N(exb_rms) < 33, "one planner slot per entry, one for exe");
const ExTable kExTables[2][2] = {
    {{exf_rms, GBN_N(exf_rms), (const void *)&fwd_exe<false>}, {exb_rms, GBN_N(exb_rms), (const void *)&bwd_exe<false>}},
    {{exf_ln, GBN_N(exf_ln), (const void *)&fwd_exe<true>}, {exb_ln, GBN_N(exb_ln), (const void *)&bwd_exe<true>}},
};

}  // namespace gbn
