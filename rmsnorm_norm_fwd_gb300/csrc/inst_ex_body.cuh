// inst_ex_body.cuh -- general-form kernel instantiations of one direction
// (the including unit defines GBN_EX_DIR: 0 forward, 1 backward).  Ring
// kernels come in four builds per geometry: the row storage type fixed to
// bf16, fp16 or fp32 (taken when x and y / dy share that type), then the
// build that reads every type from the call.
#include "ex_kernels.cuh"

namespace gbn {

// Register kernels (TPR, VPT, CTA, MINB): capacity TPR * VPT * 8 elements,
// MINB CTAs per SM of the launch bound.  The backward holds four arrays of
// VPT * 8 floats per thread (x - mean, dy, dgamma and dbeta sums): more
// threads per row, fewer chunks each.
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

#if GBN_EX_DIR == 0
#define GBN_EXR_K(LN, TPR, VPT, NT, XT) fwd_exr<LN, TPR, VPT, NT, XT>
#define GBN_EXR_NAME(TPR, VPT, NT, SFX) "exrf" #TPR "x" #VPT "b" #NT SFX
#define GBN_EXG(LN, TPR, VPT, CTA, MINB) \
    ExVariant{"exf" #TPR "x" #VPT "b" #CTA, (const void *)&fwd_ex<LN, TPR, VPT, CTA, MINB>, TPR, VPT, CTA},
#define GBN_EX_GEOMS GBN_EXF_GEOMS
#define GBN_EX_ELEM(LN) (const void *)&fwd_exe<LN>
#define GBN_EX_TABLES kExFwdTables
#else
#define GBN_EXR_K(LN, TPR, VPT, NT, XT) bwd_exr<LN, TPR, VPT, NT, XT>
#define GBN_EXR_NAME(TPR, VPT, NT, SFX) "exrb" #TPR "x" #VPT "b" #NT SFX
#define GBN_EXG(LN, TPR, VPT, CTA, MINB) \
    ExVariant{"exb" #TPR "x" #VPT "b" #CTA, (const void *)&bwd_ex<LN, TPR, VPT, CTA, MINB>, TPR, VPT, CTA},
#define GBN_EX_GEOMS GBN_EXB_GEOMS
#define GBN_EX_ELEM(LN) (const void *)&bwd_exe<LN>
#define GBN_EX_TABLES kExBwdTables
#endif

#define GBN_EXR1(LN, TPR, VPT, NT, XT, SFX) \
    ExVariant{GBN_EXR_NAME(TPR, VPT, NT, SFX), (const void *)&GBN_EXR_K(LN, TPR, VPT, NT, XT), TPR, VPT, NT, 1, XT},
#define GBN_EXR4(LN, TPR, VPT, NT)                                                        \
    GBN_EXR1(LN, TPR, VPT, NT, 2, "_bf16") GBN_EXR1(LN, TPR, VPT, NT, 1, "_fp16")          \
    GBN_EXR1(LN, TPR, VPT, NT, 0, "_fp32") GBN_EXR1(LN, TPR, VPT, NT, -1, "")
#define GBN_EXR_RMS(TPR, VPT, NT) GBN_EXR4(false, TPR, VPT, NT)
#define GBN_EXR_LN(TPR, VPT, NT) GBN_EXR4(true, TPR, VPT, NT)
#define GBN_EXG_RMS(TPR, VPT, CTA, MINB) GBN_EXG(false, TPR, VPT, CTA, MINB)
#define GBN_EXG_LN(TPR, VPT, CTA, MINB) GBN_EXG(true, TPR, VPT, CTA, MINB)

static const ExVariant ex_rms[] = {GBN_EXR_GEOMS(GBN_EXR_RMS) GBN_EX_GEOMS(GBN_EXG_RMS)};
static const ExVariant ex_ln[] = {GBN_EXR_GEOMS(GBN_EXR_LN) GBN_EX_GEOMS(GBN_EXG_LN)};

#define GBN_N(a) (int)(sizeof(a) / sizeof(ExVariant))
static_assert(GBN_N(ex_rms) < kExMaxVariants && GBN_N(ex_ln) < kExMaxVariants,
              "one planner slot per entry, one for exe");
const ExTable GBN_EX_TABLES[2] = {
    {ex_rms, GBN_N(ex_rms), GBN_EX_ELEM(false)},
    {ex_ln, GBN_N(ex_ln), GBN_EX_ELEM(true)},
};

}  // namespace gbn
