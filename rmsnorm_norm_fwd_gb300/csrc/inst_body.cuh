// inst_body.cuh -- instantiates every kernel variant of one dtype and one
// direction.  The including unit defines GBN_T (element type), GBN_SFX (table
// name suffix) and exactly one of GBN_FWD / GBN_BWD.
#include "norm_kernels.cuh"
#include "variants.inc"

namespace gbn {

#define GBN_CAT2(a, b) a##b
#define GBN_CAT(a, b) GBN_CAT2(a, b)

#ifdef GBN_FWD
#define GBN_ROW(LN, TPR, VPT, R, CL, CTA)                                                     \
    Variant{GBN_VNAME(TPR, VPT, R, CL, CTA), (const void *)&fwd_rows<GBN_T, LN, TPR, VPT, R, CL, CTA>, \
            TPR, VPT, R, CL, CTA, VecTraits<GBN_T>::E},
#define GBN_X_RMS(TPR, VPT, R, CL, CTA) GBN_ROW(false, TPR, VPT, R, CL, CTA)
#define GBN_X_LN(TPR, VPT, R, CL, CTA) GBN_ROW(true, TPR, VPT, R, CL, CTA)
static const Variant rms_variants[] = {
    GBN_FWD_GEOMS(GBN_X_RMS)
    Variant{"elem", (const void *)&fwd_elem<GBN_T, false>, kElemCTA, 0, 1, 1, kElemCTA, 1}};
static const Variant ln_variants[] = {
    GBN_FWD_GEOMS(GBN_X_LN)
    Variant{"elem", (const void *)&fwd_elem<GBN_T, true>, kElemCTA, 0, 1, 1, kElemCTA, 1}};
const VariantTable GBN_CAT(kFwdRms_, GBN_SFX) = {rms_variants, (int)(sizeof(rms_variants) / sizeof(Variant))};
const VariantTable GBN_CAT(kFwdLn_, GBN_SFX) = {ln_variants, (int)(sizeof(ln_variants) / sizeof(Variant))};
#endif

#ifdef GBN_BWD
#define GBN_ROW(LN, TPR, VPT, R, CL, CTA)                                                     \
    Variant{GBN_VNAME(TPR, VPT, R, CL, CTA), (const void *)&bwd_rows<GBN_T, LN, TPR, VPT, R, CL, CTA>, \
            TPR, VPT, R, CL, CTA, VecTraits<GBN_T>::E},
#define GBN_X_RMS(TPR, VPT, R, CL, CTA) GBN_ROW(false, TPR, VPT, R, CL, CTA)
#define GBN_X_LN(TPR, VPT, R, CL, CTA) GBN_ROW(true, TPR, VPT, R, CL, CTA)
static const Variant rms_variants[] = {
    GBN_BWD_GEOMS(GBN_X_RMS)
    Variant{"elem", (const void *)&bwd_elem<GBN_T, false>, kElemCTA, 0, 1, 1, kElemCTA, 1}};
static const Variant ln_variants[] = {
    GBN_BWD_GEOMS(GBN_X_LN)
    Variant{"elem", (const void *)&bwd_elem<GBN_T, true>, kElemCTA, 0, 1, 1, kElemCTA, 1}};
const VariantTable GBN_CAT(kBwdRms_, GBN_SFX) = {rms_variants, (int)(sizeof(rms_variants) / sizeof(Variant))};
const VariantTable GBN_CAT(kBwdLn_, GBN_SFX) = {ln_variants, (int)(sizeof(ln_variants) / sizeof(Variant))};
#endif

}  // namespace gbn
