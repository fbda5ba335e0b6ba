// inst_body.cuh -- instantiates every kernel variant of one dtype and one
// direction.  The including unit defines GBN_T (element type), GBN_SFX (table
// name suffix) and exactly one of GBN_FWD / GBN_BWD.
#include "norm_kernels.cuh"
#include "tma_kernels.cuh"
#include "tma_cluster_kernels.cuh"
#include "wide_kernels.cuh"
#include "wtma_kernels.cuh"
#include "wcs_kernels.cuh"
#include "variants.inc"

namespace gbn {

#define GBN_CAT2(a, b) a##b
#define GBN_CAT(a, b) GBN_CAT2(a, b)

#ifdef GBN_FWD
#define GBN_ROW(LN, TPR, VPT, R, CL, CTA)                                                     \
    Variant{GBN_VNAME(TPR, VPT, R, CL, CTA), (const void *)&fwd_rows<GBN_T, LN, TPR, VPT, R, CL, CTA>, \
            kRows, TPR, VPT, R, CL, CTA, VecTraits<GBN_T>::E, 0, 0},
#define GBN_X_RMS(TPR, VPT, R, CL, CTA) GBN_ROW(false, TPR, VPT, R, CL, CTA)
#define GBN_X_LN(TPR, VPT, R, CL, CTA) GBN_ROW(true, TPR, VPT, R, CL, CTA)
#define GBN_TMA(LN, TPR, VPT, CW)                                                              \
    Variant{GBN_TMA_VNAME(TPR, VPT, CW), (const void *)&fwd_tma<GBN_T, LN, TPR, VPT, CW>, kTma, TPR, \
            VPT, 0, 1, (CW + 1) * 32, VecTraits<GBN_T>::E, 1, 32768},
#define GBN_T_RMS(TPR, VPT, CW) GBN_TMA(false, TPR, VPT, CW)
#define GBN_T_LN(TPR, VPT, CW) GBN_TMA(true, TPR, VPT, CW)
#define GBN_TMAC(LN, CL, VPT, RS)                                                              \
    Variant{GBN_TMAC_VNAME(CL, VPT, RS), (const void *)&fwd_tmac<GBN_T, LN, VPT, CL, RS>, kTmaCl,  \
            kTmacNT, VPT, RS, CL, (kTmacCW + 1) * 32, VecTraits<GBN_T>::E, 1, 0},
#define GBN_C_RMS(CL, VPT, RS) GBN_TMAC(false, CL, VPT, RS)
#define GBN_C_LN(CL, VPT, RS) GBN_TMAC(true, CL, VPT, RS)
#define GBN_WIDE(LN, NT, U, MINB, PF, R)                                                       \
    Variant{GBN_WIDE_VNAME(NT, U, MINB, PF, R), (const void *)&fwd_wide<GBN_T, LN, NT, U, MINB, PF, R>, \
            kWide, NT, U, R, 1, NT, VecTraits<GBN_T>::E, MINB, 0},
#define GBN_W_RMS(NT, U, MINB, PF, R) GBN_WIDE(false, NT, U, MINB, PF, R)
#define GBN_W_LN(NT, U, MINB, PF, R) GBN_WIDE(true, NT, U, MINB, PF, R)
#define GBN_ROWS_S(LN, TPR, VPT, CTA, MINB)                                                    \
    Variant{GBN_FWD_S_VNAME(TPR, VPT, CTA, MINB), (const void *)&fwd_rows_s<GBN_T, LN, TPR, VPT, CTA, MINB>, \
            kRowsS, TPR, VPT, 1, 1, CTA, VecTraits<GBN_T>::E, MINB, 0},
#define GBN_S_RMS(TPR, VPT, CTA, MINB) GBN_ROWS_S(false, TPR, VPT, CTA, MINB)
#define GBN_S_LN(TPR, VPT, CTA, MINB) GBN_ROWS_S(true, TPR, VPT, CTA, MINB)
#define GBN_ROWS_SR(LN, TPR, VPT, CTA, MINB)                                                   \
    Variant{GBN_FWD_SR_VNAME(TPR, VPT, CTA, MINB),                                             \
            (const void *)&fwd_rows_s<GBN_T, LN, TPR, VPT, CTA, MINB, true>, kRowsS, TPR, VPT, 1, 1, CTA, \
            VecTraits<GBN_T>::E, MINB, 0, 0, 0, 1},
#define GBN_SR_RMS(TPR, VPT, CTA, MINB) GBN_ROWS_SR(false, TPR, VPT, CTA, MINB)
#define GBN_SR_LN(TPR, VPT, CTA, MINB) GBN_ROWS_SR(true, TPR, VPT, CTA, MINB)
#define GBN_FTMP(LN, TPR, VPT, NT)                                                             \
    Variant{GBN_TMP_VNAME(TPR, VPT, NT), (const void *)&fwd_tmp<GBN_T, LN, TPR, VPT, NT>, kTmaP, TPR, \
            VPT, 0, 1, NT, VecTraits<GBN_T>::E, 1, 32768},
#define GBN_FP_RMS(TPR, VPT, NT) GBN_FTMP(false, TPR, VPT, NT)
#define GBN_FP_LN(TPR, VPT, NT) GBN_FTMP(true, TPR, VPT, NT)
#define GBN_WTMA(LN, CW, U)                                                                    \
    Variant{GBN_WTMA_VNAME(CW, U), (const void *)&fwd_wtma<GBN_T, LN, CW, U>, kWtma, (CW) * 32, U, 0, 1, \
            ((CW) + 1) * 32, VecTraits<GBN_T>::E, 1, 0},
#define GBN_WT_RMS(CW, U) GBN_WTMA(false, CW, U)
#define GBN_WT_LN(CW, U) GBN_WTMA(true, CW, U)
#define GBN_FWIDER(LN, NT, K, CL, PF, MINB, F)                                                 \
    Variant{GBN_FWIDER_VNAME(NT, K, CL, PF, MINB, F),                                          \
            (const void *)&fwd_wider<GBN_T, LN, NT, K, CL, PF, MINB, F>, kWideF, NT, K, 1, CL, NT, \
            VecTraits<GBN_T>::E, MINB, 0},
#define GBN_FWR_RMS(NT, K, CL, PF, MINB, F) GBN_FWIDER(false, NT, K, CL, PF, MINB, F)
#define GBN_FWR_LN(NT, K, CL, PF, MINB, F) GBN_FWIDER(true, NT, K, CL, PF, MINB, F)
#define GBN_FWCS(LN, NT, VPT, CL)                                                              \
    Variant{GBN_WCS_VNAME(NT, VPT, CL), (const void *)&fwd_wcs<GBN_T, LN, NT, VPT, CL>, kWcs, NT, VPT, 1, \
            CL, NT, VecTraits<GBN_T>::E, 1, 0},
#define GBN_FWCS_RMS(NT, VPT, CL) GBN_FWCS(false, NT, VPT, CL)
#define GBN_FWCS_LN(NT, VPT, CL) GBN_FWCS(true, NT, VPT, CL)
static const Variant rms_variants[] = {
    GBN_FWIDER_GEOMS(GBN_FWR_RMS)
    GBN_WCS_GEOMS(GBN_FWCS_RMS)
    GBN_WTMA_FWD_GEOMS(GBN_WT_RMS)
    GBN_TMP_FWD_GEOMS(GBN_FP_RMS)
    GBN_TMA_FWD_GEOMS(GBN_T_RMS)
    GBN_TMAC_FWD_GEOMS(GBN_C_RMS)
    GBN_WIDE_FWD_GEOMS(GBN_W_RMS)
    GBN_FWD_S_GEOMS(GBN_S_RMS)
    GBN_FWD_SR_GEOMS(GBN_SR_RMS)
    GBN_FWD_GEOMS(GBN_X_RMS)
    Variant{"elem", (const void *)&fwd_elem<GBN_T, false>, kElem, kElemCTA, 0, 1, 1, kElemCTA, 1, 0, 0}};
static const Variant ln_variants[] = {
    GBN_FWIDER_GEOMS(GBN_FWR_LN)
    GBN_WCS_GEOMS(GBN_FWCS_LN)
    GBN_WTMA_FWD_GEOMS(GBN_WT_LN)
    GBN_TMP_FWD_GEOMS(GBN_FP_LN)
    GBN_TMA_FWD_GEOMS(GBN_T_LN)
    GBN_TMAC_FWD_GEOMS(GBN_C_LN)
    GBN_WIDE_FWD_GEOMS(GBN_W_LN)
    GBN_FWD_S_GEOMS(GBN_S_LN)
    GBN_FWD_SR_GEOMS(GBN_SR_LN)
    GBN_FWD_GEOMS(GBN_X_LN)
    Variant{"elem", (const void *)&fwd_elem<GBN_T, true>, kElem, kElemCTA, 0, 1, 1, kElemCTA, 1, 0, 0}};
const VariantTable GBN_CAT(kFwdRms_, GBN_SFX) = {rms_variants, (int)(sizeof(rms_variants) / sizeof(Variant))};
const VariantTable GBN_CAT(kFwdLn_, GBN_SFX) = {ln_variants, (int)(sizeof(ln_variants) / sizeof(Variant))};
#undef GBN_ROW
#undef GBN_X_RMS
#undef GBN_X_LN
#undef GBN_TMA
#undef GBN_T_RMS
#undef GBN_T_LN
#undef GBN_TMAC
#undef GBN_C_RMS
#undef GBN_C_LN
#undef GBN_WIDE
#undef GBN_W_RMS
#undef GBN_W_LN
#undef GBN_ROWS_S
#undef GBN_ROWS_SR
#undef GBN_SR_RMS
#undef GBN_SR_LN
#undef GBN_S_RMS
#undef GBN_S_LN
#undef GBN_FTMP
#undef GBN_FP_RMS
#undef GBN_FP_LN
#undef GBN_WTMA
#undef GBN_WT_RMS
#undef GBN_WT_LN
#undef GBN_FWCS
#undef GBN_FWIDER
#undef GBN_FWR_RMS
#undef GBN_FWR_LN
#undef GBN_FWCS_RMS
#undef GBN_FWCS_LN
#endif

#ifdef GBN_BWD
#define GBN_ROW(LN, TPR, VPT, R, CL, CTA)                                                     \
    Variant{GBN_VNAME(TPR, VPT, R, CL, CTA), (const void *)&bwd_rows<GBN_T, LN, TPR, VPT, R, CL, CTA>, \
            kRows, TPR, VPT, R, CL, CTA, VecTraits<GBN_T>::E, 0, 0},
#define GBN_X_RMS(TPR, VPT, R, CL, CTA) GBN_ROW(false, TPR, VPT, R, CL, CTA)
#define GBN_X_LN(TPR, VPT, R, CL, CTA) GBN_ROW(true, TPR, VPT, R, CL, CTA)
#define GBN_TMA(LN, TPR, VPT, CW)                                                              \
    Variant{GBN_TMA_VNAME(TPR, VPT, CW), (const void *)&bwd_tma<GBN_T, LN, TPR, VPT, CW>, kTma, TPR, \
            VPT, 0, 1, (CW + 1) * 32, VecTraits<GBN_T>::E, 1, 32768},
#define GBN_T_RMS(TPR, VPT, CW) GBN_TMA(false, TPR, VPT, CW)
#define GBN_T_LN(TPR, VPT, CW) GBN_TMA(true, TPR, VPT, CW)
#define GBN_TMAC(LN, CL, VPT, RS)                                                              \
    Variant{GBN_TMAC_VNAME(CL, VPT, RS), (const void *)&bwd_tmac<GBN_T, LN, VPT, CL, RS>, kTmaCl,  \
            kTmacNT, VPT, RS, CL, (kTmacCW + 1) * 32, VecTraits<GBN_T>::E, 1, 0},
#define GBN_C_RMS(CL, VPT, RS) GBN_TMAC(false, CL, VPT, RS)
#define GBN_C_LN(CL, VPT, RS) GBN_TMAC(true, CL, VPT, RS)
#define GBN_BWIDE(LN, NT, U, CL, PF, F, MINB)                                                  \
    Variant{GBN_BWIDE_VNAME(NT, U, CL, PF, F, MINB),                                           \
            (const void *)&bwd_wide<GBN_T, LN, NT, U, CL, PF, F, MINB>, kWide, NT, U, 1, CL, NT,   \
            VecTraits<GBN_T>::E, MINB, 0},
#define GBN_W_RMS(NT, U, CL, PF, F, MINB) GBN_BWIDE(false, NT, U, CL, PF, F, MINB)
#define GBN_W_LN(NT, U, CL, PF, F, MINB) GBN_BWIDE(true, NT, U, CL, PF, F, MINB)
#define GBN_TMP(LN, TPR, VPT, NT)                                                              \
    Variant{GBN_TMP_VNAME(TPR, VPT, NT), (const void *)&bwd_tmp<GBN_T, LN, TPR, VPT, NT>, kTmaP, TPR, \
            VPT, 0, 1, NT, VecTraits<GBN_T>::E, 1, 32768},
#define GBN_P_RMS(TPR, VPT, NT) GBN_TMP(false, TPR, VPT, NT)
#define GBN_P_LN(TPR, VPT, NT) GBN_TMP(true, TPR, VPT, NT)
// single-kernel variants: the same kernels summing their partial rows themselves
#define GBN_SKTMA(LN, TPR, VPT, CW)                                                            \
    Variant{"sk" GBN_TMA_VNAME(TPR, VPT, CW), (const void *)&bwd_tma<GBN_T, LN, TPR, VPT, CW, true>, kTma, \
            TPR, VPT, 0, 1, (CW + 1) * 32, VecTraits<GBN_T>::E, 1, 32768, 1},
#define GBN_SKT_RMS(TPR, VPT, CW) GBN_SKTMA(false, TPR, VPT, CW)
#define GBN_SKT_LN(TPR, VPT, CW) GBN_SKTMA(true, TPR, VPT, CW)
#define GBN_SKTMP(LN, TPR, VPT, NT)                                                            \
    Variant{"sk" GBN_TMP_VNAME(TPR, VPT, NT), (const void *)&bwd_tmp<GBN_T, LN, TPR, VPT, NT, true>, kTmaP, \
            TPR, VPT, 0, 1, NT, VecTraits<GBN_T>::E, 1, 32768, 1},
#define GBN_SKP_RMS(TPR, VPT, NT) GBN_SKTMP(false, TPR, VPT, NT)
#define GBN_SKP_LN(TPR, VPT, NT) GBN_SKTMP(true, TPR, VPT, NT)
#define GBN_BWTMA(LN, CL, K)                                                                   \
    Variant{GBN_BWTMA_VNAME(CL, K), (const void *)&bwd_wtma<GBN_T, LN, CL, K>, kWtmaC, 512, K, 0, CL, 544, \
            VecTraits<GBN_T>::E, 1, 0},
#define GBN_BWT_RMS(CL, K) GBN_BWTMA(false, CL, K)
#define GBN_BWT_LN(CL, K) GBN_BWTMA(true, CL, K)
#define GBN_WIDER(LN, NT, K, CL, PF, MINB, F)                                                  \
    Variant{GBN_WIDER_VNAME(NT, K, CL, PF, MINB, F), (const void *)&bwd_wider<GBN_T, LN, NT, K, CL, PF, MINB, F>, \
            kWideR, NT, K, 1, CL, NT, VecTraits<GBN_T>::E, MINB, 0},
#define GBN_WIDER_DB(NT, K, CL, PF, MINB, F)                                                   \
    Variant{GBN_WIDER_VNAME(NT, K, CL, PF, MINB, F) "d",                                       \
            (const void *)&bwd_wider<GBN_T, true, NT, K, CL, PF, MINB, F, 1>, kWideR, NT, K, 1, CL, NT, \
            VecTraits<GBN_T>::E, MINB, 0, 0, 1},
#define GBN_WIDER_DG(NT, K, CL, PF, MINB, F)                                                   \
    Variant{GBN_WIDER_VNAME(NT, K, CL, PF, MINB, F) "g",                                       \
            (const void *)&bwd_wider<GBN_T, true, NT, K, CL, PF, MINB, F, 2>, kWideR, NT, K, 1, CL, NT, \
            VecTraits<GBN_T>::E, MINB, 0, 0, 2},
#define GBN_WR_RMS(NT, K, CL, PF, MINB, F) GBN_WIDER(false, NT, K, CL, PF, MINB, F)
#define GBN_WR_LN(NT, K, CL, PF, MINB, F) GBN_WIDER(true, NT, K, CL, PF, MINB, F)
#define GBN_BWCS(LN, NT, VPT, CL)                                                              \
    Variant{GBN_WCS_VNAME(NT, VPT, CL), (const void *)&bwd_wcs<GBN_T, LN, NT, VPT, CL>, kWcs, NT, VPT, 1, \
            CL, NT, VecTraits<GBN_T>::E, 1, 0},
#define GBN_BWCS_RMS(NT, VPT, CL) GBN_BWCS(false, NT, VPT, CL)
#define GBN_BWCS_LN(NT, VPT, CL) GBN_BWCS(true, NT, VPT, CL)
static const Variant rms_variants[] = {
    GBN_WCS_GEOMS(GBN_BWCS_RMS)
    GBN_WIDER_BWD_GEOMS(GBN_WR_RMS)
    GBN_BWTMA_BWD_GEOMS(GBN_BWT_RMS)
    GBN_TMA_BWD_GEOMS(GBN_T_RMS)
    GBN_TMP_BWD_GEOMS(GBN_P_RMS)
    GBN_SK_TMA_BWD_GEOMS(GBN_SKT_RMS)
    GBN_SK_TMP_BWD_GEOMS(GBN_SKP_RMS)
    GBN_TMAC_BWD_GEOMS(GBN_C_RMS)
    GBN_WIDE_BWD_GEOMS(GBN_W_RMS)
    GBN_BWD_GEOMS(GBN_X_RMS)
    Variant{"elem", (const void *)&bwd_elem<GBN_T, false>, kElem, kElemCTA, 0, 1, 1, kElemCTA, 1, 0, 0}};
static const Variant ln_variants[] = {
    GBN_WCS_GEOMS(GBN_BWCS_LN)
    GBN_WIDER_DB_GEOMS(GBN_WIDER_DB)
    GBN_WIDER_DG_GEOMS(GBN_WIDER_DG)
    GBN_WIDER_BWD_GEOMS(GBN_WR_LN)
    GBN_BWTMA_BWD_GEOMS(GBN_BWT_LN)
    GBN_TMA_BWD_GEOMS(GBN_T_LN)
    GBN_TMP_BWD_GEOMS(GBN_P_LN)
    GBN_SK_TMA_BWD_GEOMS(GBN_SKT_LN)
    GBN_SK_TMP_BWD_GEOMS(GBN_SKP_LN)
    GBN_TMAC_BWD_GEOMS(GBN_C_LN)
    GBN_WIDE_BWD_GEOMS(GBN_W_LN)
    GBN_BWD_GEOMS(GBN_X_LN)
    Variant{"elem", (const void *)&bwd_elem<GBN_T, true>, kElem, kElemCTA, 0, 1, 1, kElemCTA, 1, 0, 0}};
const VariantTable GBN_CAT(kBwdRms_, GBN_SFX) = {rms_variants, (int)(sizeof(rms_variants) / sizeof(Variant))};
const VariantTable GBN_CAT(kBwdLn_, GBN_SFX) = {ln_variants, (int)(sizeof(ln_variants) / sizeof(Variant))};
#undef GBN_BWIDE
#undef GBN_W_RMS
#undef GBN_W_LN
#undef GBN_TMP
#undef GBN_P_RMS
#undef GBN_P_LN
#undef GBN_BWTMA
#undef GBN_BWT_RMS
#undef GBN_BWT_LN
#undef GBN_WIDER
#undef GBN_WR_RMS
#undef GBN_WR_LN
#undef GBN_BWCS
#undef GBN_WIDER_DB
#undef GBN_WIDER_DG
#undef GBN_BWCS_RMS
#undef GBN_BWCS_LN
#undef GBN_SKTMA
#undef GBN_SKT_RMS
#undef GBN_SKT_LN
#undef GBN_SKTMP
#undef GBN_SKP_RMS
#undef GBN_SKP_LN
#endif

}  // namespace gbn
