// Kernel instantiations: fwdward, element type __nv_bfloat16.
#define GBN_T __nv_bfloat16
#define GBN_SFX bf16
#define GBN_FWD 1
#include "inst_body.cuh"
