// Kernel instantiations: bwdward, element type __half.
#define GBN_T __half
#define GBN_SFX f16
#define GBN_BWD 1
#include "inst_body.cuh"
