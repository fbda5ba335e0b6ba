// Kernel instantiations: bwdward, element type float.
#define GBN_T float
#define GBN_SFX f32
#define GBN_BWD 1
#include "inst_body.cuh"
