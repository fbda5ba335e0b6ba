// General-form kernel instantiations: forward.
#define GBN_EX_DIR 0
#include "inst_ex_body.cuh"
