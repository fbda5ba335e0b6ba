// General-form kernel instantiations: backward.
#define GBN_EX_DIR 1
#include "inst_ex_body.cuh"
