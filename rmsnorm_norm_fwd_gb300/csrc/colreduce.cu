// Column-reduce kernel instantiations (stage two of the dgamma/dbeta reduction).
#include "norm_kernels.cuh"

namespace gbn {
const void *const kColReduceVec4 = (const void *)&colreduce<4>;
const void *const kColReduceScalar = (const void *)&colreduce<1>;
}  // namespace gbn
