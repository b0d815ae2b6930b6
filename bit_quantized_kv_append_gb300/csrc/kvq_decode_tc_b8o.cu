// Tensor-core decode kernels (head_dim 128) for 8-bit codes, caches with outliers.
#include "kvq_decode_tc_inst.cuh"

namespace kvq {
KVQ_INSTANTIATE_TC(8, true, false)
}  // namespace kvq
