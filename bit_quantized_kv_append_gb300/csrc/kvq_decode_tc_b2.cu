// Tensor-core decode kernels (head_dim 128) for 2-bit codes, caches without outliers.
#include "kvq_decode_tc_inst.cuh"

namespace kvq {
KVQ_INSTANTIATE_TC(2, false, false)
}  // namespace kvq
