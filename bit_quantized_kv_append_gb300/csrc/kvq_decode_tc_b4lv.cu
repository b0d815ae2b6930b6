// Tensor-core decode kernels (head_dim 128) for 4-bit codes against a level table.
#include "kvq_decode_tc_inst.cuh"

namespace kvq {
KVQ_INSTANTIATE_TC_LV(4, false)
KVQ_INSTANTIATE_TC_LV(4, true)
}  // namespace kvq
