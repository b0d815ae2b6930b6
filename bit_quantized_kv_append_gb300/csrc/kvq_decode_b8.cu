// Decode partial kernels for 8-bit codes (head_dim 64).
#include "kvq_decode_inst.cuh"

namespace kvq {
KVQ_INSTANTIATE_DECODE(8)
}  // namespace kvq
