// Decode partial kernels for 8-bit codes (head_dim 64 and 128; the
// tensor-core kernel's fragment geometry covers 2-4 bit codes).
#include "kvq_decode_inst.cuh"

namespace kvq {
KVQ_INSTANTIATE_DECODE_D(8, 64)
KVQ_INSTANTIATE_DECODE_D(8, 128)
}  // namespace kvq
