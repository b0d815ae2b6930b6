// Decode partial kernels for 3-bit codes.
#include "kvq_decode_inst.cuh"

namespace kvq {
KVQ_INSTANTIATE_DECODE(3)
}  // namespace kvq
