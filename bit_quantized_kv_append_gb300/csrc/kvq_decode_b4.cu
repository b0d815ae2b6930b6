// Decode partial kernels for 4-bit codes.
#include "kvq_decode_inst.cuh"

namespace kvq {
KVQ_INSTANTIATE_DECODE(4)
}  // namespace kvq
