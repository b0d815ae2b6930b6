// Decode partial kernels for 2-bit codes.
#include "kvq_decode_inst.cuh"

namespace kvq {
KVQ_INSTANTIATE_DECODE(2)
}  // namespace kvq
