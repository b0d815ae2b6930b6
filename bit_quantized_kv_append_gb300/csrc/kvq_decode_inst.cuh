// Launch and occupancy helpers of the decode partial kernel; included by one
// translation unit per code width so the instantiations compile in parallel.
#pragma once

#include "kvq_decode.cuh"

namespace kvq {

template <int BITS, int D, int G>
cudaError_t launch_partial(const DecodeArgs& a, cudaStream_t st) {
  const dim3 grid(a.n_split, a.d.B * a.d.H_kv);
  decode_partial_kernel<BITS, D, G><<<grid, kDecThreads, 0, st>>>(a);
  return cudaGetLastError();
}

template <int BITS, int D, int G>
int partial_occupancy() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_partial_kernel<BITS, D, G>,
                                                    kDecThreads, 0) != cudaSuccess)
    n = 1;
  return n < 1 ? 1 : n;
}

#define KVQ_INSTANTIATE_DECODE_D(BITS, D)                                          \
  template cudaError_t launch_partial<BITS, D, 1>(const DecodeArgs&, cudaStream_t);   \
  template cudaError_t launch_partial<BITS, D, 2>(const DecodeArgs&, cudaStream_t);   \
  template cudaError_t launch_partial<BITS, D, 4>(const DecodeArgs&, cudaStream_t);   \
  template cudaError_t launch_partial<BITS, D, 8>(const DecodeArgs&, cudaStream_t);   \
  template int partial_occupancy<BITS, D, 1>();                                     \
  template int partial_occupancy<BITS, D, 2>();                                     \
  template int partial_occupancy<BITS, D, 4>();                                     \
  template int partial_occupancy<BITS, D, 8>();
#define KVQ_INSTANTIATE_DECODE(BITS) KVQ_INSTANTIATE_DECODE_D(BITS, 64)

}  // namespace kvq
