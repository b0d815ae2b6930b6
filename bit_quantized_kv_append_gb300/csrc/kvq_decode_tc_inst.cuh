// Launch and occupancy helpers of the tensor-core decode kernel; included by
// one translation unit per code width so the instantiations build in parallel.
#pragma once

#include <atomic>

#include "kvq_decode_tc.cuh"

namespace kvq {

template <int BITS, int G, int SL, bool OUTL, bool PAGED, int MODE>
cudaError_t launch_tc(const DecodeArgs& a, const tc::StageLayout& L, const CUtensorMap& tk,
                      const CUtensorMap& tv, size_t smem, cudaStream_t st) {
  auto kern = tc::decode_tc_kernel<BITS, G, SL, OUTL, PAGED, MODE>;
  // largest dynamic shared memory requested so far, per device (a function attribute per device)
  static std::atomic<size_t> smem_set[kMaxDevices];
  int dev = 0;
  if (current_device(&dev) != KVQ_OK) return cudaErrorInvalidDevice;
  if (smem_set[dev].load(std::memory_order_acquire) < smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    size_t cur = smem_set[dev].load(std::memory_order_relaxed);
    while (cur < smem && !smem_set[dev].compare_exchange_weak(cur, smem, std::memory_order_acq_rel)) {
    }
  }
  const dim3 grid(a.n_split, a.d.B * a.d.H_kv);
  kern<<<grid, tc::kThreads, smem, st>>>(a, L, tk, tv);
  return cudaGetLastError();
}

template <int BITS, int G, int SL, bool OUTL, bool PAGED, int MODE>
int tc_occupancy(size_t smem) {
  auto kern = tc::decode_tc_kernel<BITS, G, SL, OUTL, PAGED, MODE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, tc::kThreads, smem) != cudaSuccess) n = 1;
  return n < 1 ? 1 : n;
}

#define KVQ_TC_ONE_P(BITS, G, SL, OUTL, PAGED, MODE)                                                         \
  template cudaError_t launch_tc<BITS, G, SL, OUTL, PAGED, MODE>(const DecodeArgs&, const tc::StageLayout&,     \
                                                                 const CUtensorMap&, const CUtensorMap&, size_t, \
                                                                 cudaStream_t);                                  \
  template int tc_occupancy<BITS, G, SL, OUTL, PAGED, MODE>(size_t);
// modes 0 (fp16-operand scores) and 1 (precise scores)
#define KVQ_TC_ONE(BITS, G, SL, OUTL, PAGED) \
  KVQ_TC_ONE_P(BITS, G, SL, OUTL, PAGED, 0) \
  KVQ_TC_ONE_P(BITS, G, SL, OUTL, PAGED, 1)
// mode 2 (level tables): contiguous caches
#define KVQ_INSTANTIATE_TC_LV(BITS, OUTL)      \
  KVQ_TC_ONE_P(BITS, 1, 1, OUTL, false, 2)     \
  KVQ_TC_ONE_P(BITS, 2, 1, OUTL, false, 2)     \
  KVQ_TC_ONE_P(BITS, 4, 1, OUTL, false, 2)     \
  KVQ_TC_ONE_P(BITS, 8, 1, OUTL, false, 2)     \
  KVQ_TC_ONE_P(BITS, 1, 2, OUTL, false, 2)     \
  KVQ_TC_ONE_P(BITS, 2, 2, OUTL, false, 2)     \
  KVQ_TC_ONE_P(BITS, 4, 2, OUTL, false, 2)     \
  KVQ_TC_ONE_P(BITS, 8, 2, OUTL, false, 2)
#define KVQ_INSTANTIATE_TC(BITS, OUTL, PAGED) \
  KVQ_TC_ONE(BITS, 1, 1, OUTL, PAGED)         \
  KVQ_TC_ONE(BITS, 2, 1, OUTL, PAGED)         \
  KVQ_TC_ONE(BITS, 4, 1, OUTL, PAGED)         \
  KVQ_TC_ONE(BITS, 8, 1, OUTL, PAGED)         \
  KVQ_TC_ONE(BITS, 1, 2, OUTL, PAGED)         \
  KVQ_TC_ONE(BITS, 2, 2, OUTL, PAGED)         \
  KVQ_TC_ONE(BITS, 4, 2, OUTL, PAGED)         \
  KVQ_TC_ONE(BITS, 8, 2, OUTL, PAGED)

}  // namespace kvq
