// Level tables of the non-uniform codes (kvq_levels.cu) and their launchers.
#pragma once

#include "kvq_common.cuh"

namespace kvq {

// A table in the kernels' parameters: the 2^b levels and the binary32
// midpoints fp32(0.5 (l_k + l_k+1)) between neighbours.
struct LevelTable {
  float lv[256];
  float mid[255];
  int L;  // 2^bits - 1
};

cudaError_t launch_decode_levels(const Dims& d, const kvq_cache& c, const __half* q, int H_q, int q_pos,
                                 const float2* rope, float sm_scale, __half* out, float* ws,
                                 const LevelTable& t, cudaStream_t st);

}  // namespace kvq
