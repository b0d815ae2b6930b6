// RoPE angle tables (KVQuant "Pre-RoPE Key Quantization": the rotation is
// applied to keys after dequantization, so decode needs cos/sin for every
// cached position). Angles are formed in binary64 so that positions near 2^24
// keep full accuracy; the tables store binary32 cos/sin.
#include "kvq_common.cuh"

namespace kvq {
namespace {

__global__ void rope_init_kernel(Dims d, double theta, float2* __restrict__ tab) {
  const int half = d.D / 2;
  const size_t n = rope_entries(d);
  const size_t lo = rope_lo_off(d), hi = rope_hi_off(d);
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    int i;
    double pos;
    if (e < lo) {                       // fine: [i][j], angle j * w_i
      i = (int)(e / d.Bk);
      pos = (double)(e % d.Bk);
    } else if (e < hi) {                // coarse: [m][i], angle Bk * m * w_i
      const size_t r = e - lo;
      i = (int)(r % half);
      pos = (double)d.Bk * (double)(r / half);
    } else {                            // high: [m][i], angle 256 * Bk * m * w_i
      const size_t r = e - hi;
      i = (int)(r % half);
      pos = (double)kRopeLo * d.Bk * (double)(r / half);
    }
    const double w = pow(theta, -2.0 * i / d.D);
    double s, c;
    sincos(pos * w, &s, &c);
    tab[e] = make_float2((float)c, (float)s);
  }
}

}  // namespace

cudaError_t launch_rope_init(const Dims& d, double theta, float2* tab, cudaStream_t st) {
  const size_t n = rope_entries(d);
  const int threads = 256;
  const int blocks = (int)((n + threads - 1) / threads < 4096 ? (n + threads - 1) / threads : 4096);
  rope_init_kernel<<<blocks, threads, 0, st>>>(d, theta, tab);
  return cudaGetLastError();
}

}  // namespace kvq
