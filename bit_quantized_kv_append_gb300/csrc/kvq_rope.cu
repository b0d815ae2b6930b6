// RoPE angle tables (KVQuant "Pre-RoPE Key Quantization": the rotation is
// applied to keys after dequantization, so decode needs cos/sin for every
// cached position). Angles are formed in binary64 so that positions near 2^24
// keep full accuracy; the tables store binary32 cos/sin.
#include "kvq_tc_geom.cuh"

namespace kvq {
namespace {

__global__ void rope_init_kernel(Dims d, double theta, float2* __restrict__ tab) {
  const int half = d.D / 2;
  const size_t n = rope_hi_off(d) + (size_t)d.rope_n_hi * half;
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

// In-block rotations R(j), j < 64, of the tensor-core kernel's fragments
// (kvq_tc_geom.cuh): one uint4 of fp16 {cos, cos, sin, sin} per
// (warp, n-tile, k-step, lane), angles in binary64.
template <int BITS>
__global__ void rope_frag_kernel(double theta, uint4* __restrict__ frag) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= tc::kRotFragQuads) return;
  const int lane = e & 31, kq = (e >> 5) & 3, nt = (e >> 7) & 1, w = e >> 8;
  const int g = lane >> 2, r = lane & 3;
  const int j = 16 * w + 8 * nt + tc::tperm(g);
  uint16_t c[4], s[4];
  for (int k = 0; k < 4; ++k) {
    const int i = tc::kchan<BITS>(r, kq, k);
    double sn, cs;
    sincos((double)j * pow(theta, -2.0 * i / tc::kD), &sn, &cs);
    c[k] = __half_as_ushort(__double2half(cs));
    s[k] = __half_as_ushort(__double2half(sn));
  }
  frag[e] = make_uint4(c[0] | ((uint32_t)c[1] << 16), c[2] | ((uint32_t)c[3] << 16),
                       s[0] | ((uint32_t)s[1] << 16), s[2] | ((uint32_t)s[3] << 16));
}

}  // namespace

cudaError_t launch_rope_init(const Dims& d, double theta, float2* tab, cudaStream_t st) {
  const size_t n = rope_hi_off(d) + (size_t)d.rope_n_hi * (d.D / 2);
  const int threads = 256;
  const int blocks = (int)((n + threads - 1) / threads < 4096 ? (n + threads - 1) / threads : 4096);
  rope_init_kernel<<<blocks, threads, 0, st>>>(d, theta, tab);
  if (d.D == tc::kD) {
    uint4* frag = reinterpret_cast<uint4*>(tab + rope_frag_off(d));
    const int fb = tc::kRotFragQuads / threads;
    if (d.bits == 8) rope_frag_kernel<8><<<fb, threads, 0, st>>>(theta, frag);
    else if (d.bits == 4) rope_frag_kernel<4><<<fb, threads, 0, st>>>(theta, frag);
    else if (d.bits == 3) rope_frag_kernel<3><<<fb, threads, 0, st>>>(theta, frag);
    else rope_frag_kernel<2><<<fb, threads, 0, st>>>(theta, frag);
  }
  return cudaGetLastError();
}

}  // namespace kvq
