// Decode dispatch: choose the T split, launch the partial kernel, then merge the
// splits (log-sum-exp in base 2) into the fp16 output.
#include "kvq_decode.cuh"

namespace kvq {
namespace {

template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const float* __restrict__ ws,
                                                           __half* __restrict__ out, int n_split,
                                                           int S) {
  const int bhq = blockIdx.x;
  const float* p = ws + (size_t)bhq * S * (D + 2);
  const int c = threadIdx.x;
  float M = -INFINITY;
  for (int s = 0; s < n_split; ++s) M = fmaxf(M, p[(size_t)s * (D + 2) + D]);
  float L = 0.0f, acc = 0.0f;
  for (int s = 0; s < n_split; ++s) {
    const float* ps = p + (size_t)s * (D + 2);
    const float m = ps[D];
    if (m == -INFINITY) continue;          // split without tokens
    const float w = exp2f(m - M);
    L = fmaf(w, ps[D + 1], L);
    acc = fmaf(w, ps[c], acc);
  }
  out[(size_t)bhq * D + c] = __float2half_rn(acc / L);
}

using LaunchFn = cudaError_t (*)(const DecodeArgs&, cudaStream_t);
using OccFn = int (*)();

template <int BITS, int D>
void pick_g(int G, LaunchFn* f, OccFn* o) {
  switch (G) {
    case 1: *f = launch_partial<BITS, D, 1>; *o = partial_occupancy<BITS, D, 1>; break;
    case 2: *f = launch_partial<BITS, D, 2>; *o = partial_occupancy<BITS, D, 2>; break;
    case 4: *f = launch_partial<BITS, D, 4>; *o = partial_occupancy<BITS, D, 4>; break;
    default: *f = launch_partial<BITS, D, 8>; *o = partial_occupancy<BITS, D, 8>; break;
  }
}

template <int BITS>
void pick_d(int D, int G, LaunchFn* f, OccFn* o) {
  if (D == 64) pick_g<BITS, 64>(G, f, o);
  else pick_g<BITS, 128>(G, f, o);
}

// Occupancy (CTAs per SM) of each kernel variant, per device, computed once.
int cached_occupancy(int dev, int bits, int D, int G, OccFn fn) {
  static int cache[16][3][2][4];
  const int gi = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
  int& slot = cache[dev & 15][bits - 2][D == 128][gi];
  if (slot == 0) slot = fn();
  return slot;
}

// Splits per stream: minimize (waves of CTAs) x (key blocks in the longest split),
// preferring fewer splits on ties (less combine work).
int choose_splits(int streams, int units, int slots, int max_split) {
  int best = 1;
  double best_cost = 1e300;
  const int hi = units < max_split ? units : max_split;
  for (int n = 1; n <= hi; ++n) {
    const long long ctas = (long long)streams * n;
    const long long waves = (ctas + slots - 1) / slots;
    const int per = (units + n - 1) / n;
    const double cost = (double)waves * (per + 0.25);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = n;
    }
  }
  return best;
}

}  // namespace

cudaError_t launch_decode(const Dims& d, const kvq_cache& c, const __half* q, int H_q, int q_pos,
                          const float2* rope, float sm_scale, __half* out, float* ws,
                          cudaStream_t st) {
  DecodeArgs a;
  a.d = d;
  a.k_codes = static_cast<const uint8_t*>(c.k_codes);
  a.k_meta = static_cast<const uint32_t*>(c.k_meta);
  a.k_tail = static_cast<const __half*>(c.k_tail);
  a.k_outl = static_cast<const uint32_t*>(c.k_outl);
  a.v_codes = static_cast<const uint8_t*>(c.v_codes);
  a.v_meta = static_cast<const uint32_t*>(c.v_meta);
  a.v_outl = static_cast<const uint32_t*>(c.v_outl);
  a.q = q;
  a.rope = rope;
  a.ws = ws;
  a.T = c.T_cur;
  a.n_full = c.T_cur / d.Bk;
  a.tail_len = c.T_cur % d.Bk;
  a.H_q = H_q;
  a.q_pos = q_pos;
  a.S = max_splits(d);
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  const int G = H_q / d.H_kv;

  LaunchFn fn = nullptr;
  OccFn occ_fn = nullptr;
  switch (d.bits) {
    case 2: pick_d<2>(d.D, G, &fn, &occ_fn); break;
    case 3: pick_d<3>(d.D, G, &fn, &occ_fn); break;
    default: pick_d<4>(d.D, G, &fn, &occ_fn); break;
  }
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int occ = cached_occupancy(dev, d.bits, d.D, G, occ_fn);
  const int units = a.n_full + (a.tail_len > 0 ? 1 : 0);
  a.n_split = choose_splits(d.B * d.H_kv, units, sms * occ, a.S);

  e = fn(a, st);
  if (e != cudaSuccess) return e;
  if (d.D == 64)
    decode_combine_kernel<64><<<d.B * H_q, 64, 0, st>>>(ws, out, a.n_split, a.S);
  else
    decode_combine_kernel<128><<<d.B * H_q, 128, 0, st>>>(ws, out, a.n_split, a.S);
  return cudaGetLastError();
}

}  // namespace kvq
