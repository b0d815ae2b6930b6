// Decode dispatch: choose the T split, launch the partial kernel (tensor-core
// kernel for head_dim 128, CUDA-core kernel for head_dim 64), then merge the
// splits (log-sum-exp in base 2) into the fp16 output.
#include <cuda.h>

#include <mutex>

#include "kvq_decode_tc.cuh"

namespace kvq {
namespace {

template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const float* __restrict__ ws,
                                                           __half* __restrict__ out, int n_split,
                                                           int S) {
  __shared__ float s_w[kMaxSplits];
  __shared__ float s_red[D / 32];
  const int bhq = blockIdx.x;
  const float* p = ws + (size_t)bhq * S * (D + 2);
  const int c = threadIdx.x;
  // the largest split maximum, the splits read in parallel
  float M = -INFINITY;
  for (int s = c; s < n_split; s += D) M = fmaxf(M, p[(size_t)s * (D + 2) + D]);
  M = warp_max(M);
  if ((c & 31) == 0) s_red[c >> 5] = M;
  __syncthreads();
  M = s_red[0];
#pragma unroll
  for (int k = 1; k < D / 32; ++k) M = fmaxf(M, s_red[k]);
  // split weights 2^(m_s - M): 0 for a split without tokens; the NaN partials
  // of a split whose waits expired give NaN, which stays NaN below
  for (int s = c; s < n_split; s += D) {
    const float m = p[(size_t)s * (D + 2) + D];
    s_w[s] = (m == -INFINITY) ? 0.0f : exp2f(m - M);
  }
  __syncthreads();
  float L = 0.0f, acc = 0.0f;
#pragma unroll 8
  for (int s = 0; s < n_split; ++s) {
    const float w = s_w[s];
    const float* ps = p + (size_t)s * (D + 2);
    L = fmaf(w, ps[D + 1], L);
    acc = fmaf(w, ps[c], acc);
  }
  // a sequence without tokens: 0
  out[(size_t)bhq * D + c] = __float2half_rn(L == 0.0f ? 0.0f : acc / L);
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

// Occupancy (CTAs per SM) of each kernel variant, per device, computed once.
int cached_occupancy(int dev, int bits, int D, int G, OccFn fn) {
  static std::mutex mu;
  static int cache[kMaxDevices][4][2][4];
  const int gi = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
  std::lock_guard<std::mutex> lock(mu);
  int& slot = cache[dev][bits == 8 ? 3 : bits - 2][D == 128][gi];
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

// Paged, ragged batches: every sequence gets the same number of splits, so a
// CTA's work follows its sequence's length. When a uniform batch of the
// longest length would fill a single wave, twice its splits leave the
// hardware scheduler shorter CTAs to even the load out across the SMs.
int paged_splits(const Dims& d, int units_max, int slots, int max_split) {
  int n = choose_splits(d.B * d.H_kv, units_max, slots, max_split);
  if ((long long)n * d.B * d.H_kv <= slots) n *= 2;
  if (n > units_max) n = units_max;
  if (n > max_split) n = max_split;
  return n < 1 ? 1 : n;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once (thread-safe static init).
EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return nullptr;
  }();
  return fn;
}

// 3-D map over a packed code buffer: [stream][T_max rows][row byte]
// (contiguous cache) or [physical block x H_kv][Bk rows][row byte] (paged
// pools, `pool_units` > 0); box = one key block. INT8 rows (128 B) get the
// 128 B swizzle, INT4 rows (64 B) 64 B, INT2 rows (32 B) 32 B.
bool encode_codes(CUtensorMap* m, const void* base, const Dims& d, size_t pool_units) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t rows = pool_units ? (cuuint64_t)d.Bk : (cuuint64_t)d.T_max;
  const cuuint64_t dims[3] = {(cuuint64_t)d.cb, rows, pool_units ? (cuuint64_t)pool_units : (cuuint64_t)d.B * d.H_kv};
  const cuuint64_t strides[2] = {(cuuint64_t)d.cb, rows * d.cb};
  const cuuint32_t box[3] = {(cuuint32_t)d.cb, (cuuint32_t)d.Bk, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = d.bits == 8   ? CU_TENSOR_MAP_SWIZZLE_128B
                                : d.bits == 4 ? CU_TENSOR_MAP_SWIZZLE_64B
                                : d.bits == 2 ? CU_TENSOR_MAP_SWIZZLE_32B
                                              : CU_TENSOR_MAP_SWIZZLE_NONE;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

tc::StageLayout stage_layout(const Dims& d) {
  tc::StageLayout L;
  L.code_bytes = (uint32_t)(d.Bk * d.cb);
  L.km_bytes = (uint32_t)(d.D * 4);
  L.vm_bytes = (uint32_t)(d.Bk * d.ng * 4);
  L.outl_bytes = (uint32_t)(d.Bk * d.n_out * 4);
  L.kc = 0;
  L.vc = align_up(L.code_bytes, 1024);
  L.km = align_up(L.vc + L.code_bytes, 16);
  L.vm = L.km + L.km_bytes;
  L.ko = align_up(L.vm + L.vm_bytes, 16);
  L.vo = L.ko + L.outl_bytes;
  L.stage_bytes = align_up(L.vo + L.outl_bytes, 1024);
  L.tx_bytes = 2 * L.code_bytes + L.km_bytes + L.vm_bytes + 2 * L.outl_bytes;
  return L;
}

using TcLaunchFn = cudaError_t (*)(const DecodeArgs&, const tc::StageLayout&, const CUtensorMap&,
                                   const CUtensorMap&, size_t, cudaStream_t);
using TcOccFn = int (*)(size_t);

template <int BITS, int SL, bool OUTL, bool PAGED, int MODE>
void pick_tc_g(int G, TcLaunchFn* f, TcOccFn* o) {
  switch (G) {
    case 1: *f = launch_tc<BITS, 1, SL, OUTL, PAGED, MODE>; *o = tc_occupancy<BITS, 1, SL, OUTL, PAGED, MODE>; break;
    case 2: *f = launch_tc<BITS, 2, SL, OUTL, PAGED, MODE>; *o = tc_occupancy<BITS, 2, SL, OUTL, PAGED, MODE>; break;
    case 4: *f = launch_tc<BITS, 4, SL, OUTL, PAGED, MODE>; *o = tc_occupancy<BITS, 4, SL, OUTL, PAGED, MODE>; break;
    default: *f = launch_tc<BITS, 8, SL, OUTL, PAGED, MODE>; *o = tc_occupancy<BITS, 8, SL, OUTL, PAGED, MODE>; break;
  }
}

template <int BITS, bool PAGED, int MODE>
void pick_tc_p(int Bk, int G, bool outl, TcLaunchFn* f, TcOccFn* o) {
  if (Bk == 64)
    outl ? pick_tc_g<BITS, 1, true, PAGED, MODE>(G, f, o) : pick_tc_g<BITS, 1, false, PAGED, MODE>(G, f, o);
  else
    outl ? pick_tc_g<BITS, 2, true, PAGED, MODE>(G, f, o) : pick_tc_g<BITS, 2, false, PAGED, MODE>(G, f, o);
}
// mode 0: fp16-operand scores, 1: precise scores, 2: level tables (contiguous caches only)
template <int BITS>
void pick_tc(int Bk, int G, bool outl, bool paged, int mode, TcLaunchFn* f, TcOccFn* o) {
  if (mode == 2) {
    pick_tc_p<BITS, false, 2>(Bk, G, outl, f, o);
    return;
  }
  if (mode == 1) paged ? pick_tc_p<BITS, true, 1>(Bk, G, outl, f, o) : pick_tc_p<BITS, false, 1>(Bk, G, outl, f, o);
  else paged ? pick_tc_p<BITS, true, 0>(Bk, G, outl, f, o) : pick_tc_p<BITS, false, 0>(Bk, G, outl, f, o);
}

int cached_tc_occupancy(int dev, int bits, int Bk, int G, bool outl, bool paged, int mode, size_t smem,
                        TcOccFn fn) {
  struct Slot { size_t smem; int occ; };
  static std::mutex mu;
  static Slot cache[kMaxDevices][4][2][4][2][2][3];
  const int gi = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
  std::lock_guard<std::mutex> lock(mu);
  Slot& s = cache[dev][bits == 8 ? 3 : bits - 2][Bk == 128][gi][outl ? 1 : 0][paged ? 1 : 0][mode];
  if (s.occ == 0 || s.smem != smem) {
    s.occ = fn(smem);
    s.smem = smem;
  }
  return s.occ;
}

}  // namespace

cudaError_t launch_decode(const Dims& d, const kvq_cache& c, const __half* q, int H_q, int q_pos,
                          const float2* rope, float sm_scale, __half* out, float* ws_all,
                          cudaStream_t st, int split_cap, const Paged* pg, uint32_t tx_pad,
                          const float* levels) {
  float* ws = ws_all + kWsHeaderBytes / sizeof(float);   // the partials follow the status word
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
  a.status = reinterpret_cast<uint32_t*>(ws_all);
  a.tx_pad = tx_pad;
  for (int k = 0; k < 256; ++k) a.lv[k] = (levels && k < (1 << d.bits)) ? levels[k] : 0.0f;
  // paged: the grid is sized for the longest sequence; each CTA reads its own length
  a.T = pg ? pg->max_len : c.T_cur;
  a.n_full = a.T / d.Bk;
  a.tail_len = a.T % d.Bk;
  a.block_table = pg ? pg->block_table : nullptr;
  a.seq_len = pg ? pg->seq_len : nullptr;
  a.max_blocks = pg ? pg->max_blocks : 0;
  a.n_blocks = pg ? pg->n_blocks : 0;
  a.H_q = H_q;
  a.q_pos = q_pos;
  a.S = (split_cap > 0 && split_cap < max_splits(d)) ? split_cap : max_splits(d);
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  const int G = H_q / d.H_kv;

  int dev = 0, sms = 0;
  if (current_device(&dev) != KVQ_OK) return cudaErrorInvalidDevice;   // the API checked it first
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int units = a.n_full + (a.tail_len > 0 ? 1 : 0);

  if (d.D == 128) {
    CUtensorMap tk, tv;
    const size_t n_units = pg ? (size_t)pg->n_blocks * d.H_kv : 0;
    if (!encode_codes(&tk, c.k_codes, d, n_units) || !encode_codes(&tv, c.v_codes, d, n_units))
      return cudaErrorInvalidValue;
    const tc::StageLayout L = stage_layout(d);
    const size_t smem = (size_t)tc::ring_stages(d.Bk) * L.stage_bytes + 1024;
    TcLaunchFn fn = nullptr;
    TcOccFn occ_fn = nullptr;
    const bool paged = pg != nullptr;
    const int mode = levels ? 2 : (d.flags & KVQ_FLAG_PRECISE_SCORES) ? 1 : 0;
    if (mode == 2 && paged) return cudaErrorInvalidValue;   // the API asks for contiguous caches only
    switch (d.bits) {
      case 2: pick_tc<2>(d.Bk, G, d.n_out > 0, paged, mode, &fn, &occ_fn); break;
      case 3: pick_tc<3>(d.Bk, G, d.n_out > 0, paged, mode, &fn, &occ_fn); break;
      case 8: pick_tc<8>(d.Bk, G, d.n_out > 0, paged, mode, &fn, &occ_fn); break;
      default: pick_tc<4>(d.Bk, G, d.n_out > 0, paged, mode, &fn, &occ_fn); break;
    }
    const int occ = cached_tc_occupancy(dev, d.bits, d.Bk, G, d.n_out > 0, paged, mode, smem, occ_fn);
    a.n_split = paged ? paged_splits(d, units, sms * occ, a.S) : choose_splits(d.B * d.H_kv, units, sms * occ, a.S);
    e = fn(a, L, tk, tv, smem, st);
  } else {
    LaunchFn fn = nullptr;
    OccFn occ_fn = nullptr;
    switch (d.bits) {
      case 2: pick_g<2, 64>(G, &fn, &occ_fn); break;
      case 3: pick_g<3, 64>(G, &fn, &occ_fn); break;
      case 8: pick_g<8, 64>(G, &fn, &occ_fn); break;
      default: pick_g<4, 64>(G, &fn, &occ_fn); break;
    }
    const int occ = cached_occupancy(dev, d.bits, d.D, G, occ_fn);
    a.n_split = pg ? paged_splits(d, units, sms * occ, a.S) : choose_splits(d.B * d.H_kv, units, sms * occ, a.S);
    e = fn(a, st);
  }
  if (e != cudaSuccess) return e;
  if (d.D == 64)
    decode_combine_kernel<64><<<d.B * H_q, 64, 0, st>>>(ws, out, a.n_split, a.S);
  else
    decode_combine_kernel<128><<<d.B * H_q, 128, 0, st>>>(ws, out, a.n_split, a.S);
  return cudaGetLastError();
}

}  // namespace kvq
