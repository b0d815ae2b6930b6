// C ABI of libkvq: argument checks, buffer layout, and kernel launches.
// Every check runs on the host before any launch; the library never
// allocates, frees or synchronizes.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include <cuda.h>

#include "kvq_common.cuh"
#include "kvq_levels.cuh"

namespace kvq {
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int n_outliers(const kvq_config& c) {
  if (!(c.outlier_frac > 0.0f)) return 0;
  int n = (int)floor((double)c.outlier_frac * (double)c.D);
  return n < 1 ? 1 : n;
}

// Fills `d` from `cfg`; returns a status.
int make_dims(const kvq_config* cfg, Dims* d) {
  if (!cfg || !d) return KVQ_ERR_ARG;
  const kvq_config& c = *cfg;
  if (c.B < 1 || c.H_kv < 1 || c.T_max < 1) return KVQ_ERR_UNSUPPORTED;
  if (c.bits != 2 && c.bits != 3 && c.bits != 4 && c.bits != 8) return KVQ_ERR_UNSUPPORTED;
  if (c.D != 64 && c.D != 128) return KVQ_ERR_UNSUPPORTED;
  if (c.key_block != 64 && c.key_block != 128) return KVQ_ERR_UNSUPPORTED;
  if (c.value_group != 32 && c.value_group != 64 && c.value_group != 128) return KVQ_ERR_UNSUPPORTED;
  if (c.D % c.value_group) return KVQ_ERR_UNSUPPORTED;
  if (c.T_max % c.key_block || c.T_max >= (1 << 24)) return KVQ_ERR_UNSUPPORTED;
  if (!(c.outlier_frac >= 0.0f) || c.outlier_frac > 1.0f) return KVQ_ERR_UNSUPPORTED;
  const int n_out = n_outliers(c);
  if (n_out > KVQ_MAX_OUTLIERS) return KVQ_ERR_UNSUPPORTED;
  if ((int64_t)c.B * c.H_kv > 65535) return KVQ_ERR_UNSUPPORTED;  // grid.y
  if (c.flags & ~KVQ_FLAG_PRECISE_SCORES) return KVQ_ERR_UNSUPPORTED;
  d->B = c.B;
  d->H_kv = c.H_kv;
  d->D = c.D;
  d->T_max = c.T_max;
  d->bits = c.bits;
  d->Bk = c.key_block;
  d->Gv = c.value_group;
  d->n_out = n_out;
  d->cb = c.D * c.bits / 8;
  d->ng = c.D / c.value_group;
  d->n_blk = c.T_max / c.key_block;
  d->rope_n_hi = rope_n_hi(d->n_blk);
  d->flags = c.flags;
  return KVQ_OK;
}

bool cache_ptrs_ok(const Dims& d, const kvq_cache& c) {
  const void* must[] = {c.k_codes, c.k_meta, c.k_tail, c.v_codes, c.v_meta};
  for (const void* p : must)
    if (!p || !aligned16(p)) return false;
  if (d.n_out > 0) {
    if (!c.k_outl || !c.v_outl || !aligned16(c.k_outl) || !aligned16(c.v_outl)) return false;
  }
  return c.T_cur >= 0 && c.T_cur <= d.T_max;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Pools, table and lengths of a paged cache; the block count keeps every
// block index a valid 32-bit TMA coordinate.
bool paged_ptrs_ok(const Dims& d, const kvq_paged_cache& c) {
  const void* must[] = {c.k_codes, c.k_meta, c.k_tail, c.v_codes, c.v_meta};
  for (const void* p : must)
    if (!p || !aligned16(p)) return false;
  if (d.n_out > 0) {
    if (!c.k_outl || !c.v_outl || !aligned16(c.k_outl) || !aligned16(c.v_outl)) return false;
  }
  if (!c.block_table || !c.seq_len || !aligned4(c.block_table) || !aligned4(c.seq_len)) return false;
  if (c.n_blocks < 1 || (int64_t)c.n_blocks * d.H_kv >= ((int64_t)1 << 31)) return false;
  return c.max_len >= 0 && c.max_len <= d.T_max;
}

// The pools as the kernels' buffer set, and the paging information.
kvq_cache pool_view(const kvq_paged_cache& c) {
  kvq_cache v;
  v.k_codes = c.k_codes;
  v.k_meta = c.k_meta;
  v.k_tail = c.k_tail;
  v.k_outl = c.k_outl;
  v.v_codes = c.v_codes;
  v.v_meta = c.v_meta;
  v.v_outl = c.v_outl;
  v.T_cur = 0;
  return v;
}
Paged paging(const Dims& d, const kvq_paged_cache& c) {
  Paged pg;
  pg.block_table = c.block_table;
  pg.seq_len = c.seq_len;
  pg.max_blocks = d.n_blk;
  pg.n_blocks = c.n_blocks;
  pg.max_len = c.max_len;
  return pg;
}

// Host checks of kvq_decode_attn for a cache holding T_cur tokens.
int decode_checks(const kvq_config* cfg, const Dims& d, const kvq_cache* cache, int32_t T_cur,
                  const void* q, int32_t H_q, int32_t q_pos, const void* rope_tab, float sm_scale,
                  const void* out, const void* workspace, size_t workspace_bytes) {
  if (H_q < 1 || H_q % d.H_kv) return KVQ_ERR_UNSUPPORTED;
  const int G = H_q / d.H_kv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return KVQ_ERR_UNSUPPORTED;
  if (!cache || !cache_ptrs_ok(d, *cache) || T_cur < 1) return KVQ_ERR_ARG;
  if (!q || !out || !workspace || !aligned16(q) || !aligned16(out) || !aligned16(workspace))
    return KVQ_ERR_ARG;
  if (q_pos < 0 || q_pos >= d.T_max || !isfinite(sm_scale)) return KVQ_ERR_ARG;
  if (rope_tab && !aligned16(rope_tab)) return KVQ_ERR_ARG;
  kvq_layout_t lay;
  const int rc = kvq_layout(cfg, H_q, &lay);
  if (rc) return rc;
  if (workspace_bytes < lay.workspace_bytes) return KVQ_ERR_WORKSPACE;
  return KVQ_OK;
}

// Scratch of kvq_decode_attn_noalloc: the split partials live in this
// file-scope device array instead of a caller-provided workspace. Every device
// that loads the library holds it until the process exits.
constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

// The driver's cuCtxGetCurrent, looked up once (thread-safe static init).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static const CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(p);
    return nullptr;
  }();
  return fn;
}

// Device address of g_noalloc_scratch on the current device. In host code
// the array's name is only a stand-in symbol, so the address is looked up
// with the device current and remembered per device together with the
// context it belongs to; a new context on the device (after cudaDeviceReset,
// say) reloads the module, so the address is looked up again.
int noalloc_scratch(float** out) {
  struct Entry {
    CUcontext ctx;
    float* addr;
  };
  static std::mutex mu;
  static Entry known[kMaxDevices] = {};
  int dev = 0;
  int rc = current_device(&dev);
  if (rc) return rc;
  const CtxGetCurrentFn get = ctx_get_current();
  if (!get) return KVQ_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return KVQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!ctx || known[dev].ctx != ctx || !known[dev].addr) {
    void* p = nullptr;   // the lookup also creates the device's context if there is none yet
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KVQ_ERR_CUDA;
    if (get(&ctx) != CUDA_SUCCESS || !ctx) return KVQ_ERR_CUDA;
    known[dev].ctx = ctx;
    known[dev].addr = static_cast<float*>(p);
  }
  *out = known[dev].addr;
  return KVQ_OK;
}

// The calling thread's device, if the library's per-device tables cover it.
int device_ok() {
  int dev = 0;
  return current_device(&dev);
}

// A level table from the caller's 2^bits levels: 0 first, 1 last, strictly
// increasing and finite; the midpoints are formed here in binary32.
bool make_levels(const float* levels, int bits, LevelTable* t) {
  if (!levels) return false;
  const int L = (1 << bits) - 1;
  if (!(levels[0] == 0.0f) || !(levels[L] == 1.0f)) return false;
  for (int k = 0; k < L; ++k)
    if (!(levels[k] < levels[k + 1])) return false;
  memset(t, 0, sizeof(*t));
  t->L = L;
  for (int k = 0; k <= L; ++k) t->lv[k] = levels[k];
  for (int k = 0; k < L; ++k) t->mid[k] = (levels[k] + levels[k + 1]) * 0.5f;
  return true;
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" {

int kvq_layout(const kvq_config* cfg, int32_t H_q, kvq_layout_t* out) {
  if (!cfg || !out) return KVQ_ERR_ARG;
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc) return rc;
  if (H_q < 1 || H_q % d.H_kv) return KVQ_ERR_UNSUPPORTED;
  memset(out, 0, sizeof(*out));
  const size_t streams = (size_t)d.B * d.H_kv;
  out->stream_bytes[KVQ_K_CODES] = k_codes_stream(d);
  out->stream_bytes[KVQ_K_META] = k_meta_stream(d) * 4;
  out->stream_bytes[KVQ_K_TAIL] = k_tail_stream(d) * 2;
  out->stream_bytes[KVQ_K_OUTL] = outl_stream(d) * 4;
  out->stream_bytes[KVQ_V_CODES] = k_codes_stream(d);
  out->stream_bytes[KVQ_V_META] = v_meta_stream(d) * 4;
  out->stream_bytes[KVQ_V_OUTL] = outl_stream(d) * 4;
  for (int i = 0; i < KVQ_NBUF; ++i) {
    out->bytes[i] = out->stream_bytes[i] * streams;
    out->cache_bytes += out->bytes[i];
  }
  out->fp16_equiv_bytes = 2 * streams * (size_t)d.T_max * d.D * 2;
  out->rope_bytes = rope_entries(d) * sizeof(float2);
  out->workspace_bytes = kWsHeaderBytes + (size_t)d.B * H_q * max_splits(d) * (d.D + 2) * sizeof(float);
  out->n_out = d.n_out;
  out->code_row_bytes = d.cb;
  return KVQ_OK;
}

int kvq_rope_init(const kvq_config* cfg, double rope_theta, void* rope_tab, size_t rope_bytes,
                  void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc) return rc;
  if (!rope_tab || !aligned16(rope_tab) || !(rope_theta > 0.0) || !isfinite(rope_theta))
    return KVQ_ERR_ARG;
  if (rope_bytes < rope_entries(d) * sizeof(float2)) return KVQ_ERR_WORKSPACE;
  rc = device_ok();
  if (rc) return rc;
  return cuda_status(launch_rope_init(d, rope_theta, static_cast<float2*>(rope_tab),
                                      static_cast<cudaStream_t>(stream)));
}

int kvq_append(const kvq_config* cfg, kvq_cache* cache, const void* k_new, const void* v_new,
               int32_t n_new, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc) return rc;
  if (!cache || n_new < 0 || !cache_ptrs_ok(d, *cache)) return KVQ_ERR_ARG;
  if (n_new == 0) return KVQ_OK;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_ARG;
  if ((int64_t)cache->T_cur + n_new > d.T_max) return KVQ_ERR_CAPACITY;
  rc = device_ok();
  if (rc) return rc;
  rc = cuda_status(launch_append(d, *cache, static_cast<const __half*>(k_new),
                                 static_cast<const __half*>(v_new), n_new,
                                 static_cast<cudaStream_t>(stream)));
  if (rc == KVQ_OK) cache->T_cur += n_new;
  return rc;
}

int kvq_append_window(const kvq_config* cfg, kvq_cache* cache, const void* k_new, const void* v_new,
                      int32_t n_new, int32_t window, void* k_bstat, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc) return rc;
  if (window < d.Bk || window % d.Bk) return KVQ_ERR_UNSUPPORTED;
  if (!cache || n_new < 0 || !cache_ptrs_ok(d, *cache)) return KVQ_ERR_ARG;
  if (!k_bstat || !aligned16(k_bstat)) return KVQ_ERR_ARG;
  if (n_new == 0) return KVQ_OK;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_ARG;
  if ((int64_t)cache->T_cur + n_new > d.T_max) return KVQ_ERR_CAPACITY;
  rc = device_ok();
  if (rc) return rc;
  rc = cuda_status(launch_append(d, *cache, static_cast<const __half*>(k_new), static_cast<const __half*>(v_new),
                                 n_new, static_cast<cudaStream_t>(stream), nullptr, window / d.Bk,
                                 static_cast<uint32_t*>(k_bstat)));
  if (rc == KVQ_OK) cache->T_cur += n_new;
  return rc;
}

int kvq_decode_attn(const kvq_config* cfg, const kvq_cache* cache, const void* q, int32_t H_q,
                    int32_t q_pos, const void* rope_tab, float sm_scale, void* out,
                    void* workspace, size_t workspace_bytes, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc) return rc;
  rc = decode_checks(cfg, d, cache, cache ? cache->T_cur : 0, q, H_q, q_pos, rope_tab, sm_scale, out,
                     workspace, workspace_bytes);
  if (rc) return rc;
  rc = device_ok();
  if (rc) return rc;
  return cuda_status(launch_decode(d, *cache, static_cast<const __half*>(q), H_q, q_pos,
                                   static_cast<const float2*>(rope_tab), sm_scale,
                                   static_cast<__half*>(out), static_cast<float*>(workspace),
                                   static_cast<cudaStream_t>(stream)));
}

int kvq_decode_attn_diag(const kvq_config* cfg, const kvq_cache* cache, const void* q, int32_t H_q,
                         int32_t q_pos, const void* rope_tab, float sm_scale, void* out, void* workspace,
                         size_t workspace_bytes, uint32_t tx_pad, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc) return rc;
  rc = decode_checks(cfg, d, cache, cache ? cache->T_cur : 0, q, H_q, q_pos, rope_tab, sm_scale, out,
                     workspace, workspace_bytes);
  if (rc) return rc;
  if (d.D != 128 || (tx_pad & 15u)) return KVQ_ERR_UNSUPPORTED;
  rc = device_ok();
  if (rc) return rc;
  return cuda_status(launch_decode(d, *cache, static_cast<const __half*>(q), H_q, q_pos,
                                   static_cast<const float2*>(rope_tab), sm_scale,
                                   static_cast<__half*>(out), static_cast<float*>(workspace),
                                   static_cast<cudaStream_t>(stream), 0, nullptr, tx_pad));
}

int kvq_decode_step(const kvq_config* cfg, kvq_cache* cache, const void* k_new, const void* v_new,
                    const void* q, int32_t H_q, const void* rope_tab, float sm_scale, void* out,
                    void* workspace, size_t workspace_bytes, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc) return rc;
  if (!cache || !cache_ptrs_ok(d, *cache)) return KVQ_ERR_ARG;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_ARG;
  if (cache->T_cur + 1 > d.T_max) return KVQ_ERR_CAPACITY;
  const int32_t pos = cache->T_cur;                  // the new token's position
  rc = decode_checks(cfg, d, cache, pos + 1, q, H_q, pos, rope_tab, sm_scale, out, workspace,
                     workspace_bytes);
  if (rc) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = device_ok();
  if (rc) return rc;
  rc = cuda_status(launch_append(d, *cache, static_cast<const __half*>(k_new),
                                 static_cast<const __half*>(v_new), 1, st));
  if (rc) return rc;
  cache->T_cur = pos + 1;
  return cuda_status(launch_decode(d, *cache, static_cast<const __half*>(q), H_q, pos,
                                   static_cast<const float2*>(rope_tab), sm_scale,
                                   static_cast<__half*>(out), static_cast<float*>(workspace), st));
}

int kvq_decode_attn_noalloc(const kvq_config* cfg, const kvq_cache* cache, const void* q, int32_t H_q,
                            int32_t q_pos, const void* rope_tab, float sm_scale, void* out,
                            void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc) return rc;
  if (H_q < 1 || H_q % d.H_kv) return KVQ_ERR_UNSUPPORTED;
  const int G = H_q / d.H_kv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return KVQ_ERR_UNSUPPORTED;
  if (!cache || !cache_ptrs_ok(d, *cache) || cache->T_cur < 1) return KVQ_ERR_ARG;
  if (!q || !out || !aligned16(q) || !aligned16(out)) return KVQ_ERR_ARG;
  if (q_pos < 0 || q_pos >= d.T_max || !isfinite(sm_scale)) return KVQ_ERR_ARG;
  if (rope_tab && !aligned16(rope_tab)) return KVQ_ERR_ARG;
  // one T split needs (D + 2) floats per (sequence, query head)
  const size_t split_bytes = (size_t)d.B * H_q * (d.D + 2) * sizeof(float);
  const size_t fit = (kNoAllocScratchBytes - kWsHeaderBytes) / split_bytes;
  if (fit < 1) return KVQ_ERR_WORKSPACE;
  float* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  return cuda_status(launch_decode(d, *cache, static_cast<const __half*>(q), H_q, q_pos,
                                   static_cast<const float2*>(rope_tab), sm_scale,
                                   static_cast<__half*>(out), scratch,
                                   static_cast<cudaStream_t>(stream), fit > 256 ? 256 : (int)fit));
}

int kvq_paged_layout(const kvq_config* cfg, int32_t n_blocks, int32_t H_q, kvq_layout_t* out) {
  if (!cfg || !out) return KVQ_ERR_ARG;
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc) return rc;
  if (H_q < 1 || H_q % d.H_kv) return KVQ_ERR_UNSUPPORTED;
  if (n_blocks < 1 || (int64_t)n_blocks * d.H_kv >= ((int64_t)1 << 31)) return KVQ_ERR_UNSUPPORTED;
  kvq_layout_t base;
  rc = kvq_layout(cfg, H_q, &base);
  if (rc) return rc;
  memset(out, 0, sizeof(*out));
  const size_t rows = (size_t)d.H_kv * d.Bk;      // rows of one physical block, all heads
  out->stream_bytes[KVQ_K_CODES] = rows * d.cb;
  out->stream_bytes[KVQ_K_META] = (size_t)d.H_kv * d.D * 4;
  out->stream_bytes[KVQ_K_TAIL] = k_tail_stream(d) * 2 * d.H_kv;   // per sequence
  out->stream_bytes[KVQ_K_OUTL] = rows * d.n_out * 4;
  out->stream_bytes[KVQ_V_CODES] = rows * d.cb;
  out->stream_bytes[KVQ_V_META] = rows * d.ng * 4;
  out->stream_bytes[KVQ_V_OUTL] = rows * d.n_out * 4;
  for (int i = 0; i < KVQ_NBUF; ++i) {
    out->bytes[i] = out->stream_bytes[i] * (i == KVQ_K_TAIL ? (size_t)d.B : (size_t)n_blocks);
    out->cache_bytes += out->bytes[i];
  }
  out->fp16_equiv_bytes = 2 * (size_t)n_blocks * rows * d.D * 2;
  out->rope_bytes = base.rope_bytes;
  out->workspace_bytes = base.workspace_bytes;
  out->n_out = d.n_out;
  out->code_row_bytes = d.cb;
  return KVQ_OK;
}

int kvq_paged_append(const kvq_config* cfg, kvq_paged_cache* cache, const void* k_new, const void* v_new,
                     int32_t n_new, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc) return rc;
  if (!cache || n_new < 0 || !paged_ptrs_ok(d, *cache)) return KVQ_ERR_ARG;
  if (n_new == 0) return KVQ_OK;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_ARG;
  if ((int64_t)cache->max_len + n_new > d.T_max) return KVQ_ERR_CAPACITY;
  const Paged pg = paging(d, *cache);
  rc = device_ok();
  if (rc) return rc;
  rc = cuda_status(launch_append(d, pool_view(*cache), static_cast<const __half*>(k_new),
                                 static_cast<const __half*>(v_new), n_new, static_cast<cudaStream_t>(stream), &pg));
  if (rc == KVQ_OK) cache->max_len += n_new;
  return rc;
}

int kvq_paged_decode_attn(const kvq_config* cfg, const kvq_paged_cache* cache, const void* q, int32_t H_q,
                          const void* rope_tab, float sm_scale, void* out, void* workspace,
                          size_t workspace_bytes, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc) return rc;
  if (H_q < 1 || H_q % d.H_kv) return KVQ_ERR_UNSUPPORTED;
  const int G = H_q / d.H_kv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return KVQ_ERR_UNSUPPORTED;
  if (!cache || !paged_ptrs_ok(d, *cache)) return KVQ_ERR_ARG;
  if (!q || !out || !workspace || !aligned16(q) || !aligned16(out) || !aligned16(workspace))
    return KVQ_ERR_ARG;
  if (!isfinite(sm_scale)) return KVQ_ERR_ARG;
  if (rope_tab && !aligned16(rope_tab)) return KVQ_ERR_ARG;
  kvq_layout_t lay;
  rc = kvq_layout(cfg, H_q, &lay);
  if (rc) return rc;
  if (workspace_bytes < lay.workspace_bytes) return KVQ_ERR_WORKSPACE;
  const Paged pg = paging(d, *cache);
  rc = device_ok();
  if (rc) return rc;
  return cuda_status(launch_decode(d, pool_view(*cache), static_cast<const __half*>(q), H_q, 0,
                                   static_cast<const float2*>(rope_tab), sm_scale, static_cast<__half*>(out),
                                   static_cast<float*>(workspace), static_cast<cudaStream_t>(stream), 0, &pg));
}

int kvq_fit_levels(const double* u, size_t n, int32_t bits, int32_t iters, float* levels) {
  if (!u || !levels || iters < 0) return KVQ_ERR_ARG;
  if (bits != 2 && bits != 3 && bits != 4 && bits != 8) return KVQ_ERR_UNSUPPORTED;
  const int L = (1 << bits) - 1;
  // Lloyd iterations on the sorted samples: a cell is a run of the sorted
  // values, found by binary search; its mean comes from prefix sums.
  std::vector<double> x(u, u + n);
  for (double v : x)
    if (!(v >= 0.0 && v <= 1.0)) return KVQ_ERR_ARG;
  std::sort(x.begin(), x.end());
  std::vector<double> pre(n + 1, 0.0);
  for (size_t i = 0; i < n; ++i) pre[i + 1] = pre[i] + x[i];
  std::vector<double> lv(L + 1), edge(L + 1);
  for (int k = 0; k <= L; ++k) lv[k] = (double)k / L;
  for (int it = 0; it < iters; ++it) {
    // cell k holds the samples in (mid_{k-1}, mid_k]: ties go to the lower level
    edge[0] = 0;
    for (int k = 0; k < L; ++k) {
      const double mid = 0.5 * (lv[k] + lv[k + 1]);
      edge[k + 1] = (double)(std::upper_bound(x.begin(), x.end(), mid) - x.begin());
    }
    for (int k = 1; k < L; ++k) {
      const size_t lo = (size_t)edge[k], hi = (size_t)edge[k + 1];
      if (hi > lo) lv[k] = (pre[hi] - pre[lo]) / (double)(hi - lo);
    }
  }
  for (int k = 0; k <= L; ++k) levels[k] = (float)lv[k];
  // Levels distinct in binary64 can round to one binary32 value (tightly
  // clustered samples); keep the table strictly increasing, as the append and
  // decode calls require, by moving such a level up by one ulp (a backward
  // pass keeps every interior level below l_L = 1).
  for (int k = 1; k < L; ++k)
    if (!(levels[k] > levels[k - 1])) levels[k] = nextafterf(levels[k - 1], 2.0f);
  for (int k = L - 1; k >= 1; --k)
    if (!(levels[k] < levels[k + 1])) levels[k] = nextafterf(levels[k + 1], -1.0f);
  return KVQ_OK;
}

int kvq_append_levels(const kvq_config* cfg, kvq_cache* cache, const void* k_new, const void* v_new,
                      int32_t n_new, const float* levels, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc) return rc;
  if (!cache || n_new < 0 || !cache_ptrs_ok(d, *cache)) return KVQ_ERR_ARG;
  LevelTable t;
  if (!make_levels(levels, d.bits, &t)) return KVQ_ERR_ARG;
  if (n_new == 0) return KVQ_OK;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_ARG;
  if ((int64_t)cache->T_cur + n_new > d.T_max) return KVQ_ERR_CAPACITY;
  rc = device_ok();
  if (rc) return rc;
  // the uniform append's kernel in its level-table mode (fp16 tail of an unfinished key block included)
  rc = cuda_status(launch_append(d, *cache, static_cast<const __half*>(k_new), static_cast<const __half*>(v_new),
                                 n_new, static_cast<cudaStream_t>(stream), nullptr, 0, nullptr, t.mid));
  if (rc == KVQ_OK) cache->T_cur += n_new;
  return rc;
}

int kvq_decode_attn_levels(const kvq_config* cfg, const kvq_cache* cache, const void* q, int32_t H_q,
                           int32_t q_pos, const void* rope_tab, float sm_scale, void* out, void* workspace,
                           size_t workspace_bytes, const float* levels, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc) return rc;
  rc = decode_checks(cfg, d, cache, cache ? cache->T_cur : 0, q, H_q, q_pos, rope_tab, sm_scale, out,
                     workspace, workspace_bytes);
  if (rc) return rc;
  LevelTable t;
  if (!make_levels(levels, d.bits, &t)) return KVQ_ERR_ARG;
  rc = device_ok();
  if (rc) return rc;
  if (d.D == 128 && !(d.flags & KVQ_FLAG_PRECISE_SCORES))   // the tensor-core kernel
    return cuda_status(launch_decode(d, *cache, static_cast<const __half*>(q), H_q, q_pos,
                                     static_cast<const float2*>(rope_tab), sm_scale, static_cast<__half*>(out),
                                     static_cast<float*>(workspace), static_cast<cudaStream_t>(stream), 0, nullptr,
                                     0, t.lv));
  return cuda_status(launch_decode_levels(d, *cache, static_cast<const __half*>(q), H_q, q_pos,
                                          static_cast<const float2*>(rope_tab), sm_scale,
                                          static_cast<__half*>(out), static_cast<float*>(workspace), t,
                                          static_cast<cudaStream_t>(stream)));
}

int kvq_decode_step_levels(const kvq_config* cfg, kvq_cache* cache, const void* k_new, const void* v_new,
                           const void* q, int32_t H_q, const void* rope_tab, float sm_scale, void* out,
                           void* workspace, size_t workspace_bytes, const float* levels, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc) return rc;
  if (!cache || !cache_ptrs_ok(d, *cache)) return KVQ_ERR_ARG;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_ARG;
  LevelTable t;
  if (!make_levels(levels, d.bits, &t)) return KVQ_ERR_ARG;
  if (cache->T_cur + 1 > d.T_max) return KVQ_ERR_CAPACITY;
  const int32_t pos = cache->T_cur;                  // the new token's position
  rc = decode_checks(cfg, d, cache, pos + 1, q, H_q, pos, rope_tab, sm_scale, out, workspace,
                     workspace_bytes);
  if (rc) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = device_ok();
  if (rc) return rc;
  rc = cuda_status(launch_append(d, *cache, static_cast<const __half*>(k_new), static_cast<const __half*>(v_new),
                                 1, st, nullptr, 0, nullptr, t.mid));
  if (rc) return rc;
  cache->T_cur = pos + 1;
  if (d.D == 128 && !(d.flags & KVQ_FLAG_PRECISE_SCORES))   // the tensor-core kernel
    return cuda_status(launch_decode(d, *cache, static_cast<const __half*>(q), H_q, pos,
                                     static_cast<const float2*>(rope_tab), sm_scale, static_cast<__half*>(out),
                                     static_cast<float*>(workspace), st, 0, nullptr, 0, t.lv));
  return cuda_status(launch_decode_levels(d, *cache, static_cast<const __half*>(q), H_q, pos,
                                          static_cast<const float2*>(rope_tab), sm_scale,
                                          static_cast<__half*>(out), static_cast<float*>(workspace), t, st));
}

const char* kvq_status_string(int status) {
  switch (status) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_ARG: return "KVQ_ERR_ARG: invalid argument (NULL/misaligned pointer, bad count or position)";
    case KVQ_ERR_UNSUPPORTED: return "KVQ_ERR_UNSUPPORTED: configuration outside the supported set";
    case KVQ_ERR_CAPACITY: return "KVQ_ERR_CAPACITY: T_cur + n_new exceeds T_max";
    case KVQ_ERR_WORKSPACE: return "KVQ_ERR_WORKSPACE: workspace or table smaller than kvq_layout() requires";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA: CUDA launch error";
    case KVQ_ERR_TIMEOUT: return "KVQ_ERR_TIMEOUT: a bounded wait of a kernel expired (status word)";
    default: return "KVQ_ERR_UNKNOWN";
  }
}

const char* kvq_version(void) { return "kvq 0.2.0 sm_103a"; }

}  // extern "C"
