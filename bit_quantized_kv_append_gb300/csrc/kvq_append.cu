// kvq_append: quantize new keys and values into the packed cache.
//
// KV Cache量化技术介绍 (developer.horizon.auto/blog/13163):
//   KVQuant "Per-Vector Dense-and-Sparse Quantization" -> step B (outliers);
//   KVQuant "Per-Channel Key Quantization"             -> step C, keys;
//   Quanto steps 1-2 (block scale and zero_point)       -> step C, values;
//   codes and LSB-first packing                         -> step D.
// Grid: (key block touched by the append, (b, h_kv) stream, {values, keys}).
// A value CTA quantizes the block's new value rows; a key CTA quantizes the
// block's keys when the append completes it (keys read so far come back from
// K_TAIL) and otherwise copies the new keys into K_TAIL. Rows are staged in
// shared memory; then, in the method's order:
//   B. outliers: the n_out largest |x| of every row (two threads per row for
//      n_out = 1, a warp per row otherwise); their staged copies become NaN,
//      which the fp16 min/max of step C skip;
//   C. scale and zero: values per (row, group) by one thread, keys per
//      channel by four or eight threads over row slices;
//   D. codes: 32 channels of a row per thread, two at a time in packed fp32
//      (x - z, times 1/s, rounded by the 1.5 * 2^23 addition), packed and
//      stored with one or three vector stores. The product with 1/s (1 ulp)
//      is within 4e-6 of the binary32 quotient for codes below 16, so a chunk
//      whose values all sit further than 1e-5 from a rounding tie gets the
//      codes of the exact division; a chunk with a near tie is recomputed
//      with it.
//      Outlier positions are recomputed from their stored value.
// All rounding follows the library's stated arithmetic: binary32 RN subtract
// and divide, fp16 round-up for the scale, round-half-even codes.
//
// Level tables (KVQuant "Non-Uniform KV Cache Quantization", same page; LV):
// the same kernel with r = fp16_round_up(fp32(max) - fp32(min)) in the scale's
// slot and the code of x the nearest level of u = fp32(fp32(x - z) / r): the
// number of binary32 midpoints of neighbouring levels below u (ties to the
// lower level), found by a binary search over the midpoints in shared memory.
#include <atomic>
#include <type_traits>

#include "kvq_common.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxGroups = 4;       // D / Gv <= 128 / 32
// |t| above 0.5 - guard: recompute the chunk exactly. The guard exceeds the
// distance between y and the binary32 quotient, at most 2^-22 |y| (below
// 3.9e-6 for codes under 16, 6.2e-5 for the 8-bit codes under 256).
template <int BITS>
__host__ __device__ constexpr float tie_guard() { return BITS <= 4 ? 1e-5f : 1e-4f; }
constexpr float kMagic = 12582912.0f;   // 1.5 * 2^23: x + kMagic rounds x to an integer (ties even)

struct AppendArgs {
  Dims d;
  uint8_t* k_codes;
  uint32_t* k_meta;
  __half* k_tail;
  uint32_t* k_outl;
  uint8_t* v_codes;
  uint32_t* v_meta;
  uint32_t* v_outl;
  const __half* k_new;
  const __half* v_new;
  int T_cur, n_new, first_blk;
  int tail_in_kernel;  // 1: an unfinished last block's keys go to K_TAIL in this launch
  const int32_t* block_table;  // paged cache (NULL: contiguous streams); then the
  const int32_t* seq_len;      // position, first block and tail rule are per sequence
  int max_blocks, n_blocks;
  // Sliding-window key statistics (0: the block's own statistics). Phase 1
  // quantizes the values, selects the key outliers and stores each finished
  // key block's dense {min, max} per channel in k_bstat; phase 2 (key CTAs
  // only, a later launch) takes (s, z) from the last window_blocks blocks'
  // {min, max} and writes the key codes and metadata.
  int phase;
  int window_blocks;
  uint32_t* k_bstat;
};

// Paged append: position of sequence b (its length, kept inside the capacity).
__device__ __forceinline__ int paged_pos(const AppendArgs& a, int b) {
  const int t = __ldg(a.seq_len + b), hi = a.d.T_max - a.n_new;
  return t < 0 ? 0 : (t > hi ? hi : t);
}
// An append whose first block reads the old tail and whose last block is
// unfinished and different writes that last block's keys in a second launch.
__device__ __host__ __forceinline__ bool tail_deferred(int T_cur, int n_new, int Bk) {
  const int first = T_cur / Bk, last = (T_cur + n_new - 1) / Bk;
  return ((T_cur + n_new) % Bk) != 0 && first != last && (T_cur % Bk) != 0;
}

__device__ __forceinline__ uint16_t hbits(__half h) { return __half_as_ushort(h); }

// fp32(h) + c, rounded once (the fp16 -> fp32 widening is exact).
__device__ __forceinline__ float add_h_f(uint16_t h, float c) {
  float d;
  asm("add.rn.f32.f16 %0, %1, %2;" : "=f"(d) : "h"(h), "f"(c));
  return d;
}

// 1/s to within 1 ulp (hardware approximation); 0 for s = 0. With it the
// products below are within 4e-6 of the quotients for |y| < 16, inside the
// tie guard.
__device__ __forceinline__ float rcp_or_zero(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return s > 0.0f ? r : 0.0f;
}

// clamp(rint(fl((x - z) / s)), 0, L) in binary32 round-to-nearest (0 when
// s = 0), computed without a division: y = (x - z) * r with r within 1 ulp of
// 1/s is within 2^-22 |y| of the binary32 quotient Q = fl((x - z) / s) (4e-6
// for |y| < 16, 6.2e-5 for |y| < 256). Away from the half-integers the
// rounding of y is that of Q. Near
// a half-integer h the exact residual rho = (x - z) - h*s (one fma, exact) and
// half an ulp of h, times s (exact), tell whether Q rounds to h (then ties go
// to the even integer) or to a neighbour; "near" is the width's tie guard,
// which exceeds the distance between y and Q. Beyond [-0.75, L + 0.75] the
// clamp decides.
template <int BITS>
__device__ __forceinline__ uint32_t exact_code(float x, float z, float s, float r) {
  constexpr int L = (1 << BITS) - 1;
  if (!(s > 0.0f)) return 0u;
  const float d = __fsub_rn(x, z);
  const float y = __fmul_rn(d, r);
  if (y > (float)L + 0.75f) return (uint32_t)L;
  if (!(y > -0.75f)) return 0u;
  const float fl = floorf(y), h = fl + 0.5f;
  float q;
  if (fabsf(y - h) > tie_guard<BITS>()) {
    q = rintf(y);
  } else {
    const float rho = __fmaf_rn(-h, s, d);
    const int e = ilogbf(h);                                     // ulp(h) = 2^(e - 23)
    const float hs = s * __int_as_float((e - 24 + 127) << 23);   // half an ulp of h, times s
    if (rho > hs) q = fl + 1.0f;
    else if (rho < -hs) q = fl;
    else q = (((int)fl) & 1) ? fl + 1.0f : fl;                  // Q == h: ties to even
  }
  q = fminf(fmaxf(q, 0.0f), (float)L);
  return (uint32_t)q;
}

// Scale and zero of one group from the min/max of its dense elements.
// Returns the packed fp16 pair {s (low half), z (high half)}.
__device__ __forceinline__ uint32_t group_params(float mn, float mx, bool any, float Lf,
                                                 float2* sz) {
  if (!any) {  // every element of the group is an outlier
    *sz = make_float2(0.0f, 0.0f);
    return 0u;
  }
  const __half sh = __float2half_ru(__fdiv_rn(__fsub_rn(mx, mn), Lf));
  const float z = (mn == 0.0f) ? 0.0f : mn;     // -0 stored as +0
  const __half zh = __float2half_rn(z);         // exact: mn is an fp16 value
  *sz = make_float2(__half2float(sh), z);
  return (uint32_t)hbits(sh) | ((uint32_t)hbits(zh) << 16);
}

// Level tables: range and zero of a group, {r (low half), z (high half)} as
// fp16 bits; sz = (r, z) in binary32. No dense element: r = z = 0.
__device__ __forceinline__ uint32_t range_zero(float mn, float mx, bool any, float2* sz) {
  if (!any) {
    *sz = make_float2(0.0f, 0.0f);
    return 0u;
  }
  const __half rh = __float2half_ru(__fsub_rn(mx, mn));
  const float z = (mn == 0.0f) ? 0.0f : mn;     // -0 stored as +0; mn is an fp16 value: exact
  *sz = make_float2(__half2float(rh), z);
  return (uint32_t)hbits(rh) | ((uint32_t)hbits(__float2half_rn(z)) << 16);
}
// The midpoints of a table of 2^BITS levels, in the launch's parameters.
struct LvMid {
  float mid[255];
};
struct NoLv {
  int unused;
};
template <bool LV>
using LvParam = typename std::conditional<LV, LvMid, NoLv>::type;
// Number of midpoints below u (mid[0..2^BITS - 2], increasing); NaN: 0.
template <int BITS>
__device__ __forceinline__ uint32_t level_index(float u, const float* mid) {
  uint32_t q = 0u;
#pragma unroll
  for (int st = 1 << (BITS - 1); st > 0; st >>= 1)
    if (u > mid[q + st - 1]) q += st;
  return q;
}
// Level code of x with d = fp32(x - z) already formed; 0 when r = 0.
template <int BITS>
__device__ __forceinline__ uint32_t level_code_d(float d, float r, const float* mid) {
  return r > 0.0f ? level_index<BITS>(__fdiv_rn(d, r), mid) : 0u;
}
// The same code from y = d * (1/r), 1/r within one ulp (rcp_or_zero): y is
// within 2^-22 of fp32(d / r) for quotients up to 1, so a y further than
// 2^-20 from both neighbouring midpoints has the code of the exact quotient;
// otherwise the exact rule decides. NaN gives 0.
template <int BITS>
__device__ __forceinline__ uint32_t level_code_fast(float y, float d, float r, const float* mid) {
  constexpr uint32_t L = (1u << BITS) - 1u;
  constexpr float kEps = 9.5367431640625e-07f;   // 2^-20
  const uint32_t q = level_index<BITS>(y, mid);
  const float lo = q > 0u ? mid[q - 1u] : -INFINITY, hi = q < L ? mid[q] : INFINITY;
  if (!(y - lo <= kEps) && !(hi - y <= kEps)) return q;
  return level_code_d<BITS>(d, r, mid);
}

// Code-carrying bit patterns -> packed LSB-first words. A pattern is the
// float bits of y + kMagic for a code y in [0, 2^22): kMagicBits plus the code
// (every dense element is inside its group's range, and step C' sets the
// outlier positions to the group's zero, so every pattern of finite inputs
// has this form).
constexpr uint32_t kMagicBits = 0x4B400000u;   // float bits of 1.5 * 2^23
// 2, 3 and 4 bits: a word is the sum of its patterns shifted into their fields
// (one shift-add each, modulo 2^32) less the same shifts of kMagicBits, a
// compile-time constant; a code that straddles two words adds its high bits
// to the second from the bare code.
template <int BITS>
__host__ __device__ constexpr uint32_t pack_bias(int k) {
  uint32_t c = 0u;
  for (int e = 0; e < 32; ++e)
    if ((e * BITS) >> 5 == k) c += kMagicBits << ((e * BITS) & 31);
  return c;
}
template <int BITS>
__device__ __forceinline__ void pack_bits(const uint32_t (&mb)[32], uint32_t (&w)[BITS]) {
  if constexpr (BITS == 8) {
#pragma unroll
    for (int k = 0; k < 8; ++k)   // low byte of each pattern is the code
      w[k] = __byte_perm(__byte_perm(mb[4 * k], mb[4 * k + 1], 0x0040u),
                         __byte_perm(mb[4 * k + 2], mb[4 * k + 3], 0x0040u), 0x5410u);
  } else {
#pragma unroll
    for (int k = 0; k < BITS; ++k) w[k] = 0u - pack_bias<BITS>(k);
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int bit = e * BITS, sh = bit & 31;
      w[bit >> 5] += mb[e] << sh;
      if (sh + BITS > 32) w[(bit >> 5) + 1] += (mb[e] - kMagicBits) >> (32 - sh);
    }
  }
}

// Replace code e of a packed 32-code chunk.
template <int BITS>
__device__ __forceinline__ void set_code(uint32_t (&w)[BITS], int e, uint32_t q) {
  constexpr uint32_t M = (1u << BITS) - 1u;
  const int bit = e * BITS, wi = bit >> 5, sh = bit & 31;
#pragma unroll
  for (int k = 0; k < BITS; ++k) {
    if (k == wi) {
      w[k] = (w[k] & ~(M << sh)) | (q << sh);
      if (sh + BITS > 32 && k + 1 < BITS) {
        const int hi = sh + BITS - 32;
        w[k + 1] = (w[k + 1] & ~((1u << hi) - 1u)) | (q >> (32 - sh));
      }
    }
  }
}

// Staged rows are stored with their 16-byte chunks XOR-swizzled by the row
// (chunk c of row r at c ^ (r & 7)), so the row-parallel passes below read
// eight different bank groups per quarter warp.
__device__ __forceinline__ int sw_off(int r, int D, int col) {
  return r * D + ((((col >> 3) ^ (r & 7))) << 3) + (col & 7);
}

// Step D for one 32-channel chunk of row r: codes from the packed fp32 path,
// the exact rule for the elements near a rounding tie, and the outlier
// positions' codes (computed in step C'); returns the packed words.
template <int BITS, bool KEYS, bool LV>
__device__ __forceinline__ void chunk_codes(const __half* sX, const float4* sPv, const float4* sPk,
                                           const float* sS, const uint32_t* sO, const uint8_t* sQ, int D,
                                           int Bk, int r, int ch, int grp, int n_out, const float* mid,
                                           uint32_t (&w)[BITS]) {
  const float2 magic2 = make_float2(kMagic, kMagic), nmagic2 = make_float2(-kMagic, -kMagic);
  const float2 neg1 = make_float2(-1.0f, -1.0f);
  float4 vp = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!KEYS) vp = sPv[grp * Bk + r];
  uint32_t mb[32];
  uint32_t near = 0u;   // bit e: element e's quotient is within the guard of a rounding tie
  constexpr float kNear = 0.5f - tie_guard<BITS>();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 v = *reinterpret_cast<const uint4*>(sX + r * D + ((((4 * ch + k) ^ (r & 7))) << 3));
    const uint32_t hw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 8 * k + 2 * j;
      float2 nz2, r2;
      if (KEYS) {
        const float4 kp = sPk[(ch * 32 + e) >> 1];
        nz2 = make_float2(kp.x, kp.y);
        r2 = make_float2(kp.z, kp.w);
      } else {
        nz2 = make_float2(vp.x, vp.x);
        r2 = make_float2(vp.y, vp.y);
      }
      const float2 d2 = make_float2(add_h_f((uint16_t)(hw[j] & 0xFFFFu), nz2.x), add_h_f((uint16_t)(hw[j] >> 16), nz2.y));
      if constexpr (LV) {
        // r2 holds 1/r: the product, the midpoint search, the exact quotient
        // only next to a midpoint (outlier positions hold z: code 0, patched
        // below)
        const float2 u2 = __fmul2_rn(d2, r2);
        const float ra = KEYS ? sS[ch * 32 + e] : vp.z, rb = KEYS ? sS[ch * 32 + e + 1] : vp.z;
        mb[e] = kMagicBits | level_code_fast<BITS>(u2.x, d2.x, ra, mid);
        mb[e + 1] = kMagicBits | level_code_fast<BITS>(u2.y, d2.y, rb, mid);
        continue;
      }
      const float2 y2 = __fmul2_rn(d2, r2);
      const float2 m2 = __fadd2_rn(y2, magic2);
      const float2 t2 = __ffma2_rn(__fadd2_rn(m2, nmagic2), neg1, y2);   // y - rint(y)
      // NaN compares false
      near |= (fabsf(t2.x) > kNear ? 1u : 0u) << e;
      near |= (fabsf(t2.y) > kNear ? 1u : 0u) << (e + 1);
      mb[e] = __float_as_uint(m2.x);
      mb[e + 1] = __float_as_uint(m2.y);
    }
  }
  pack_bits<BITS>(mb, w);
  // the few elements near a tie: exact rule, one element at a time
  while (near) {
    const int e = __ffs(near) - 1;
    near &= near - 1u;
    const int c = ch * 32 + e;
    const float x = __half2float(sX[sw_off(r, D, c)]);
    float z, sc, rc;
    if (KEYS) {
      z = -reinterpret_cast<const float*>(&sPk[c >> 1])[c & 1];
      rc = reinterpret_cast<const float*>(&sPk[c >> 1])[2 + (c & 1)];
      sc = sS[c];
    } else {
      z = -vp.x;
      rc = vp.y;
      sc = vp.z;
    }
    set_code<BITS>(w, e, exact_code<BITS>(x, z, sc, rc));
  }
  for (int o = 0; o < n_out; ++o) {
    const int c = (int)(sO[o * Bk + r] & 0xFFFFu);
    if ((c >> 5) == ch) set_code<BITS>(w, c & 31, sQ[o * Bk + r]);
  }
}

template <int BITS, int D, bool LV>
__global__ void __launch_bounds__(kThreads) append_kernel(const AppendArgs a, const LvParam<LV> lp) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ float s_mid[LV ? 256 : 1];   // LV: the table's midpoints
  if constexpr (LV) {
    for (int k = threadIdx.x; k < (1 << BITS) - 1; k += kThreads) s_mid[k] = lp.mid[k];
  }
  const Dims d = a.d;
  const int Bk = d.Bk, n_out = d.n_out;
  const int tid = threadIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / d.H_kv, h = bh - b * d.H_kv;
  const bool isK = a.phase == 2 || blockIdx.z != 0;
  int T_cur = a.T_cur, first_blk = a.first_blk, tail_in_kernel = a.tail_in_kernel;
  if (a.block_table) {
    T_cur = paged_pos(a, b);
    first_blk = T_cur / Bk;
    if (first_blk + (int)blockIdx.x > (T_cur + a.n_new - 1) / Bk) return;   // this sequence touches fewer blocks
    tail_in_kernel = tail_deferred(T_cur, a.n_new, Bk) ? 0 : 1;
  }
  const int blk = first_blk + blockIdx.x;
  const int t_blk0 = blk * Bk;
  // rows of this block in the code / value-metadata / outlier buffers: row_base + t
  const size_t kblk = unit_block(d, a.block_table, a.max_blocks, a.n_blocks, b, h, blk);
  const long long row_base = (long long)(kblk * Bk) - (long long)t_blk0;
  const int t_end = T_cur + a.n_new;
  const int t_lo = max(t_blk0, T_cur);
  const int t_hi = min(t_blk0 + Bk, t_end);
  const int nv = t_hi - t_lo;                      // new tokens in this block, >= 1
  const bool complete = t_blk0 + Bk <= t_end;
  const float Lf = (float)((1 << BITS) - 1);
  constexpr int vpr = D / 8;                       // 16-byte vectors per row
  __half* tail = a.k_tail + (size_t)bh * Bk * D;

  if (isK && !complete) {
    // unfinished block: keep the new keys as fp16 rows t % Bk of the tail
    if (tail_in_kernel && a.phase != 2) {
      for (int i = tid; i < nv * vpr; i += kThreads) {
        const int r = i / vpr, c = i % vpr;
        const int t = t_lo + r;
        reinterpret_cast<uint4*>(tail + (size_t)(t - t_blk0) * D)[c] = __ldg(
            reinterpret_cast<const uint4*>(a.k_new + ((size_t)bh * a.n_new + (t - T_cur)) * D) + c);
      }
    }
    return;
  }
  const int rows = isK ? Bk : nv;
  const int t_row0 = isK ? t_blk0 : t_lo;          // token of staged row 0

  __half* sX = reinterpret_cast<__half*>(smem);                              // [rows][D], swizzled
  uint32_t* sO = reinterpret_cast<uint32_t*>(sX + Bk * D);                   // [KVQ_MAX_OUTLIERS][Bk]
  float4* sPv = reinterpret_cast<float4*>(sO + Bk * KVQ_MAX_OUTLIERS);       // values: [group][Bk] {-z, 1/s, s}
  float4* sPk = sPv;                                                         // keys: [D/2] {-z0, -z1, 1/s0, 1/s1}
  float* sS = reinterpret_cast<float*>(sPv + Bk * kMaxGroups);               // keys: s per channel [D]
  __half2* sRed = reinterpret_cast<__half2*>(sS + D);                        // keys: [16][D/2] {min | max}
  uint8_t* sQ = reinterpret_cast<uint8_t*>(sRed);                            // after C: outlier codes [n_out][Bk]

  // ---- A. stage rows in shared memory (16-byte vectors, all loads in flight
  // before the first store). Thread: vector c of rows r0, r0 + RPI, ... A row's
  // source is the old tail (keys before T_cur) or the new rows. With 64-token
  // blocks the sources are addressed from two linear bases; with 128-token
  // blocks (every vector slot in use) per-vector addressing measured faster.
  {
    constexpr int kMaxVec = 128 * vpr / kThreads;  // rows <= 128
    constexpr int RPI = kThreads / vpr;            // rows per pass (a multiple of 8)
    const int c = tid % vpr, r0 = tid / vpr;
    uint4 v[kMaxVec];
    if (Bk == 64) {
      const long long new_row0 = (long long)bh * a.n_new + (t_row0 - T_cur);   // new-row index of staged row 0
      const __half* new_base = (isK ? a.k_new : a.v_new) + new_row0 * D;
      const int r_split = isK ? T_cur - t_row0 : 0;  // rows below come from the tail
#pragma unroll
      for (int k = 0; k < kMaxVec; ++k) {
        const int r = r0 + k * RPI;
        if (r < rows) {
          const __half* src = (r < r_split ? tail : new_base) + (size_t)r * D;
          v[k] = __ldg(reinterpret_cast<const uint4*>(src) + c);
        }
      }
    } else {
#pragma unroll
      for (int k = 0; k < kMaxVec; ++k) {
        const int r = r0 + k * RPI;
        if (r < rows) {
          const int t = t_row0 + r;
          const __half* src = isK ? ((t < T_cur) ? tail + (size_t)r * D
                                                 : a.k_new + ((size_t)bh * a.n_new + (t - T_cur)) * D)
                                  : a.v_new + ((size_t)bh * a.n_new + (t - T_cur)) * D;
          v[k] = __ldg(reinterpret_cast<const uint4*>(src) + c);
        }
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(sX + r0 * D) + (c ^ (r0 & 7));   // (r0 + k RPI) & 7 == r0 & 7
#pragma unroll
    for (int k = 0; k < kMaxVec; ++k)
      if (r0 + k * RPI < rows) dst[k * RPI * vpr] = v[k];
  }
  __syncthreads();

  // ---- B. dense-and-sparse split: per row, the n_out largest |x|
  uint32_t* gout_base = (isK ? a.k_outl : a.v_outl) + (size_t)(row_base + t_row0) * n_out;
  const __half nanh = __ushort_as_half((uint16_t)0x7E00u);   // marks outliers for step C
  if (a.phase == 2) {
    // window keys, phase 2: the outliers phase 1 selected (their codes are
    // patched in step C'; the statistics come from the window)
    for (int it = tid; it < n_out * Bk; it += kThreads) {
      const int k = it / Bk, r = it % Bk;
      sO[k * Bk + r] = gout_base[(size_t)r * n_out + k];
    }
  } else if (n_out == 1 && D == 128) {
    // four threads per row, 32 channels (four 16-byte chunks) each. The fp16
    // magnitude bits (x & 0x7FFF) order like |x|, so the largest |x| is an
    // unsigned 16-bit maximum; then the lowest channel holding it.
    const int quarter = tid & 3;
    for (int r0 = 0; r0 < rows; r0 += kThreads / 4) {     // same trip count in every thread
      const int row = r0 + (tid >> 2);
      const bool active = row < rows;                     // the four threads of a row agree
      uint32_t cmax[4] = {0u, 0u, 0u, 0u};               // per chunk, max magnitude in both halves
      if (active) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = reinterpret_cast<const uint4*>(sX + row * D)[(4 * quarter + k) ^ (row & 7)];
          cmax[k] = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                             __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
        }
      }
      uint32_t mx = __vmaxu2(__vmaxu2(cmax[0], cmax[1]), __vmaxu2(cmax[2], cmax[3]));
      mx = max(mx & 0xFFFFu, mx >> 16);
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));  // the row's largest magnitude
      uint32_t c_best = 0xFFFFu;
      if (active) {
        int kc = 4;                                       // first chunk holding it
#pragma unroll
        for (int k = 3; k >= 0; --k) kc = (max(cmax[k] & 0xFFFFu, cmax[k] >> 16) == mx) ? k : kc;
        if (kc < 4) {
          const uint4 v = reinterpret_cast<const uint4*>(sX + row * D)[(4 * quarter + kc) ^ (row & 7)];
          const uint32_t wv[4] = {v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu, v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu};
          int idx = 8;
#pragma unroll
          for (int j = 3; j >= 0; --j) {
            idx = ((wv[j] >> 16) == mx) ? 2 * j + 1 : idx;
            idx = ((wv[j] & 0xFFFFu) == mx) ? 2 * j : idx;
          }
          c_best = 32 * quarter + 8 * kc + idx;
        }
      }
      c_best = min(c_best, __shfl_xor_sync(0xffffffffu, c_best, 1));
      c_best = min(c_best, __shfl_xor_sync(0xffffffffu, c_best, 2));
      if (active && quarter == 0) {
        const uint32_t c = min(c_best, (uint32_t)(D - 1));
        const int off = sw_off(row, D, (int)c);
        const uint32_t e = c | ((uint32_t)hbits(sX[off]) << 16);
        sO[row] = e;
        gout_base[row] = e;
        sX[off] = nanh;
      }
    }
  } else if (n_out > 0) {
    // a warp per row: keys |x| bits (15) above (255 - channel); the max is the
    // largest |x|, lowest channel on ties; keys of distinct channels differ
    const int warp = tid >> 5, lane = tid & 31;
    const int E = D >> 5;                          // elements per lane (2 or 4)
    for (int r = warp; r < rows; r += kThreads / 32) {
      uint32_t key[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = lane * E + e;
        key[e] = (e < E) ? (((uint32_t)(hbits(sX[sw_off(r, D, c)]) & 0x7FFF) << 8) | (uint32_t)(255 - c)) : 0u;
      }
      uint32_t pick[KVQ_MAX_OUTLIERS];
      for (int k = 0; k < n_out; ++k) {
        uint32_t best = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) best = max(best, key[e]);
        best = __reduce_max_sync(0xffffffffu, best);
#pragma unroll
        for (int e = 0; e < 4; ++e) key[e] = (key[e] == best) ? 0u : key[e];
        pick[k] = 255u - (best & 0xFFu);
      }
      __syncwarp();
      if (lane == 0) {
        for (int k = 0; k < n_out; ++k) {
          const uint32_t c = pick[k];
          const uint32_t e = c | ((uint32_t)hbits(sX[sw_off(r, D, (int)c)]) << 16);
          sO[k * Bk + r] = e;
          gout_base[(size_t)r * n_out + k] = e;
        }
        for (int k = 0; k < n_out; ++k) sX[sw_off(r, D, (int)pick[k])] = nanh;
      }
      __syncwarp();
    }
  }
  __syncthreads();

  // ---- C. scale and zero (fp16 min/max skip the NaN-marked outliers)
  if (!isK) {
    const int Gv = d.Gv, ng = d.ng, cpg = Gv / 8;  // 16-byte chunks per group
    const int bk_sh = __ffs(Bk) - 1;
    for (int it = tid; it < (ng << bk_sh); it += kThreads) {
      const int g = it >> bk_sh, r = it & (Bk - 1);   // consecutive threads: consecutive rows
      if (r >= rows) continue;
      const uint4* xr = reinterpret_cast<const uint4*>(sX + r * D);
      __half2 mn2 = __halves2half2(nanh, nanh), mx2 = mn2;
      for (int k = 0; k < cpg; ++k) {
        const uint4 v = xr[(g * cpg + k) ^ (r & 7)];
        const __half2 a0 = *reinterpret_cast<const __half2*>(&v.x), a1 = *reinterpret_cast<const __half2*>(&v.y);
        const __half2 a2 = *reinterpret_cast<const __half2*>(&v.z), a3 = *reinterpret_cast<const __half2*>(&v.w);
        mn2 = __hmin2(mn2, __hmin2(__hmin2(a0, a1), __hmin2(a2, a3)));
        mx2 = __hmax2(mx2, __hmax2(__hmax2(a0, a1), __hmax2(a2, a3)));
      }
      const float mn = fminf(__low2float(mn2), __high2float(mn2));
      const float mx = fmaxf(__low2float(mx2), __high2float(mx2));
      float2 sz;
      const uint32_t packed = LV ? range_zero(mn, mx, !isnan(mn), &sz) : group_params(mn, mx, !isnan(mn), Lf, &sz);
      a.v_meta[(size_t)(row_base + t_row0 + r) * ng + g] = packed;
      // {-z, 1/s, s} (LV: 1/r, r)
      sPv[g * Bk + r] = make_float4(-sz.y, rcp_or_zero(sz.x), sz.x, 0.0f);
    }
  } else if (a.phase == 2) {
    // window keys: min and max of the dense elements of the last
    // window_blocks blocks (this block and the ones before it), from the
    // {min, max} pairs phase 1 stored; +inf / -inf mark a block without dense
    // elements in the channel
    if (tid < D) {
      const int c = tid, cp = c >> 1, hc = c & 1;
      float mn = INFINITY, mx = -INFINITY;
      const int u_lo = blk - a.window_blocks + 1 > 0 ? blk - a.window_blocks + 1 : 0;
      for (int u = u_lo; u <= blk; ++u) {
        const size_t ub = unit_block(d, a.block_table, a.max_blocks, a.n_blocks, b, h, u);
        const uint32_t e = a.k_bstat[ub * D + c];
        mn = fminf(mn, h2f((uint16_t)(e & 0xFFFFu)));
        mx = fmaxf(mx, h2f((uint16_t)(e >> 16)));
      }
      float2 sz;
      const uint32_t packed = group_params(mn, mx, mn <= mx, Lf, &sz);
      a.k_meta[kblk * D + c] = packed;
      float* pk = reinterpret_cast<float*>(&sPk[cp]);
      pk[hc] = -sz.y;
      pk[2 + hc] = rcp_or_zero(sz.x);
      sS[c] = sz.x;
    }
  } else {
    // channel pairs p < D/2, row slices q < S: partial fp16 min/max, then combined
    const int P = D / 2, S = kThreads / P;
    const int p = tid % P, q = tid / P;
    __half2 mn2 = __halves2half2(nanh, nanh), mx2 = mn2;
    const int pc = p >> 2, pw = p & 3;             // 16-byte chunk and half2 within it
    for (int j = q; j < Bk; j += S) {
      const __half2 v = reinterpret_cast<const __half2*>(sX + j * D)[((pc ^ (j & 7)) << 2) + pw];
      mn2 = __hmin2(mn2, v);
      mx2 = __hmax2(mx2, v);
    }
    sRed[(2 * q) * P + p] = mn2;
    sRed[(2 * q + 1) * P + p] = mx2;
    __syncthreads();
    if (tid < D) {
      const int c = tid, cp = c >> 1, hc = c & 1;
      float mn = NAN, mx = NAN;
      for (int qq = 0; qq < S; ++qq) {
        const __half2 a2 = sRed[(2 * qq) * P + cp], b2 = sRed[(2 * qq + 1) * P + cp];
        mn = fminf(mn, hc ? __high2float(a2) : __low2float(a2));
        mx = fmaxf(mx, hc ? __high2float(b2) : __low2float(b2));
      }
      if (a.phase == 1) {
        // window keys, phase 1: the block's dense {min, max} (fp16 values;
        // +inf / -inf when every element of the channel is an outlier)
        const uint16_t lo = isnan(mn) ? (uint16_t)0x7C00u : hbits(__float2half_rn(mn));
        const uint16_t hi = isnan(mn) ? (uint16_t)0xFC00u : hbits(__float2half_rn(mx));
        a.k_bstat[kblk * D + c] = (uint32_t)lo | ((uint32_t)hi << 16);
      } else {
        float2 sz;
        const uint32_t packed = LV ? range_zero(mn, mx, !isnan(mn), &sz) : group_params(mn, mx, !isnan(mn), Lf, &sz);
        a.k_meta[kblk * D + c] = packed;
        float* pk = reinterpret_cast<float*>(&sPk[cp]);
        pk[hc] = -sz.y;
        pk[2 + hc] = rcp_or_zero(sz.x);
        sS[c] = sz.x;
      }
    }
  }
  __syncthreads();
  if (isK && a.phase == 1) return;   // window keys: codes in phase 2

  // ---- C'. codes of the outlier positions, from their stored values
  if (n_out > 0) {
    const int bk_sh = __ffs(Bk) - 1, gv_sh = __ffs(d.Gv) - 1;
    for (int it = tid; it < (n_out << bk_sh); it += kThreads) {
      const int o = it >> bk_sh, r = it & (Bk - 1);
      if (r >= rows) continue;
      const uint32_t ev = sO[o * Bk + r];
      const int c = (int)(ev & 0xFFFFu);
      float z, sc, rc;
      if (isK) {
        z = -reinterpret_cast<const float*>(&sPk[c >> 1])[c & 1];
        rc = reinterpret_cast<const float*>(&sPk[c >> 1])[2 + (c & 1)];
        sc = sS[c];
      } else {
        const float4 vp = sPv[(c >> gv_sh) * Bk + r];
        z = -vp.x;
        rc = vp.y;
        sc = vp.z;
      }
      const float xo = __half2float(__ushort_as_half((uint16_t)(ev >> 16)));
      if constexpr (LV) sQ[o * Bk + r] = (uint8_t)level_code_d<BITS>(__fsub_rn(xo, z), sc, s_mid);
      else sQ[o * Bk + r] = (uint8_t)exact_code<BITS>(xo, z, sc, rc);
      // the staged copy takes the group's zero (an fp16 value): step D then
      // codes it 0, a clean pattern, before the stored code replaces it
      sX[sw_off(r, D, c)] = __float2half_rn(z);
    }
    __syncthreads();
  }

  // ---- D. codes for every element, packed
  {
    constexpr int nch = D / 32;
    const int gv_sh = __ffs(d.Gv) - 1;
    uint8_t* base = isK ? a.k_codes : a.v_codes;
    const int bk_sh = __ffs(Bk) - 1;
    for (int it = tid; it < (nch << bk_sh); it += kThreads) {
      const int ch = it >> bk_sh, r = it & (Bk - 1);  // consecutive threads: consecutive rows
      if (r >= rows) continue;
      uint32_t w[BITS];
      if (isK)
        chunk_codes<BITS, true, LV>(sX, sPv, sPk, sS, sO, sQ, D, Bk, r, ch, 0, n_out, s_mid, w);
      else
        chunk_codes<BITS, false, LV>(sX, sPv, sPk, sS, sO, sQ, D, Bk, r, ch, (ch * 32) >> gv_sh, n_out, s_mid, w);
      uint32_t* dst = reinterpret_cast<uint32_t*>(base + (size_t)(row_base + t_row0 + r) * d.cb) + ch * BITS;
      if constexpr (BITS == 8) {
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
      } else if constexpr (BITS == 4) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
      } else if constexpr (BITS == 2) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
      } else {
#pragma unroll
        for (int b = 0; b < BITS; ++b) dst[b] = w[b];
      }
    }
  }
}

// Keys of the last, unfinished block of a multi-block append whose first block
// read the old tail: written after the main launch so the two never overlap.
// Paged (a.seq_len set): each sequence decides from its own position.
__global__ void tail_copy_kernel(const AppendArgs a, __half* __restrict__ k_tail, const __half* __restrict__ k_new,
                                 int Bk, int D, int n_new, int T_cur, int t_from, int t_to) {
  const int bh = blockIdx.y;
  if (a.seq_len) {
    T_cur = paged_pos(a, bh / a.d.H_kv);
    if (!tail_deferred(T_cur, n_new, Bk)) return;
    t_to = T_cur + n_new;
    t_from = (t_to - 1) / Bk * Bk;
  }
  const int vpr = D / 8;
  const int n = (t_to - t_from) * vpr;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int r = i / vpr, c = i % vpr;
    const int t = t_from + r;
    reinterpret_cast<uint4*>(k_tail + ((size_t)bh * Bk + (t % Bk)) * D)[c] = __ldg(
        reinterpret_cast<const uint4*>(k_new + ((size_t)bh * n_new + (t - T_cur)) * D) + c);
  }
}

size_t append_smem(const Dims& d) {
  return (size_t)d.Bk * d.D * sizeof(__half) + (size_t)d.Bk * KVQ_MAX_OUTLIERS * sizeof(uint32_t) +
         (size_t)d.Bk * kMaxGroups * sizeof(float4) + (size_t)d.D * sizeof(float) +
         (size_t)16 * (d.D / 2) * sizeof(__half2);
}

template <int BITS, int D, bool LV>
cudaError_t launch_bd(const AppendArgs& a, const LvParam<LV>& lp, dim3 grid, size_t smem, cudaStream_t st) {
  // the shared-memory limit is a per-device function attribute: set it once on each device
  static std::atomic<bool> attr_set[kMaxDevices];
  int dev = 0;
  if (current_device(&dev) != KVQ_OK) return cudaErrorInvalidDevice;   // the API checked it first
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    const cudaError_t e =
        cudaFuncSetAttribute(append_kernel<BITS, D, LV>, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  append_kernel<BITS, D, LV><<<grid, kThreads, smem, st>>>(a, lp);
  return cudaGetLastError();
}
// lv_mid: the 2^BITS - 1 midpoints of a level table (host memory), or NULL
template <int BITS>
cudaError_t launch_bits(const AppendArgs& a, dim3 grid, size_t smem, cudaStream_t st, const float* lv_mid) {
  if (lv_mid) {
    LvMid m;
    for (int k = 0; k < 255; ++k) m.mid[k] = k < (1 << BITS) - 1 ? lv_mid[k] : 0.0f;
    return a.d.D == 64 ? launch_bd<BITS, 64, true>(a, m, grid, smem, st) : launch_bd<BITS, 128, true>(a, m, grid, smem, st);
  }
  const NoLv n{0};
  return a.d.D == 64 ? launch_bd<BITS, 64, false>(a, n, grid, smem, st) : launch_bd<BITS, 128, false>(a, n, grid, smem, st);
}

}  // namespace

// Paged append: every sequence's length grows by n_new once its tokens are stored.
__global__ void seq_len_advance_kernel(int32_t* seq_len, int B, int n_new, int T_max) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int t = seq_len[b], hi = T_max - n_new;
  seq_len[b] = (t < 0 ? 0 : (t > hi ? hi : t)) + n_new;   // the position the append used, advanced
}

cudaError_t launch_append(const Dims& d, const kvq_cache& c, const __half* k_new,
                          const __half* v_new, int n_new, cudaStream_t st, const Paged* pg,
                          int window_blocks, uint32_t* k_bstat, const float* lv_mid) {
  AppendArgs a;
  a.d = d;
  a.phase = window_blocks > 0 ? 1 : 0;
  a.window_blocks = window_blocks;
  a.k_bstat = k_bstat;
  a.k_codes = static_cast<uint8_t*>(c.k_codes);
  a.k_meta = static_cast<uint32_t*>(c.k_meta);
  a.k_tail = static_cast<__half*>(c.k_tail);
  a.k_outl = static_cast<uint32_t*>(c.k_outl);
  a.v_codes = static_cast<uint8_t*>(c.v_codes);
  a.v_meta = static_cast<uint32_t*>(c.v_meta);
  a.v_outl = static_cast<uint32_t*>(c.v_outl);
  a.k_new = k_new;
  a.v_new = v_new;
  a.n_new = n_new;
  a.block_table = pg ? pg->block_table : nullptr;
  a.seq_len = pg ? pg->seq_len : nullptr;
  a.max_blocks = pg ? pg->max_blocks : 0;
  a.n_blocks = pg ? pg->n_blocks : 0;

  int blocks_x;
  bool defer_tail;
  int t_from = 0, t_end = 0;
  if (pg) {
    // positions are per sequence on the device: size the grid for the most
    // blocks n_new tokens can touch; the kernels read their own positions
    a.T_cur = 0;
    a.first_blk = 0;
    a.tail_in_kernel = 1;
    blocks_x = (n_new + d.Bk - 2) / d.Bk + 1;
    defer_tail = n_new > 1;
  } else {
    const int T_cur = c.T_cur;
    t_end = T_cur + n_new;
    const int first = T_cur / d.Bk, last = (t_end - 1) / d.Bk;
    defer_tail = tail_deferred(T_cur, n_new, d.Bk);
    a.T_cur = T_cur;
    a.first_blk = first;
    a.tail_in_kernel = defer_tail ? 0 : 1;
    blocks_x = last - first + 1;
    t_from = last * d.Bk;
  }

  const dim3 grid(blocks_x, d.B * d.H_kv, 2);
  const size_t smem = append_smem(d);
  cudaError_t e;
  switch (d.bits) {
    case 2: e = launch_bits<2>(a, grid, smem, st, lv_mid); break;
    case 3: e = launch_bits<3>(a, grid, smem, st, lv_mid); break;
    case 8: e = launch_bits<8>(a, grid, smem, st, lv_mid); break;
    default: e = launch_bits<4>(a, grid, smem, st, lv_mid); break;
  }
  if (e != cudaSuccess) return e;
  if (window_blocks > 0) {
    // window keys, phase 2: every block statistic of phase 1 is stored now
    a.phase = 2;
    const dim3 grid2(blocks_x, d.B * d.H_kv, 1);
    switch (d.bits) {
      case 2: e = launch_bits<2>(a, grid2, smem, st, nullptr); break;
      case 3: e = launch_bits<3>(a, grid2, smem, st, nullptr); break;
      case 8: e = launch_bits<8>(a, grid2, smem, st, nullptr); break;
      default: e = launch_bits<4>(a, grid2, smem, st, nullptr); break;
    }
    if (e != cudaSuccess) return e;
  }
  if (defer_tail) {
    const int rows = pg ? d.Bk - 1 : t_end - t_from;   // paged: at most Bk - 1 unfinished rows
    const int blocks = (rows * (d.D / 8) + 255) / 256;
    tail_copy_kernel<<<dim3(blocks, d.B * d.H_kv), 256, 0, st>>>(a, static_cast<__half*>(c.k_tail), k_new, d.Bk,
                                                                 d.D, n_new, a.T_cur, t_from, t_end);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (pg) {
    seq_len_advance_kernel<<<(d.B + 255) / 256, 256, 0, st>>>(pg->seq_len, d.B, n_new, d.T_max);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace kvq
