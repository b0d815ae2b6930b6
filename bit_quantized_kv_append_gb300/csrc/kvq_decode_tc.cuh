// Tensor-core decode attention for head_dim 128 (sm_103a).
//
// Same method as the CUDA-core kernel in kvq_decode.cuh (KVQuant "Pre-RoPE
// Key Quantization": dequantize, rotate, q . k; Quanto step 3: dequantize at
// read time), arranged so the issue slots go to what cannot be avoided:
//
//  * data: a shared-memory ring per CTA (3 stages of 64-token blocks, 2 of
//    128-token blocks) fed by TMA. Code tiles arrive through 3-D tensor maps
//    with a 64 B (INT4) or 32 B (INT2) swizzle; metadata and outliers as 1-D
//    bulk copies. One thread issues, every thread waits on the stage's
//    mbarrier (bounded; on expiry the CTA drains its copies, writes NaN
//    partials and exits).
//  * work split: warp w owns 16 tokens of every 64-token slice and keeps its
//    own running softmax state; warps meet once per block (stage release)
//    and merge once per split.
//  * q . k (mma.m16n8k16, f16 in, f32 out): A = the queries rotated back to
//    the slice start (rows = the G query heads of this kv head); B = the
//    lane's dequantized, rotated keys. Lane quarter r owns 16 contiguous
//    channels and their RoPE partners (kvq_tc_geom.cuh), so a lane reads its
//    codes with two 64-bit loads, turns them into exact half2 integers with
//    one LOP3 each (magic-number trick), dequantizes with one HFMA2 (s, z
//    halved so the rotation cannot overflow fp16) and rotates with the
//    in-block table R(j), j < 64, read through L1 in fragment order.
//  * softmax: base 2, running (m, l) per warp and head.
//  * outliers, once per block in the preparation (one token per thread): a
//    key outlier's score term (x_out - x_dense) * <q, R(t) e_c> for every
//    head, in fp32, which the warps add to their scores; a value outlier's
//    x_out - x_dense, written back into its list entry in the ring, which the
//    warps scale by p and add into the shared sums with shared atomics.
//  * P . V, transposed (rows = channels, columns = heads): A = value codes as
//    exact fp16 subnormals (q * 2^-24, power-of-two rescale at the flush),
//    B = p*s split into fp16 hi + lo; zero points as sum_t p*z per group.
//  * precise scores (PREC, the caller's KVQ_FLAG_PRECISE_SCORES): the keys are
//    dequantized and rotated in fp32 (the rotation from the fp32 in-block
//    table), and both operands of q . k are split into fp16 hi + lo parts with
//    three mma per product (hi.hi + lo.hi + hi.lo), so the scores carry about
//    22 bits instead of 11; P . V takes p*s as hi + lo as well.
//  * accumulation: the tensor-core accumulators move every kFlush blocks into
//    fp32 shared sums (long accumulations on the tensor core drift low). The
//    shared sums and the value-outlier corrections p*(x_out - x_dense) live
//    in a lazily renormalised frame (factor 2^(m - m_frame)), so a new
//    running max rescales only registers.
#pragma once

#include <cuda.h>

#include "kvq_decode.cuh"
#include "kvq_tc_geom.cuh"

namespace kvq {
namespace tc {

#ifndef KVQ_TC_QK_CHAINS
#define KVQ_TC_QK_CHAINS 1   // accumulator chains per n-tile in q . k (1: first half and partner share one)
#endif
#ifndef KVQ_TC_PV_LO
#define KVQ_TC_PV_LO 0       // 1: B = p*s as fp16 hi + lo (two mma); 0: hi only
#endif
#ifndef KVQ_TC_MINB
#define KVQ_TC_MINB 4        // CTAs per SM the register allocation is held to
#endif

constexpr int kFlush = 8;                   // blocks between P.V accumulator flushes
constexpr float kFrameGap = 64.0f;          // renormalise the shared sums past 2^64

// Ring stages: 3 of 64-token blocks, 2 of 128-token blocks.
__host__ __device__ constexpr int ring_stages(int Bk) { return Bk == 64 ? 3 : 2; }

// Byte offsets of one ring stage (host-computed; stages 1024 B aligned).
struct StageLayout {
  uint32_t kc, vc, km, ko, vm, vo;
  uint32_t code_bytes, km_bytes, outl_bytes, vm_bytes;
  uint32_t stage_bytes, tx_bytes;
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: false if the phase did not complete within kWaitNs of the
// GPU's global timer (time rather than a poll count, so the bound does not
// depend on how long one try_wait suspends the thread); a poll count of 2^26
// caps it as well.
constexpr uint64_t kWaitNs = 1000000000ull;   // one second
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < (1u << 26); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitNs) return false;
  }
  return false;
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint4& a, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}
// (a & mask) | orv in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t orv) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(orv));
  return d;
}
__device__ __forceinline__ float ex2(float x) {   // 2^x, hardware approximation (2 ulp)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Small non-negative integer as float without a conversion instruction.
__device__ __forceinline__ float small_int_f(uint32_t q) {
  return __int_as_float(0x4B000000 | q) - 8388608.0f;
}
__device__ __forceinline__ __half2 as_h2(uint32_t u) {
  __half2 h;
  memcpy(&h, &u, 4);
  return h;
}
__device__ __forceinline__ uint32_t as_u32(__half2 h) {
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}
__device__ __forceinline__ uint32_t ld_s32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint2 ld_s64(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ float ld_h(const uint8_t* p) {
  return __half2float(*reinterpret_cast<const __half*>(p));
}

constexpr uint32_t kMagic = 0x64006400u;      // half2(1024, 1024)
// (1024 + 2^k c) * 2^-k - 1024 * 2^-k = c for k = 2, 4, 6
constexpr uint32_t kQuarter = 0x34003400u, kMinus256 = 0xDC00DC00u;
constexpr uint32_t kSixteenth = 0x2C002C00u, kMinus64 = 0xD400D400u;
constexpr uint32_t kSixtyFourth = 0x24002400u, kMinus16 = 0xCC00CC00u;

__device__ __forceinline__ uint32_t fix1(uint32_t h) { return as_u32(__hsub2(as_h2(h), as_h2(kMagic))); }
__device__ __forceinline__ uint32_t fixk(uint32_t h, uint32_t mul, uint32_t add) {
  return as_u32(__hfma2(as_h2(h), as_h2(mul), as_h2(add)));
}

// Identity rotation in fragment order (RoPE off).
#define KVQ_ROT_ID1 {0x3C003C00u, 0x3C003C00u, 0u, 0u}
#define KVQ_ROT_ID4 KVQ_ROT_ID1, KVQ_ROT_ID1, KVQ_ROT_ID1, KVQ_ROT_ID1
#define KVQ_ROT_ID16 KVQ_ROT_ID4, KVQ_ROT_ID4, KVQ_ROT_ID4, KVQ_ROT_ID4
#define KVQ_ROT_ID64 KVQ_ROT_ID16, KVQ_ROT_ID16, KVQ_ROT_ID16, KVQ_ROT_ID16
#define KVQ_ROT_ID256 KVQ_ROT_ID64, KVQ_ROT_ID64, KVQ_ROT_ID64, KVQ_ROT_ID64
static __device__ const uint4 g_rot_identity[kRotFragQuads] = {KVQ_ROT_ID256, KVQ_ROT_ID256, KVQ_ROT_ID256,
                                                               KVQ_ROT_ID256};
#undef KVQ_ROT_ID1
#undef KVQ_ROT_ID4
#undef KVQ_ROT_ID16
#undef KVQ_ROT_ID64
#undef KVQ_ROT_ID256

// ------------------------------------------------------------------ code tiles
// Byte offset of (row, byte) in a code tile as the TMA swizzle lays it out.
template <int BITS>
__device__ __forceinline__ uint32_t code_off(int row, int byte) {
  if constexpr (BITS == 8) return row * 128 + ((((byte >> 4) ^ (row & 7)) << 4) | (byte & 15));
  else if constexpr (BITS == 4) return row * 64 + ((((byte >> 4) ^ ((row >> 1) & 3)) << 4) | (byte & 15));
  else if constexpr (BITS == 2) return row * 32 + ((((byte >> 4) ^ ((row >> 2) & 1)) << 4) | (byte & 15));
  else return row * 48 + byte;
}
// Code of (row, channel c) in a tile.
template <int BITS>
__device__ __forceinline__ uint32_t tile_code(const uint8_t* tile, int row, int c) {
  const int bit = BITS * c, byte = bit >> 3, sh = bit & 7;
  uint32_t v = (uint32_t)tile[code_off<BITS>(row, byte)] >> sh;
  if (sh + BITS > 8) v |= (uint32_t)tile[code_off<BITS>(row, byte + 1)] << (8 - sh);
  return v & ((1u << BITS) - 1u);
}

// Per-lane byte offsets into the code tiles (row 16 w + tperm(g) for keys,
// 16 w + tperm(2 r) for values; slices and n-tiles add compile-time rows).
// The swizzle term of every row a lane reads depends only on the lane.
struct LaneOff {
  uint32_t kf, kp;      // key: first-half and partner codes
  uint32_t ksh;         // INT3: bit shift of the lane's 48-bit key window
  uint32_t vb, vx;      // value tile: row base and swizzle (chunk c at vb + ((c << 4) ^ vx))
  uint32_t vsh;         // INT3: bit shift of the lane's value codes; INT8: the lane's 16-byte chunk in a 32-byte group
  uint32_t sel0, sel1;  // byte_perm selectors of the lane's value bytes
};

template <int BITS>
__device__ __forceinline__ LaneOff lane_offsets(int w, int g, int r) {
  LaneOff o;
  o.vb = o.vx = 0u;
  o.ksh = o.vsh = o.sel0 = o.sel1 = 0u;
  const int tk = tperm(g), tv = tperm(2 * r);
  const int krow = 16 * w + tk, vrow = 16 * w + tv;
  if constexpr (BITS == 8) {
    // 128-byte rows, 128 B swizzle (16-byte chunk ^ row % 8): first-half
    // channels [16r, 16r + 16) are chunk r, their partners chunk 4 + r
    const int ksw = krow & 7;
    o.kf = 128 * krow + ((r ^ ksw) << 4);
    o.kp = 128 * krow + (((4 + r) ^ ksw) << 4);
    o.vb = 128 * vrow + 4 * (g & 3);
    o.vx = (uint32_t)((vrow & 7) << 4);
    o.vsh = (uint32_t)(g >> 2);
  } else if constexpr (BITS == 4) {
    const int ksw = (tk >> 1) & 3, vsw = (tv >> 1) & 3, bb = 2 * (g & 1);
    o.kf = 64 * krow + (((r >> 1) ^ ksw) << 4) + 8 * (r & 1);
    o.kp = 64 * krow + (((2 + (r >> 1)) ^ ksw) << 4) + 8 * (r & 1);
    o.vb = 64 * vrow + 4 * (g >> 1);
    o.vx = vsw << 4;
    o.sel0 = (uint32_t)(bb | ((bb + 4) << 8));
    o.sel1 = (uint32_t)((bb + 1) | ((bb + 5) << 8));
  } else if constexpr (BITS == 2) {
    const int ksw = (tk >> 2) & 1, vsw = (tv >> 2) & 1, bb = g & 3;
    o.kf = 32 * krow + (ksw << 4) + 4 * r;
    o.kp = 32 * krow + ((1 ^ ksw) << 4) + 4 * r;
    o.vb = 32 * vrow + 4 * (g >> 2);
    o.vx = vsw << 4;
    o.sel0 = (uint32_t)(bb | ((bb + 4) << 8));
  } else {
    o.kf = 48 * krow + 4 * ((6 * r) >> 2);
    o.kp = o.kf + 24;
    o.ksh = 16 * (r & 1);
    o.vb = 48 * vrow + 4 * ((12 * g) >> 5);
    o.vsh = (12 * g) & 31;
  }
  return o;
}

// The lane's raw key code words of one token row (first half, partner).
struct KeyWords {
  uint32_t f[2], p[2];
};
template <int BITS>
__device__ __forceinline__ KeyWords key_words(const uint8_t* kc, const LaneOff& o, int row0) {
  constexpr int CB = 16 * BITS;   // code row bytes for D = 128
  KeyWords k;
  const uint8_t* base = kc + CB * row0;
  if constexpr (BITS == 4) {
    const uint2 f = ld_s64(base + o.kf), p = ld_s64(base + o.kp);
    k.f[0] = f.x;
    k.f[1] = f.y;
    k.p[0] = p.x;
    k.p[1] = p.y;
  } else if constexpr (BITS == 2) {
    k.f[0] = ld_s32(base + o.kf);
    k.p[0] = ld_s32(base + o.kp);
    k.f[1] = k.p[1] = 0u;
  } else {
    k.f[0] = ld_s32(base + o.kf);
    k.f[1] = ld_s32(base + o.kf + 4);
    k.p[0] = ld_s32(base + o.kp);
    k.p[1] = ld_s32(base + o.kp + 4);
  }
  return k;
}

// INT8: exact integer codes (half2) of a word's bytes (0, 1) -> x0 and
// (2, 3) -> x1 (byte b becomes the fp16 1024 + b, then 1024 is taken off).
__device__ __forceinline__ void key_codes8(uint32_t W, uint32_t& x0, uint32_t& x1) {
  x0 = fix1(__byte_perm(W, kMagic, 0x7150u));
  x1 = fix1(__byte_perm(W, kMagic, 0x7352u));
}

// Exact integer codes (half2) of k-step kq's slots (0, 1) -> x0 and (2, 3)
// -> x1 from one half's code words, in kchan order.
template <int BITS>
__device__ __forceinline__ void key_codes(const uint32_t (&wd)[2], uint32_t ksh, int kq, uint32_t& x0,
                                          uint32_t& x1) {
  if constexpr (BITS == 4) {
    uint32_t W = wd[kq >> 1];
    if (kq & 1) W >>= 8;
    x0 = fix1(and_or(W, 0x000F000Fu, kMagic));
    x1 = fixk(and_or(W, 0x00F000F0u, kMagic), kSixteenth, kMinus64);
  } else if constexpr (BITS == 2) {
    uint32_t W = wd[0];
    if (kq >= 2) W >>= 8;
    if ((kq & 1) == 0) {
      x0 = fix1(and_or(W, 0x00030003u, kMagic));
      x1 = fixk(and_or(W, 0x000C000Cu, kMagic), kQuarter, kMinus256);
    } else {
      x0 = fixk(and_or(W, 0x00300030u, kMagic), kSixteenth, kMinus64);
      x1 = fixk(and_or(W, 0x00C000C0u, kMagic), kSixtyFourth, kMinus16);
    }
  } else {
    const uint64_t X = (((uint64_t)wd[1] << 32) | wd[0]) >> ksh;
    const uint32_t t0 = (uint32_t)(X >> (12 * kq)), t1 = (uint32_t)(X >> (12 * kq + 6));
    x0 = fix1(and_or(t0 << 13, 0x00070000u, and_or(t0, 0x7u, kMagic)));
    x1 = fix1(and_or(t1 << 13, 0x00070000u, and_or(t1, 0x7u, kMagic)));
  }
}

// Value codes of the lane's channels 32 c4 + 4 g + {0..3} for the token pair
// (t, t+1), t = 64 sl + 16 w + tperm(2 r) + 8 rp, as fp16 subnormals
// (code << shift) * 2^-24: b[2 m] is channel 32 c4 + 4 g + 2 m, b[2 m + 1] the next.
template <int BITS>
__device__ __forceinline__ void value_pair(const uint8_t* vc, const LaneOff& o, int sl, int rp, int c4,
                                           uint32_t (&b)[4]) {
  if constexpr (BITS == 8) {
    // rows t (even) and t + 1: their swizzles differ in the low bit only
    const uint8_t* p = vc + o.vb + 8192 * sl + 1024 * rp;
    const uint32_t ca = (((2 * c4 + o.vsh) << 4) ^ o.vx);
    const uint32_t A = ld_s32(p + ca), B = ld_s32(p + 128 + (ca ^ 16u));
#pragma unroll
    for (int e = 0; e < 4; ++e) b[e] = __byte_perm(A, B, (uint32_t)(e | ((e + 4) << 8))) & 0x00FF00FFu;
  } else if constexpr (BITS == 4) {
    const uint8_t* p = vc + (o.vb + ((c4 << 4) ^ o.vx)) + 4096 * sl + 512 * rp;
    const uint32_t A = ld_s32(p), B = ld_s32(p + 64);
    const uint32_t x0 = __byte_perm(A, B, o.sel0), x1 = __byte_perm(A, B, o.sel1);
    b[0] = x0 & 0x000F000Fu;
    b[1] = x0 & 0x00F000F0u;
    b[2] = x1 & 0x000F000Fu;
    b[3] = x1 & 0x00F000F0u;
  } else if constexpr (BITS == 2) {
    const uint8_t* p = vc + (o.vb + (((c4 >> 1) << 4) ^ o.vx)) + 2048 * sl + 256 * rp + 8 * (c4 & 1);
    const uint32_t x = __byte_perm(ld_s32(p), ld_s32(p + 32), o.sel0);
    b[0] = x & 0x00030003u;
    b[1] = x & 0x000C000Cu;
    b[2] = x & 0x00300030u;
    b[3] = x & 0x00C000C0u;
  } else {
    const uint8_t* p = vc + o.vb + 3072 * sl + 384 * rp + 12 * c4;
    const uint32_t a0 = ld_s32(p), b0 = ld_s32(p + 48);
    uint32_t a1 = 0u, b1 = 0u;
    if (o.vsh + 12 > 32) {
      a1 = ld_s32(p + 4);
      b1 = ld_s32(p + 52);
    }
    const uint32_t tA = __funnelshift_r(a0, a1, o.vsh) & 0xFFFu, tB = __funnelshift_r(b0, b1, o.vsh) & 0xFFFu;
    const uint32_t x = tA | (tB << 16), x6 = x >> 6;
    b[0] = x & 0x00070007u;
    b[1] = x & 0x00380038u;
    b[2] = x6 & 0x00070007u;
    b[3] = x6 & 0x00380038u;
  }
}
// Level tables: the codes index fp16 levels instead of the uniform grid.
// s_lut[i] = {l[i & (2^BITS - 1)], l[i >> BITS]} for a 2·BITS-bit index i (two
// codes at once; 2, 3 and 4 bits), s_lvh[c] = l[c] (8 bits).
__device__ __forceinline__ uint32_t lv_pair8(const __half* s_lvh, uint32_t lo, uint32_t hi) {
  return as_u32(__halves2half2(s_lvh[lo & 0xFFu], s_lvh[hi & 0xFFu]));
}
// Key operands of k-step kq, slots (0, 1) -> x0 and (2, 3) -> x1, as the
// uniform key_codes<BITS> pairs them, but as fp16 levels.
template <int BITS>
__device__ __forceinline__ void key_codes_lv(const uint32_t (&wd)[2], uint32_t ksh, int kq, const uint32_t* s_lut,
                                             uint32_t& x0, uint32_t& x1) {
  if constexpr (BITS == 4) {
    // slots (0, 2) from byte kq & 1 of the word, (1, 3) from byte (kq & 1) + 2
    const uint32_t W = wd[kq >> 1];
    const int sh = 8 * (kq & 1);   // kq is unrolled: a constant shift
    const uint32_t fa = s_lut[(W >> sh) & 0xFFu], fb = s_lut[(W >> (sh + 16)) & 0xFFu];
    x0 = __byte_perm(fa, fb, 0x5410u);
    x1 = __byte_perm(fa, fb, 0x7632u);
  } else if constexpr (BITS == 2) {
    // slots (0, 1): the codes at bits 2m and 16 + 2m of the word, m = 2 (kq & 1) (x0) and m + 1 (x1)
    const uint32_t W = kq >= 2 ? wd[0] >> 8 : wd[0];
    const int m = 2 * (kq & 1);
    x0 = s_lut[((W >> (2 * m)) & 3u) | ((W >> (2 * m + 14)) & 0xCu)];
    x1 = s_lut[((W >> (2 * m + 2)) & 3u) | ((W >> (2 * m + 16)) & 0xCu)];
  } else {
    // 3 bits: the 6-bit windows t0, t1 hold slots (0, 1) and (2, 3), low code first
    const uint64_t X = (((uint64_t)wd[1] << 32) | wd[0]) >> ksh;
    x0 = s_lut[(uint32_t)(X >> (12 * kq)) & 63u];
    x1 = s_lut[(uint32_t)(X >> (12 * kq + 6)) & 63u];
  }
}
// 8 bits: bytes (0, 1) -> x0, (2, 3) -> x1 as levels (the order of key_codes8).
__device__ __forceinline__ void key_codes8_lv(uint32_t W, const __half* s_lvh, uint32_t& x0, uint32_t& x1) {
  x0 = lv_pair8(s_lvh, W, W >> 8);
  x1 = lv_pair8(s_lvh, W >> 16, W >> 24);
}
// The value A operands of value_pair<BITS> (token t in the low half, t + 1 in
// the high half of b[e], channel 32 c4 + 4 g + e) as fp16 levels; the same
// addresses as value_pair<BITS>.
template <int BITS>
__device__ __forceinline__ void value_pair_lv(const uint8_t* vc, const LaneOff& o, int sl, int rp, int c4, int g,
                                              const uint32_t* s_lut, const __half* s_lvh, uint32_t (&b)[4]) {
  if constexpr (BITS == 4) {
    const int bb = 2 * (g & 1);
    const uint8_t* p = vc + (o.vb + ((c4 << 4) ^ o.vx)) + 4096 * sl + 512 * rp;
    const uint32_t A = ld_s32(p), B = ld_s32(p + 64);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t la = s_lut[(A >> (8 * (bb + h))) & 0xFFu], lb = s_lut[(B >> (8 * (bb + h))) & 0xFFu];
      b[2 * h] = __byte_perm(la, lb, 0x5410u);
      b[2 * h + 1] = __byte_perm(la, lb, 0x7632u);
    }
  } else if constexpr (BITS == 8) {
    const uint8_t* p = vc + o.vb + 8192 * sl + 1024 * rp;
    const uint32_t ca = (((2 * c4 + o.vsh) << 4) ^ o.vx);
    const uint32_t A = ld_s32(p + ca), B = ld_s32(p + 128 + (ca ^ 16u));
#pragma unroll
    for (int e = 0; e < 4; ++e) b[e] = lv_pair8(s_lvh, A >> (8 * e), B >> (8 * e));
  } else if constexpr (BITS == 2) {
    // x: token t's byte in bits 0-7, token t + 1's in bits 16-23 (as value_pair<2>)
    const uint8_t* p = vc + (o.vb + (((c4 >> 1) << 4) ^ o.vx)) + 2048 * sl + 256 * rp + 8 * (c4 & 1);
    const uint32_t x = __byte_perm(ld_s32(p), ld_s32(p + 32), o.sel0);
#pragma unroll
    for (int e = 0; e < 4; ++e) b[e] = s_lut[((x >> (2 * e)) & 3u) | ((x >> (2 * e + 14)) & 0xCu)];
  } else {
    // 3 bits: x = token t's 12-bit window | token t + 1's << 16 (as value_pair<3>)
    const uint8_t* p = vc + o.vb + 3072 * sl + 384 * rp + 12 * c4;
    const uint32_t a0 = ld_s32(p), b0 = ld_s32(p + 48);
    uint32_t a1 = 0u, b1 = 0u;
    if (o.vsh + 12 > 32) {
      a1 = ld_s32(p + 4);
      b1 = ld_s32(p + 52);
    }
    const uint32_t tA = __funnelshift_r(a0, a1, o.vsh) & 0xFFFu, tB = __funnelshift_r(b0, b1, o.vsh) & 0xFFFu;
    const uint32_t x = tA | (tB << 16);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t y = x >> (3 * e);
      b[e] = s_lut[(y & 7u) | ((y >> 13) & 0x38u)];
    }
  }
}

// Power of two that undoes the subnormal encoding of value code b[e] (level
// tables carry their fp16 levels unscaled: 1).
template <int BITS, bool LV = false>
__device__ __forceinline__ float value_scale(int e) {
  if constexpr (LV) return 1.0f;
  else if constexpr (BITS == 8) return 16777216.0f;                             // 2^24
  else if constexpr (BITS == 4) return (e & 1) ? 1048576.0f : 16777216.0f;    // 2^20 : 2^24
  else if constexpr (BITS == 2) return 16777216.0f / (float)(1 << (2 * e));    // 2^(24-2e)
  else return (e & 1) ? 2097152.0f : 16777216.0f;                             // 2^21 : 2^24
}

// PREC: (a, b) as an fp16 pair hi plus the fp16 pair of the remainders lo.
__device__ __forceinline__ void split_hilo(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  hi = as_u32(h);
  lo = as_u32(__floats2half2_rn(a - hf.x, b - hf.y));
}

// PREC: one token's keys of k-step kq in fp32: x = code * s + z (the halved
// fp16 s, z of the slots), rotated by R(j) from the fp32 in-block table
// (`fine`: [pair][Bk] {cos, sin}; NULL: no RoPE), then split into fp16 hi +
// lo B operands. f*/p*: exact half2 codes of the first-half slots (0, 1),
// (2, 3) and of their partners; kf*/kp*: {b0, b1} of the rotated first-half
// and partner keys.
template <int BITS>
__device__ __forceinline__ void prec_keys(const uint32_t (&f)[2], const uint32_t (&p)[2], const uint4& zf,
                                          const uint4& zp, const float2* fine, int Bk, int j, int r, int kq,
                                          uint32_t (&kf_hi)[2], uint32_t (&kf_lo)[2], uint32_t (&kp_hi)[2],
                                          uint32_t (&kp_lo)[2]) {
  const uint32_t sf[2] = {zf.x, zf.y}, zff[2] = {zf.z, zf.w}, sp[2] = {zp.x, zp.y}, zpp[2] = {zp.z, zp.w};
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const float2 cf = __half22float2(as_h2(f[hh])), cp = __half22float2(as_h2(p[hh]));
    const float2 s1 = __half22float2(as_h2(sf[hh])), z1 = __half22float2(as_h2(zff[hh]));
    const float2 s2 = __half22float2(as_h2(sp[hh])), z2 = __half22float2(as_h2(zpp[hh]));
    const float xf[2] = {fmaf(cf.x, s1.x, z1.x), fmaf(cf.y, s1.y, z1.y)};
    const float xp[2] = {fmaf(cp.x, s2.x, z2.x), fmaf(cp.y, s2.y, z2.y)};
    float kf[2], kp[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float2 cs = fine ? __ldg(fine + (size_t)kchan<BITS>(r, kq, 2 * hh + e) * Bk + j) : make_float2(1.0f, 0.0f);
      kf[e] = fmaf(xf[e], cs.x, -xp[e] * cs.y);
      kp[e] = fmaf(xp[e], cs.x, xf[e] * cs.y);
    }
    split_hilo(kf[0], kf[1], kf_hi[hh], kf_lo[hh]);
    split_hilo(kp[0], kp[1], kp_hi[hh], kp_lo[hh]);
  }
}

// Float offset in s_acc[w][mt][g][r'] (a float4 per lane) of channel c, head h.
template <int RQ>
__device__ __forceinline__ int acc_index(int w, int c, int h) {
  const int mt = 2 * (c >> 5) + ((c >> 1) & 1), gg = (c >> 2) & 7;
  return ((((w * 8 + mt) * 8 + gg) * RQ + (h >> 1)) << 2) + 2 * (c & 1) + (h & 1);
}

// ------------------------------------------------------------------ kernel
//   q . k:  D[head][token]   = sum_c A(q)[head][c] B(k)[c][token]
//   P . V:  D[channel][head] = sum_t A(v)[channel][t] B(p*s)[t][head]
// so the score fragment of a lane is exactly its B operand for P . V.
// OUTL: the cache keeps outliers (n_out > 0); without them the outlier code
// is not compiled in. PAGED: a paged, ragged batch (block table, per-sequence
// lengths); the contiguous instantiation holds none of that code.
// MODE 0: fp16-operand scores; 1: precise scores (PREC); 2: codes index the
// level table a.lv (LV, non-uniform codes at 4 bits).
template <int BITS, int G, int SL, bool OUTL, bool PAGED, int MODE>
__global__ void __launch_bounds__(kThreads, KVQ_TC_MINB) decode_tc_kernel(const DecodeArgs a, const StageLayout L,
                                                             const __grid_constant__ CUtensorMap tm_k,
                                                             const __grid_constant__ CUtensorMap tm_v) {
  constexpr bool PREC = MODE == 1;
  constexpr bool LV = MODE == 2;
  constexpr int LVN = (LV && BITS != 8) ? 1 << (2 * BITS) : 1;   // LV: entries of the pair table
  constexpr int HALF = kD / 2;
  constexpr int BK = 64 * SL;
  constexpr int NST = ring_stages(BK);
  constexpr int RQ = (G + 1) / 2;     // lane quarters whose columns hold real heads

  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t s_bar[NST];
  __shared__ int s_abort;
  __shared__ float s_qp[G][kD];                               // q at q_pos, times 2*sm_scale*log2(e)
  __shared__ const void* s_src[4];                            // this stream's k_meta, v_meta, k_outl, v_outl
  // q . k A fragments {a0, a2} of 2 q_block, fp16 (a1 = a3 = 0: rows g + 8 are
  // padding heads), double-buffered by block parity; PREC: the lo parts
  __shared__ __align__(16) uint2 s_qa[2][SL][8][32];
  __shared__ __align__(16) uint2 s_ql[PREC ? 2 : 1][PREC ? SL : 1][PREC ? 8 : 1][PREC ? 32 : 1];
  __shared__ __align__(16) uint4 s_kz[2][4][4][2];            // key {s01, s23, z01, z23} / 2 [k-step][quarter][half]
  __shared__ __align__(16) float4 s_acc[kWarps][8][8][RQ];    // P.V sums in the frame m_frame, fragment order
  __shared__ float s_p[OUTL ? kWarps : 1][G][16];            // p * 2^(m - m_frame) for value outliers
  // key outliers: (x_out - x_dense) <q, R(t) e_c> / 2 of every token and head,
  // [block parity][head][token], summed over the token's outliers (fp16 like
  // the scores' operands; binary32 for precise scores)
  using KcT = typename std::conditional<PREC, float, __half>::type;
  __shared__ __align__(16) KcT s_kc[OUTL ? 2 : 1][OUTL ? G : 1][OUTL ? BK : 2];
  __shared__ float s_wm[kWarps][G], s_wl[kWarps][G], s_wf[kWarps][G];
  __shared__ float s_z[kWarps][G][4];                         // zero-point sums per 32-channel block
  __shared__ uint32_t s_lut[LVN];                             // LV: {l[i & M], l[i >> BITS]} fp16, two codes
  __shared__ __half s_lvh[(LV && BITS == 8) ? 256 : 1];       // LV, 8 bits: the fp16 levels
  __shared__ float s_lvf[LV ? 1 << BITS : 1];                 // LV: the levels

  const Dims d = a.d;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g = lane >> 2, r = lane & 3;
  const int bh = blockIdx.y;
  const int b = bh / d.H_kv, hkv = bh % d.H_kv;
  const int split = blockIdx.x;
  // paged: this sequence's full blocks and tail length, read from shared memory per block
  __shared__ int s_ext[PAGED ? 2 : 1];
  const SeqExtent ex = seq_extent(a, b);
  const int units = ex.n_full + (ex.tail_len > 0 ? 1 : 0);
  if (PAGED && tid == 0) {
    s_ext[0] = ex.n_full;
    s_ext[PAGED ? 1 : 0] = ex.tail_len;
  }
  auto n_full_b = [&]() -> int {
    if constexpr (PAGED) return s_ext[0];
    else return a.n_full;
  };
  auto tail_len_b = [&]() -> int {
    if constexpr (PAGED) return s_ext[PAGED ? 1 : 0];
    else return a.tail_len;
  };
  const int u0 = (int)((long long)split * units / a.n_split);
  const int u1 = (int)((long long)(split + 1) * units / a.n_split);
  const int n_out = OUTL ? d.n_out : 0, ng = d.ng;
  const int gv_sh = __ffs(d.Gv) - 1, ng_sh = __ffs(ng) - 1;
  float* ws_base = a.ws + (((size_t)b * a.H_q + hkv * G) * a.S + split) * (kD + 2);
  const LaneOff lo = lane_offsets<BITS>(w, g, r);
  const uint4* rot_tab = a.rope ? reinterpret_cast<const uint4*>(a.rope + rope_frag_off(d)) : g_rot_identity;
  const uint4* rot = rot_tab + rot_frag_index(w, 0, 0, lane);

  uint8_t* ring = dsmem + ((1024u - (smem_addr(dsmem) & 1023u)) & 1023u);
  const uint32_t ring_s = smem_addr(ring);

  // (thread 0) copies of unit u, key block `kblk` (unit_block), into ring
  // stage `stage`; the code maps are [stream][T_max rows] (contiguous) or
  // [block][Bk rows] (paged), the other buffers are indexed by block
  auto unit_blk = [&](int u) -> size_t {
    return unit_block(d, PAGED ? a.block_table : nullptr, a.max_blocks, a.n_blocks, b, hkv, u);
  };
  auto issue = [&](int u, size_t kblk, int stage) {
    const uint32_t bar = smem_addr(&s_bar[stage]);
    const uint32_t base = ring_s + stage * L.stage_bytes;
    const int y = PAGED ? 0 : u * BK, z = PAGED ? (int)kblk : bh;
    mbar_arrive_expect_tx(bar, L.tx_bytes + a.tx_pad);
    tma_load_3d(base + L.kc, &tm_k, 0, y, z, bar);
    tma_load_3d(base + L.vc, &tm_v, 0, y, z, bar);
    bulk_load(base + L.km, static_cast<const uint8_t*>(s_src[0]) + kblk * L.km_bytes, L.km_bytes, bar);
    bulk_load(base + L.vm, static_cast<const uint8_t*>(s_src[1]) + kblk * L.vm_bytes, L.vm_bytes, bar);
    if (n_out > 0) {
      bulk_load(base + L.ko, static_cast<const uint8_t*>(s_src[2]) + kblk * L.outl_bytes, L.outl_bytes, bar);
      bulk_load(base + L.vo, static_cast<const uint8_t*>(s_src[3]) + kblk * L.outl_bytes, L.outl_bytes, bar);
    }
  };
  auto wait_unit = [&](int u) -> bool {
    const int k = u - u0;
    return mbar_wait(smem_addr(&s_bar[k % NST]), (uint32_t)((k / NST) & 1));
  };
  auto abort_split = [&](int u) {
    // report the expired wait in the status word, drain every copy still in
    // flight (bounded waits again), then write NaN partials for this split
    if (tid == 0) atomicOr(a.status, (unsigned int)KVQ_STATUS_TIMEOUT);
    for (int x = u; x < u1 && x < u + NST; ++x) wait_unit(x);
    for (int e = tid; e < G * (kD + 2); e += kThreads)
      ws_base[(size_t)(e / (kD + 2)) * a.S * (kD + 2) + e % (kD + 2)] = __int_as_float(0x7fffffff);
  };

  // ---- per-thread constants of the block preparation
  // queries: thread owns rotate-half pair qi and heads tid/64, tid/64 + 2, ...
  // (one head: threads tid and tid + 64 write the two halves of pair qi)
  const int qi = tid & (HALF - 1);
  constexpr bool q_thread = true;
  uint32_t q_off;
  {
    int rr, kq, s;
    kslot<BITS>(qi, rr, kq, s);
    q_off = (uint32_t)((kq * 32 + rr) * 8 + aslot2_byte(s));   // head 0, first half; + 32 g, + 1024 partner
  }
  // key scale/zero: thread owns channel tid
  uint32_t kz_off;
  {
    int rr, kq, s;
    kslot<BITS>(tid & (HALF - 1), rr, kq, s);
    kz_off = (uint32_t)(((kq * 4 + rr) * 2 + (tid >> 6)) * 16 + slot_byte(s));   // s; z at + 8
  }
  // rotations of pair qi: block start R(t0) from the coarse tables, slice step R(64)
  float2 r64 = make_float2(1.0f, 0.0f);
  if (a.rope && SL > 1 && q_thread) r64 = rope_fine(a.rope, d, 64, qi);
  // R(BK u) = R_hi(u / 256) R_lo(u % 256) from the coarse tables (block index u >= 0)
  constexpr uint32_t kLoOff = HALF * BK, kHiOff = kLoOff + kRopeLo * HALF;
  auto block_rot = [&](int u) -> float2 {
    if (!a.rope || !q_thread) return make_float2(1.0f, 0.0f);
    const uint32_t m = (uint32_t)u;
    const float2 lo = __ldg(a.rope + (kLoOff + ((m & (kRopeLo - 1)) << 6) + qi));
    const float2 hi = __ldg(a.rope + (kHiOff + ((m / kRopeLo) << 6) + qi));
    return rot_compose(hi, lo);
  };

  // Per-block tables shared by the warps: the queries rotated back to each
  // slice start (fp16 A quads, doubled for the halved keys) and the key
  // scale/zero (halved, fragment order).
  auto prep = [&](int u, int stage, float2 rr) {
    const int buf = (u - u0) & 1;
    uint8_t* st = ring + stage * L.stage_bytes;
    if (q_thread) {
#pragma unroll
      for (int sl = 0; sl < SL; ++sl) {
        const float2 rs = sl ? rot_compose(rr, r64) : rr;
        uint8_t* qa = reinterpret_cast<uint8_t*>(&s_qa[buf][sl][0][0]) + q_off;
        uint8_t* ql = reinterpret_cast<uint8_t*>(&s_ql[PREC ? buf : 0][PREC ? sl : 0][0][0]) + q_off;
        // fp16 value of v (PREC: hi, and the lo part v - hi)
        auto put = [&](int off, float v) {
          const __half hi = __float2half_rn(v);
          *reinterpret_cast<__half*>(qa + off) = hi;
          if constexpr (PREC) *reinterpret_cast<__half*>(ql + off) = __float2half_rn(v - __half2float(hi));
        };
        if constexpr (G == 1) {
          const float x = s_qp[0][qi], y = s_qp[0][qi + HALF];
          const bool part = tid >= HALF;
          const float v = part ? fmaf(y, rs.x, -x * rs.y) : fmaf(x, rs.x, y * rs.y);   // apply R(-t)
          put(part ? 1024 : 0, v);
        } else {
#pragma unroll
          for (int gg = tid >> 6; gg < G; gg += 2) {
            const float x = s_qp[gg][qi], y = s_qp[gg][qi + HALF];
            const float x2 = fmaf(x, rs.x, y * rs.y), y2 = fmaf(y, rs.x, -x * rs.y);   // apply R(-t)
            put(32 * gg, x2);
            put(32 * gg + 1024, y2);
          }
        }
      }
    }
    const bool tail = (u == n_full_b());
    if (!tail) {
      const uint32_t m = reinterpret_cast<const uint32_t*>(st + L.km)[tid];
      const uint32_t mh = as_u32(__hmul2(as_h2(m), __float2half2_rn(0.5f)));
      uint8_t* kz = reinterpret_cast<uint8_t*>(&s_kz[buf][0][0][0]) + kz_off;
      *reinterpret_cast<uint16_t*>(kz) = (uint16_t)(mh & 0xFFFFu);
      *reinterpret_cast<uint16_t*>(kz + 8) = (uint16_t)(mh >> 16);
    }
    // Outliers of the block, one token per thread (keys, then values): a key
    // outlier's score term (x_out - x_dense) <q, R(t) e_c> for every head, in
    // fp32 from the unrotated queries and R(t) = R(BK u) R(j) of its channel
    // pair; a value outlier's x_out - x_dense goes back into its list entry in
    // the ring (binary32 with the channel in the 7 low mantissa bits).
    if constexpr (OUTL) {
      const int ntok_u = tail ? tail_len_b() : BK;
      for (int e2 = tid; e2 < 2 * BK; e2 += kThreads) {
        const bool val = e2 >= BK;
        const int tok = val ? e2 - BK : e2;
        if (!val) {
          if (tail) continue;
          const uint32_t* ko = reinterpret_cast<const uint32_t*>(st + L.ko);
          const uint32_t* km = reinterpret_cast<const uint32_t*>(st + L.km);
          const uint8_t* kc = st + L.kc;
          float corr[G];
#pragma unroll
          for (int h = 0; h < G; ++h) corr[h] = 0.0f;
          for (int oi = 0; oi < n_out; ++oi) {
            const uint32_t e = ko[tok * n_out + oi];
            const int c = (int)(e & (kD - 1)), i = c & (HALF - 1);
            const uint32_t m = km[c];
            const uint32_t qc = tile_code<BITS>(kc, tok, c);
            const float xd = fmaf(LV ? s_lvf[LV ? qc : 0] : small_int_f(qc), h2f((uint16_t)(m & 0xFFFFu)),
                                  h2f((uint16_t)(m >> 16)));
            const float dl = 0.5f * (h2f((uint16_t)(e >> 16)) - xd);   // the scores carry q doubled
            float2 R = make_float2(1.0f, 0.0f);
            if (a.rope) {
              const uint32_t ub = (uint32_t)u;
              const float2 lo = __ldg(a.rope + (kLoOff + ((ub & (kRopeLo - 1)) << 6) + i));
              const float2 hi = __ldg(a.rope + (kHiOff + ((ub / kRopeLo) << 6) + i));
              R = rot_compose(rot_compose(hi, lo), __ldg(a.rope + (size_t)i * BK + tok));
            }
            // R(t) e_c: (cos, sin) on (i, i + D/2) for a first-half channel, (-sin, cos) for its partner
            const bool first = c < HALF;
            const float wy = first ? R.x : -R.y, wz = first ? R.y : R.x;
#pragma unroll
            for (int h = 0; h < G; ++h) corr[h] = fmaf(dl, fmaf(s_qp[h][i], wy, s_qp[h][i + HALF] * wz), corr[h]);
          }
#pragma unroll
          for (int h = 0; h < G; ++h) {
            if constexpr (PREC) s_kc[OUTL ? buf : 0][OUTL ? h : 0][OUTL ? tok : 0] = corr[h];
            else s_kc[OUTL ? buf : 0][OUTL ? h : 0][OUTL ? tok : 0] = __float2half_rn(corr[h]);
          }
        } else if (tok < ntok_u) {
          uint32_t* vo = reinterpret_cast<uint32_t*>(st + L.vo);
          const uint32_t* vm = reinterpret_cast<const uint32_t*>(st + L.vm);
          const uint8_t* vc = st + L.vc;
          for (int oi = 0; oi < n_out; ++oi) {
            const uint32_t e = vo[tok * n_out + oi];
            const int c = (int)(e & (kD - 1));
            const float2 sz = __half22float2(as_h2(vm[(tok << ng_sh) + (c >> gv_sh)]));
            const uint32_t qc = tile_code<BITS>(vc, tok, c);
            const float dv = h2f((uint16_t)(e >> 16)) - fmaf(LV ? s_lvf[LV ? qc : 0] : small_int_f(qc), sz.x, sz.y);
            vo[tok * n_out + oi] = (__float_as_uint(dv) & ~(uint32_t)(kD - 1)) | (uint32_t)c;
          }
        }
      }
    }
  };

  // ---- prologue
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(smem_addr(&s_bar[s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    s_abort = 0;
    s_src[0] = a.k_meta;
    s_src[1] = a.v_meta;
    s_src[2] = a.k_outl;
    s_src[3] = a.v_outl;
  }
  __syncthreads();
  __shared__ size_t s_next_blk;   // paged (thread 0): block of the next unit to issue, looked up a block ahead
  if (tid == 0) {
    for (int k = 0; k < NST && u0 + k < u1; ++k) issue(u0 + k, unit_blk(u0 + k), k);
    if (PAGED && u0 + NST < u1) s_next_blk = unit_blk(u0 + NST);
  }
  for (int e = tid; e < G * HALF; e += kThreads) {
    const int gg = e / HALF, i = e % HALF;
    const __half* qh = a.q + ((size_t)b * a.H_q + hkv * G + gg) * kD;
    float x = __half2float(qh[i]), y = __half2float(qh[i + HALF]);
    if (a.rope) {
      const float2 rr = rot_compose(rope_block(a.rope, d, ex.q_pos / BK, i), rope_fine(a.rope, d, ex.q_pos % BK, i));
      const float x2 = fmaf(x, rr.x, -y * rr.y), y2 = fmaf(y, rr.x, x * rr.y);
      x = x2;
      y = y2;
    }
    s_qp[gg][i] = x * (2.0f * a.scale_log2);        // doubled: the keys are halved
    s_qp[gg][i + HALF] = y * (2.0f * a.scale_log2);
  }
  {
    uint32_t* z = reinterpret_cast<uint32_t*>(&s_qa[0][0][0][0]);
    for (int e = tid; e < (int)(sizeof(s_qa) / 4); e += kThreads) z[e] = 0u;
    uint32_t* zl = reinterpret_cast<uint32_t*>(&s_ql[0][0][0][0]);
    for (int e = tid; e < (int)(sizeof(s_ql) / 4); e += kThreads) zl[e] = 0u;
    if constexpr (LV) {
      constexpr int NL = 1 << BITS;
      if constexpr (BITS == 8) {
        for (int e = tid; e < NL; e += kThreads) s_lvh[e] = __float2half_rn(a.lv[e]);
      } else {
        for (int e = tid; e < LVN; e += kThreads)
          s_lut[e] = as_u32(__floats2half2_rn(a.lv[e & (NL - 1)], a.lv[e >> BITS]));
      }
      for (int e = tid; e < NL; e += kThreads) s_lvf[e] = a.lv[e];
    }
    float* f = reinterpret_cast<float*>(&s_acc[0][0][0][0]);
    for (int e = tid; e < (int)(sizeof(s_acc) / 4); e += kThreads) f[e] = 0.0f;
  }
  float o[8][4];     // P.V accumulators: 8 m-tiles of 16 channels x heads (2r, 2r+1)
#pragma unroll
  for (int n = 0; n < 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f;
  float m_frame = -INFINITY, fac = 1.0f;   // s_acc frame of head g; fac = 2^(m_run - m_frame)
  float zacc[4] = {0.f, 0.f, 0.f, 0.f};    // sum_t p z for head g, per 32-channel block
  float2 rr_next = make_float2(1.0f, 0.0f);
  // R(BK) for pair qi: the next block's rotation is composed from this one,
  // re-anchored on the exact table every 32 blocks (drift <= 32 roundings)
  const float2 r_step = (a.rope && q_thread) ? __ldg(a.rope + (kLoOff + (1u << 6) + qi)) : make_float2(1.0f, 0.0f);
  __syncthreads();
  if (u0 < u1) {
    const float2 rr0 = block_rot(u0);
    const bool ok = wait_unit(u0);
    if (__syncthreads_or(!ok)) {
      abort_split(u0);
      return;
    }
    prep(u0, 0, rr0);
    if (u0 + 1 < u1) rr_next = block_rot(u0 + 1);
  }
  __syncthreads();

  // P.V accumulators into the shared sums (frame m_frame), then cleared
  auto flush_o = [&]() {
    const float fa = __shfl_sync(0xffffffffu, fac, 8 * r), fb = __shfl_sync(0xffffffffu, fac, (8 * r + 4) & 31);
    if (r < RQ) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const float v0 = value_scale<BITS, LV>(2 * (mt & 1)), v1 = value_scale<BITS, LV>(2 * (mt & 1) + 1);
        float4 v = s_acc[w][mt][g][r];
        v.x = fmaf(o[mt][0], v0 * fa, v.x);
        v.y = fmaf(o[mt][1], v0 * fb, v.y);
        v.z = fmaf(o[mt][2], v1 * fa, v.z);
        v.w = fmaf(o[mt][3], v1 * fb, v.w);
        s_acc[w][mt][g][r] = v;
      }
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
  };

  int stage = 0;
  uint32_t phase = 0;   // ring stage of block u and the parity of its next fill
  for (int u = u0; u < u1; ++u) {
    const int k = u - u0, buf = k & 1;
    const int nstage = (stage + 1 == NST) ? 0 : stage + 1;
    const uint32_t nphase = phase ^ (nstage == 0 ? 1u : 0u);
    const bool is_tail = (u == n_full_b());
    const int ntok = is_tail ? tail_len_b() : BK;
    const uint8_t* st = ring + stage * L.stage_bytes;
    const uint8_t* kc = st + L.kc;
    const uint8_t* vc = st + L.vc;
    const uint32_t* vm = reinterpret_cast<const uint32_t*>(st + L.vm);
    const uint32_t* vo = reinterpret_cast<const uint32_t*>(st + L.vo);

    // ---- scores of the warp's tokens (rows = heads; column n of n-tile nt
    // is token 64 sl + 16 w + 8 nt + tperm(n))
#pragma unroll 1
    for (int sl = 0; sl < SL; ++sl) {
      float sc[2][2];
      float acc[2][KVQ_TC_QK_CHAINS][4];   // [n-tile][chain]
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int h = 0; h < KVQ_TC_QK_CHAINS; ++h) acc[nt][h][0] = acc[nt][h][1] = acc[nt][h][2] = acc[nt][h][3] = 0.0f;
      if (!is_tail) {
        KeyWords kw[2];
        uint4 k8f[2], k8p[2];   // INT8: the lane's 16 first-half and 16 partner codes of each n-tile
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          if constexpr (BITS == 8) {
            const uint8_t* rowp = kc + 128 * (64 * sl + 8 * nt);
            k8f[nt] = *reinterpret_cast<const uint4*>(rowp + lo.kf);
            k8p[nt] = *reinterpret_cast<const uint4*>(rowp + lo.kp);
          } else {
            kw[nt] = key_words<BITS>(kc, lo, 64 * sl + 8 * nt);
          }
        }
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) {
          const uint2 qf2 = s_qa[buf][sl][kq][lane], qp2 = s_qa[buf][sl][kq + 4][lane];
          const uint4 qf = make_uint4(qf2.x, 0u, qf2.y, 0u), qp = make_uint4(qp2.x, 0u, qp2.y, 0u);
          const uint4 zf = s_kz[buf][kq][r][0], zp = s_kz[buf][kq][r][1];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            uint32_t f0, f1, p0, p1;
            if constexpr (BITS == 8) {
              const uint32_t wf[4] = {k8f[nt].x, k8f[nt].y, k8f[nt].z, k8f[nt].w};
              const uint32_t wp[4] = {k8p[nt].x, k8p[nt].y, k8p[nt].z, k8p[nt].w};
              if constexpr (LV) {
                key_codes8_lv(wf[kq], s_lvh, f0, f1);
                key_codes8_lv(wp[kq], s_lvh, p0, p1);
              } else {
                key_codes8(wf[kq], f0, f1);
                key_codes8(wp[kq], p0, p1);
              }
            } else if constexpr (LV) {
              key_codes_lv<BITS>(kw[nt].f, lo.ksh, kq, s_lut, f0, f1);
              key_codes_lv<BITS>(kw[nt].p, lo.ksh, kq, s_lut, p0, p1);
            } else {
              key_codes<BITS>(kw[nt].f, lo.ksh, kq, f0, f1);
              key_codes<BITS>(kw[nt].p, lo.ksh, kq, p0, p1);
            }
            if constexpr (PREC) {
              const uint2 qfl2 = s_ql[PREC ? buf : 0][PREC ? sl : 0][PREC ? kq : 0][PREC ? lane : 0];
              const uint2 qpl2 = s_ql[PREC ? buf : 0][PREC ? sl : 0][PREC ? kq + 4 : 0][PREC ? lane : 0];
              const uint4 qfl = make_uint4(qfl2.x, 0u, qfl2.y, 0u), qpl = make_uint4(qpl2.x, 0u, qpl2.y, 0u);
              const uint32_t fw[2] = {f0, f1}, pw[2] = {p0, p1};
              uint32_t kfh[2], kfl[2], kph[2], kpl[2];
              prec_keys<BITS>(fw, pw, zf, zp, a.rope, d.Bk, 16 * w + 8 * nt + tperm(g), r, kq, kfh, kfl, kph, kpl);
              mma16816(acc[nt][0], qf, kfh[0], kfh[1]);
              mma16816(acc[nt][0], qfl, kfh[0], kfh[1]);
              mma16816(acc[nt][0], qf, kfl[0], kfl[1]);
              mma16816(acc[nt][KVQ_TC_QK_CHAINS - 1], qp, kph[0], kph[1]);
              mma16816(acc[nt][KVQ_TC_QK_CHAINS - 1], qpl, kph[0], kph[1]);
              mma16816(acc[nt][KVQ_TC_QK_CHAINS - 1], qp, kpl[0], kpl[1]);
            } else {
              const __half2 xf0 = __hfma2(as_h2(f0), as_h2(zf.x), as_h2(zf.z));
              const __half2 xf1 = __hfma2(as_h2(f1), as_h2(zf.y), as_h2(zf.w));
              const __half2 xp0 = __hfma2(as_h2(p0), as_h2(zp.x), as_h2(zp.z));
              const __half2 xp1 = __hfma2(as_h2(p1), as_h2(zp.y), as_h2(zp.w));
              const uint4 rt = __ldg(rot + (nt * 4 + kq) * 32);
              const __half2 c01 = as_h2(rt.x), c23 = as_h2(rt.y), s01 = as_h2(rt.z), s23 = as_h2(rt.w);
              const __half2 kf0 = __hfma2(xf0, c01, __hneg2(__hmul2(xp0, s01)));
              const __half2 kp0 = __hfma2(xp0, c01, __hmul2(xf0, s01));
              const __half2 kf1 = __hfma2(xf1, c23, __hneg2(__hmul2(xp1, s23)));
              const __half2 kp1 = __hfma2(xp1, c23, __hmul2(xf1, s23));
              mma16816(acc[nt][0], qf, as_u32(kf0), as_u32(kf1));
              mma16816(acc[nt][KVQ_TC_QK_CHAINS - 1], qp, as_u32(kp0), as_u32(kp1));
            }
          }
        }
      } else {
        // unfinished block: fp16 keys from K_TAIL (halved), same rotation
        const __half* k_tail = a.k_tail + (size_t)bh * k_tail_stream(d);
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) {
          const uint2 qf2 = s_qa[buf][sl][kq][lane], qp2 = s_qa[buf][sl][kq + 4][lane];
          const uint4 qf = make_uint4(qf2.x, 0u, qf2.y, 0u), qp = make_uint4(qp2.x, 0u, qp2.y, 0u);
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int j = 64 * sl + 16 * w + 8 * nt + tperm(g);
            __half xs[8];
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              const int c = kchan<BITS>(r, kq, s);
              xs[s] = xs[4 + s] = __float2half_rn(0.0f);
              if (j < ntok) {
                xs[s] = __hmul(k_tail[(size_t)j * kD + c], __float2half_rn(0.5f));
                xs[4 + s] = __hmul(k_tail[(size_t)j * kD + c + HALF], __float2half_rn(0.5f));
              }
            }
            if constexpr (PREC) {
              // fp16 keys are exact codes of themselves: s = 1, z = 0 in the fp32 path
              const uint2 qfl2 = s_ql[PREC ? buf : 0][PREC ? sl : 0][PREC ? kq : 0][PREC ? lane : 0];
              const uint2 qpl2 = s_ql[PREC ? buf : 0][PREC ? sl : 0][PREC ? kq + 4 : 0][PREC ? lane : 0];
              const uint4 qfl = make_uint4(qfl2.x, 0u, qfl2.y, 0u), qpl = make_uint4(qpl2.x, 0u, qpl2.y, 0u);
              const uint32_t fw[2] = {as_u32(__halves2half2(xs[0], xs[1])), as_u32(__halves2half2(xs[2], xs[3]))};
              const uint32_t pw[2] = {as_u32(__halves2half2(xs[4], xs[5])), as_u32(__halves2half2(xs[6], xs[7]))};
              const uint4 one = make_uint4(0x3C003C00u, 0x3C003C00u, 0u, 0u);
              uint32_t kfh[2], kfl[2], kph[2], kpl[2];
              prec_keys<BITS>(fw, pw, one, one, a.rope, d.Bk, 16 * w + 8 * nt + tperm(g), r, kq, kfh, kfl, kph, kpl);
              mma16816(acc[nt][0], qf, kfh[0], kfh[1]);
              mma16816(acc[nt][0], qfl, kfh[0], kfh[1]);
              mma16816(acc[nt][0], qf, kfl[0], kfl[1]);
              mma16816(acc[nt][KVQ_TC_QK_CHAINS - 1], qp, kph[0], kph[1]);
              mma16816(acc[nt][KVQ_TC_QK_CHAINS - 1], qpl, kph[0], kph[1]);
              mma16816(acc[nt][KVQ_TC_QK_CHAINS - 1], qp, kpl[0], kpl[1]);
              continue;
            }
            const __half2 xf0 = __halves2half2(xs[0], xs[1]), xf1 = __halves2half2(xs[2], xs[3]);
            const __half2 xp0 = __halves2half2(xs[4], xs[5]), xp1 = __halves2half2(xs[6], xs[7]);
            const uint4 rt = __ldg(rot + (nt * 4 + kq) * 32);
            const __half2 c01 = as_h2(rt.x), c23 = as_h2(rt.y), s01 = as_h2(rt.z), s23 = as_h2(rt.w);
            const __half2 kf0 = __hfma2(xf0, c01, __hneg2(__hmul2(xp0, s01)));
            const __half2 kp0 = __hfma2(xp0, c01, __hmul2(xf0, s01));
            const __half2 kf1 = __hfma2(xf1, c23, __hneg2(__hmul2(xp1, s23)));
            const __half2 kp1 = __hfma2(xp1, c23, __hmul2(xf1, s23));
            mma16816(acc[nt][0], qf, as_u32(kf0), as_u32(kf1));
            mma16816(acc[nt][KVQ_TC_QK_CHAINS - 1], qp, as_u32(kp0), as_u32(kp1));
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sc[nt][0] = acc[nt][0][0];
        sc[nt][1] = acc[nt][0][1];
        if (KVQ_TC_QK_CHAINS > 1) {
          sc[nt][0] += acc[nt][KVQ_TC_QK_CHAINS - 1][0];
          sc[nt][1] += acc[nt][KVQ_TC_QK_CHAINS - 1][1];
        }
      }
      // dense-and-sparse keys: the outliers' score terms of this block
      if (OUTL && n_out > 0 && !is_tail && g < G) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const KcT* kcp = &s_kc[OUTL ? buf : 0][OUTL ? g : 0][OUTL ? 64 * sl + 16 * w + 8 * nt + tperm(2 * r) : 0];
          float2 t2;
          if constexpr (PREC) t2 = *reinterpret_cast<const float2*>(kcp);
          else t2 = __half22float2(*reinterpret_cast<const __half2*>(kcp));
          sc[nt][0] += t2.x;
          sc[nt][1] += t2.y;
        }
      }
      if (is_tail) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            if (64 * sl + 16 * w + 8 * nt + tperm(2 * r + e) >= ntok) sc[nt][e] = -INFINITY;
      }

    // ---- online softmax of this warp's tokens (row g: head g; 4 lanes per row)
    float mb = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) mb = fmaxf(mb, fmaxf(sc[nt][0], sc[nt][1]));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    const float m_new = fmaxf(m_run, mb);
    const float alpha = (m_new == -INFINITY) ? 1.0f : ex2(m_run - m_new);
    float psum = 0.0f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float p = (sc[nt][e] == -INFINITY) ? 0.0f : ex2(sc[nt][e] - m_new);
          sc[nt][e] = p;
          psum += p;
        }
    l_run = fmaf(l_run, alpha, psum);
    m_run = m_new;
    if (__any_sync(0xffffffffu, alpha != 1.0f)) {
      // P.V columns are heads 2r and 2r+1: their factors live in rows 2r, 2r+1
      const float al_a = __shfl_sync(0xffffffffu, alpha, 8 * r);
      const float al_b = __shfl_sync(0xffffffffu, alpha, (8 * r + 4) & 31);
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        o[n][0] *= al_a;
        o[n][1] *= al_b;
        o[n][2] *= al_a;
        o[n][3] *= al_b;
      }
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) zacc[c4] *= alpha;
      if (m_frame == -INFINITY) m_frame = m_run;
      fac = (m_frame == -INFINITY) ? 1.0f : ex2(m_run - m_frame);
      if (__any_sync(0xffffffffu, m_run - m_frame > kFrameGap)) {
        // move the shared sums to the current frame
        const float rf = (m_frame == -INFINITY) ? 1.0f : ex2(m_frame - m_run);
        const float ra = __shfl_sync(0xffffffffu, rf, 8 * r), rb = __shfl_sync(0xffffffffu, rf, (8 * r + 4) & 31);
        __syncwarp();
        if (r < RQ) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            float4 v = s_acc[w][mt][g][r];
            v.x *= ra;
            v.y *= rb;
            v.z *= ra;
            v.w *= rb;
            s_acc[w][mt][g][r] = v;
          }
        }
        __syncwarp();
        m_frame = m_run;
        fac = 1.0f;
      }
    }

    // ---- value outliers: p * (x_out - x_dense) into the shared sums (the
    // prep left x_out - x_dense in the list entries); tokens of the slice that
    // share a channel meet in the shared-memory atomics
    if (OUTL && n_out > 0) {
      if (g < G) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          s_p[OUTL ? w : 0][g][8 * nt + 2 * r] = sc[nt][0] * fac;
          s_p[OUTL ? w : 0][g][8 * nt + 2 * r + 1] = sc[nt][1] * fac;
        }
      }
      __syncwarp();
      const int row = 64 * sl + 16 * w + 8 * ((lane >> 3) & 1) + tperm(lane & 7);
      if (lane < 16 && row < ntok) {
        float* accs = reinterpret_cast<float*>(&s_acc[0][0][0][0]);
        for (int oi = 0; oi < n_out; ++oi) {
          const uint32_t e = vo[row * n_out + oi];
          const int c = (int)(e & (kD - 1));
          const float dv = __uint_as_float(e & ~(uint32_t)(kD - 1));
          const int base = acc_index<RQ>(w, c, 0);
#pragma unroll
          for (int h = 0; h < G; ++h) atomicAdd(accs + base + ((h >> 1) << 2) + (h & 1), s_p[OUTL ? w : 0][h][lane] * dv);
        }
      }
      __syncwarp();
    }

    // ---- P . V: A = value codes (16 channels x 16 tokens), B = p * s (fp16 hi + lo)
    {
      const int tb = 64 * sl + 16 * w + tperm(2 * r);
      const int tt[4] = {tb, tb + 1, tb + 8, tb + 9};
      const float pp[4] = {sc[0][0], sc[0][1], sc[1][0], sc[1][1]};
      uint32_t bh0 = 0u, bh1 = 0u, bl0 = 0u, bl1 = 0u;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int gr = (32 * c4) >> gv_sh;
        if (c4 == 0 || gr != ((32 * (c4 - 1)) >> gv_sh)) {
          float A[4], zs = 0.0f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            A[i] = 0.0f;
            if (!is_tail || tt[i] < ntok) {
              const float2 sz = __half22float2(as_h2(vm[(tt[i] << ng_sh) + gr]));
              A[i] = pp[i] * sz.x;
              zs = fmaf(pp[i], sz.y, zs);
            }
          }
          const __half2 h0 = __floats2half2_rn(A[0], A[1]), h1 = __floats2half2_rn(A[2], A[3]);
          bh0 = (g < G) ? as_u32(h0) : 0u;
          bh1 = (g < G) ? as_u32(h1) : 0u;
          if (KVQ_TC_PV_LO || PREC) {
            const __half2 l0 = __floats2half2_rn(A[0] - __low2float(h0), A[1] - __high2float(h0));
            const __half2 l1 = __floats2half2_rn(A[2] - __low2float(h1), A[3] - __high2float(h1));
            bl0 = (g < G) ? as_u32(l0) : 0u;
            bl1 = (g < G) ? as_u32(l1) : 0u;
          }
          zacc[c4] += zs;
        } else {
          zacc[c4] = zacc[c4 - 1];   // same value group: the two sums stay equal
        }
        uint32_t x0[4], x1[4];
        if constexpr (LV) {
          value_pair_lv<BITS>(vc, lo, sl, 0, c4, g, s_lut, s_lvh, x0);
          value_pair_lv<BITS>(vc, lo, sl, 1, c4, g, s_lut, s_lvh, x1);
        } else {
          value_pair<BITS>(vc, lo, sl, 0, c4, x0);
          value_pair<BITS>(vc, lo, sl, 1, c4, x1);
        }
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          const uint4 av = make_uint4(x0[2 * mi], x0[2 * mi + 1], x1[2 * mi], x1[2 * mi + 1]);
          mma16816(o[2 * c4 + mi], av, bh0, bh1);
          if (KVQ_TC_PV_LO || PREC) mma16816(o[2 * c4 + mi], av, bl0, bl1);
        }
      }
    }

    }  // slices

    // ---- every kFlush blocks move the P.V accumulators into the fp32 sums:
    // the tensor-core accumulation of many small positive products drifts
    // low when one accumulator runs over thousands of tokens
    if ((k + 1) % kFlush == 0) {
      __syncwarp();
      flush_o();
    }

    // ---- next block's tables; release this stage for the refill
    if (u + 1 < u1) {
      if (!mbar_wait(smem_addr(&s_bar[nstage]), nphase)) s_abort = 1;
      prep(u + 1, nstage, rr_next);
      if (u + 2 < u1) rr_next = ((u + 2 - u0) & 31) ? rot_compose(rr_next, r_step) : block_rot(u + 2);
    }
    __syncthreads();
    if (s_abort) {
      abort_split(u + 1);
      return;
    }
    if (tid == 0 && u + NST < u1) {
      // the stage took generic stores (value-outlier entries): order them
      // before the copy engine refills it
      if constexpr (OUTL) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      if constexpr (PAGED) {
        issue(u + NST, s_next_blk, stage);
        if (u + NST + 1 < u1) s_next_blk = unit_blk(u + NST + 1);
      } else {
        issue(u + NST, unit_blk(u + NST), stage);
      }
    }
    stage = nstage;
    phase = nphase;
  }

  // ---- merge the warps
  __syncwarp();
  flush_o();
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) {
    zacc[c4] += __shfl_xor_sync(0xffffffffu, zacc[c4], 1);
    zacc[c4] += __shfl_xor_sync(0xffffffffu, zacc[c4], 2);
  }
  if (g < G && r == 0) {
    s_wm[w][g] = m_run;
    s_wl[w][g] = l_run;
    s_wf[w][g] = (m_frame == -INFINITY) ? 0.0f : ex2(m_frame - m_run);
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) s_z[w][g][c4] = zacc[c4];
  }
  __syncthreads();
  const float* accs = reinterpret_cast<const float*>(&s_acc[0][0][0][0]);
  for (int e = tid; e < G * kD; e += kThreads) {
    const int gg = e / kD, ch = e % kD;
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, s_wm[ww][gg]);
    float sum = 0.0f, lsum = 0.0f;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) {
      const float f = (s_wm[ww][gg] == -INFINITY) ? 0.0f : ex2(s_wm[ww][gg] - M);
      sum = fmaf(f, fmaf(accs[acc_index<RQ>(ww, ch, gg)], s_wf[ww][gg], s_z[ww][gg][ch >> 5]), sum);
      lsum = fmaf(f, s_wl[ww][gg], lsum);
    }
    float* dst = ws_base + (size_t)gg * a.S * (kD + 2);
    dst[ch] = sum;
    if (ch == 0) {
      dst[kD] = M;
      dst[kD + 1] = lsum;
    }
  }
}

}  // namespace tc

template <int BITS, int G, int SL, bool OUTL, bool PAGED, int MODE>
cudaError_t launch_tc(const DecodeArgs& a, const tc::StageLayout& L, const CUtensorMap& tk,
                      const CUtensorMap& tv, size_t smem, cudaStream_t st);
template <int BITS, int G, int SL, bool OUTL, bool PAGED, int MODE>
int tc_occupancy(size_t smem);

}  // namespace kvq
