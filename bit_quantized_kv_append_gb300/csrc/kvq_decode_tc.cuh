// Tensor-core decode attention for head_dim 128 (sm_103a).
//
// Same method as the CUDA-core kernel in kvq_decode.cuh (KVQuant "Pre-RoPE
// Key Quantization": dequantize, rotate, q . k; Quanto step 3: dequantize at
// read time), arranged so the issue slots go to what cannot be avoided:
//
//  * data: a 3-stage shared-memory ring per CTA fed by TMA. Code tiles arrive
//    through 3-D tensor maps with a 64 B (INT4) or 32 B (INT2) swizzle, which
//    makes the row-crossing accesses below bank-conflict free; metadata and
//    outliers arrive as 1-D bulk copies. One thread issues, every thread
//    waits on the stage's mbarrier (bounded; on expiry the CTA drains its
//    copies, writes NaN partials and exits).
//  * work split: warp w owns 16 tokens of every key block (two slices of 16
//    for 128-token blocks) and keeps its own running softmax state; warps
//    meet once per block (stage release) and merge once per split.
//  * q . k: each lane turns its codes into exact half2 integers (magic-number
//    trick), dequantizes (s, z halved so the fp16 rotation cannot overflow),
//    applies the in-block rotation R(j') from registers, and feeds
//    mma.sync.m16n8k16 (f16 in, f32 accumulate) with the block-rotated
//    queries as A (rows = the G query heads of this kv head). The score
//    fragments are already laid out as the A operand of P . V.
//  * softmax: base 2, running (m, l) per warp and head; key outliers add
//    (x_out - x_dense) * <q, R(j') e_c> to their token's score.
//  * P . V, transposed (rows = channels, columns = heads): A = value codes
//    as exact fp16 subnormals (q * 2^-24, rescaled after the loop), B = p*s
//    (value scale folded into the probabilities, split into fp16 hi + lo),
//    the zero points as sum_t p*z per group, value outliers as scattered
//    corrections. Accumulators move to fp32 shared sums every kFlush blocks.
#pragma once

#include <cuda.h>

#include "kvq_decode.cuh"

namespace kvq {
namespace tc {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = 3;
constexpr int kD = 128;
constexpr uint32_t kWaitLimit = 1u << 20;   // mbarrier polls before giving up (~1 s)
constexpr int kFlush = 8;                     // blocks between P.V accumulator flushes

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
// Bounded wait: false if the phase did not complete within kWaitLimit polls.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
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
// D += A * B with A rows 8..15 zero (only the G <= 8 query heads are real).
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
// (a & mask) | orv in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t orv) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(orv));
  return d;
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

constexpr uint32_t kMagic = 0x64006400u;      // half2(1024, 1024)
constexpr uint32_t kSixteenth = 0x2C002C00u;  // half2(1/16, 1/16)
constexpr uint32_t kMinus64 = 0xD400D400u;    // half2(-64, -64)
constexpr uint32_t kHalf = 0x38003800u;       // half2(0.5, 0.5)

// ------------------------------------------------------------------ code layout
// Channel (offset within a 16-channel k-step of the first half) of lane
// quarter r, fragment slot s (0: b0.lo, 1: b0.hi, 2: b1.lo, 3: b1.hi). Chosen
// so each lane extracts its codes from one 32-bit word with a single mask.
template <int BITS>
__host__ __device__ constexpr int chan_off(int r, int s) {
  return BITS == 4   ? 8 * (r >> 1) + 2 * (r & 1) + (s == 0 ? 0 : s == 1 ? 4 : s == 2 ? 1 : 5)
         : BITS == 2 ? 2 * r + (s == 0 ? 0 : s == 1 ? 8 : s == 2 ? 1 : 9)
                     : 4 * r + s;
}
template <int BITS>
__device__ __forceinline__ void chan_slot(int o, int& r, int& s) {
  if (BITS == 4) {
    r = 2 * (o >> 3) + ((o >> 1) & 1);
    const int add = o - 8 * (r >> 1) - 2 * (r & 1);
    s = ((add & 1) << 1) | (add >> 2);
  } else if (BITS == 2) {
    r = (o & 7) >> 1;
    const int add = o - 2 * r;
    s = ((add & 1) << 1) | (add >> 3);
  } else {
    r = o >> 2;
    s = o & 3;
  }
}
// Byte offset of (row, byte) in a code tile as the TMA swizzle lays it out.
template <int BITS>
__device__ __forceinline__ uint32_t code_off(int row, int byte) {
  if constexpr (BITS == 4) return row * 64 + ((((byte >> 4) ^ ((row >> 1) & 3)) << 4) | (byte & 15));
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

// Per-lane byte offsets into the code tiles. For every row a lane reads, the
// TMA swizzle term depends only on the lane's own bits, so each load below is
// a lane offset plus a compile-time immediate.
struct LaneOff {
  uint32_t k[4];        // key tile (INT4: per 16 B chunk; INT2: per half; INT3: [0])
  uint32_t v[4];        // value tile (INT4: per 32-channel block; INT2: per pair; INT3: [0])
  uint32_t ksh, vsh;    // bit shifts of the lane's key / value codes
  uint32_t sel0, sel1;  // byte_perm selectors of the lane's value bytes
};

template <int BITS>
__device__ __forceinline__ LaneOff lane_offsets(int w, int g, int r) {
  LaneOff o;
#pragma unroll
  for (int c = 0; c < 4; ++c) o.k[c] = o.v[c] = 0u;
  o.ksh = o.vsh = o.sel0 = o.sel1 = 0u;
  if constexpr (BITS == 4) {
    const int sw = (g >> 1) & 3, bb = 2 * (g & 1);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      o.k[c] = 1024 * w + 64 * g + ((c ^ sw) << 4) + 4 * (r >> 1);
      o.v[c] = 64 * (16 * w + 2 * r) + ((c ^ r) << 4) + 4 * (g >> 1);
    }
    o.ksh = 8 * (r & 1);
    o.sel0 = (uint32_t)(bb | ((bb + 4) << 8));
    o.sel1 = (uint32_t)((bb + 1) | ((bb + 5) << 8));
  } else if constexpr (BITS == 2) {
    const int sw = (g >> 2) & 1, vsw = (r >> 1) & 1, bb = g & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      o.k[h] = 512 * w + 32 * g + ((h ^ sw) << 4);
      o.v[h] = 32 * (16 * w + 2 * r) + ((h ^ vsw) << 4) + 4 * (g >> 2);
    }
    o.ksh = 4 * r;
    o.sel0 = (uint32_t)(bb | ((bb + 4) << 8));
  } else {
    o.k[0] = 48 * (16 * w + g);
    o.v[0] = 48 * (16 * w + 2 * r) + 4 * ((12 * g) >> 5);
    o.ksh = 12 * r;
    o.vsh = (12 * g) & 31;
  }
  return o;
}

// Exact integer codes of the lane's channels of first-half k-step kq (q[0],
// q[1]) and of their RoPE partners (q[2], q[3]), key row 64 sl + 16 w + 8 nt + g.
template <int BITS>
__device__ __forceinline__ void key_codes(const uint8_t* kc, const LaneOff& o, int sl, int nt, int kq,
                                          uint32_t (&q)[4]) {
  if constexpr (BITS == 4) {
    const int ro = 4096 * sl + 512 * nt + 8 * (kq & 1);
    const uint32_t W[2] = {ld_s32(kc + o.k[kq >> 1] + ro) >> o.ksh, ld_s32(kc + o.k[(kq >> 1) + 2] + ro) >> o.ksh};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      q[2 * h] = as_u32(__hsub2(as_h2(and_or(W[h], 0x000F000Fu, kMagic)), as_h2(kMagic)));
      q[2 * h + 1] = as_u32(__hfma2(as_h2(and_or(W[h], 0x00F000F0u, kMagic)), as_h2(kSixteenth), as_h2(kMinus64)));
    }
  } else if constexpr (BITS == 2) {
    const int ro = 2048 * sl + 256 * nt + 4 * kq;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t W = ld_s32(kc + o.k[h] + ro);
      q[2 * h] = as_u32(__hsub2(as_h2(and_or(W >> o.ksh, 0x00030003u, kMagic)), as_h2(kMagic)));
      q[2 * h + 1] = as_u32(__hsub2(as_h2(and_or(W >> (o.ksh + 2), 0x00030003u, kMagic)), as_h2(kMagic)));
    }
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int bit = 192 * h + 48 * kq;
      const uint8_t* p = kc + o.k[0] + 3072 * sl + 384 * nt + 4 * (bit >> 5);
      const uint64_t v = (uint64_t)ld_s32(p) | ((uint64_t)ld_s32(p + 4) << 32);
      const uint32_t t = (uint32_t)(v >> ((bit & 31) + o.ksh));
      const uint32_t lo = and_or(t << 13, 0x00070000u, and_or(t, 0x7u, kMagic));    // c0 | c1 << 16
      const uint32_t t6 = t >> 6;
      const uint32_t hi = and_or(t6 << 13, 0x00070000u, and_or(t6, 0x7u, kMagic));  // c2 | c3 << 16
      q[2 * h] = as_u32(__hsub2(as_h2(lo), as_h2(kMagic)));
      q[2 * h + 1] = as_u32(__hsub2(as_h2(hi), as_h2(kMagic)));
    }
  }
}

// Value codes of the lane's channels 32 c4 + 4 g + {0..3} for the token pair
// (t, t+1), t = 64 sl + 16 w + 2 r + 8 rp, as fp16 subnormals (code << shift)
// * 2^-24: b[2 m] is channel 32 c4 + 4 g + 2 m, b[2 m + 1] the next channel.
template <int BITS>
__device__ __forceinline__ void value_pair(const uint8_t* vc, const LaneOff& o, int sl, int rp, int c4,
                                           uint32_t (&b)[4]) {
  if constexpr (BITS == 4) {
    const uint8_t* p = vc + o.v[c4] + 4096 * sl + 512 * rp;
    const uint32_t A = ld_s32(p), B = ld_s32(p + 64);
    const uint32_t x0 = __byte_perm(A, B, o.sel0), x1 = __byte_perm(A, B, o.sel1);
    b[0] = x0 & 0x000F000Fu;
    b[1] = x0 & 0x00F000F0u;
    b[2] = x1 & 0x000F000Fu;
    b[3] = x1 & 0x00F000F0u;
  } else if constexpr (BITS == 2) {
    const uint8_t* p = vc + o.v[c4 >> 1] + 2048 * sl + 256 * rp + 8 * (c4 & 1);
    const uint32_t x = __byte_perm(ld_s32(p), ld_s32(p + 32), o.sel0);
    b[0] = x & 0x00030003u;
    b[1] = x & 0x000C000Cu;
    b[2] = x & 0x00300030u;
    b[3] = x & 0x00C000C0u;
  } else {
    const uint8_t* p = vc + o.v[0] + 3072 * sl + 384 * rp + 12 * c4;
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
// Power of two that undoes the subnormal encoding of value code b[e].
template <int BITS>
__device__ __forceinline__ float value_scale(int e) {
  if constexpr (BITS == 4) return (e & 1) ? 1048576.0f : 16777216.0f;         // 2^20 : 2^24
  else if constexpr (BITS == 2) return 16777216.0f / (float)(1 << (2 * e));    // 2^(24-2e)
  else return (e & 1) ? 2097152.0f : 16777216.0f;                             // 2^21 : 2^24
}
__device__ __forceinline__ void mma16816f(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ kernel
// Warp w owns tokens [64 s + 16 w, 64 s + 16 w + 16) of every key block, for
// slices s < SL = BK / 64. Slice s uses the query rotated back by t0 + 64 s,
// so the in-block rotation it still needs is R(j') with j' < 64 (a shared
// table built once). Each warp keeps its own running (m, l, o) per head; the
// warps merge once at the end of the split.
//   q . k:  D[head][token]   = sum_c A(q)[head][c] B(k)[c][token]
//   P . V:  D[channel][head] = sum_t A(v)[channel][t] B(p*s)[t][head]
// so the score fragment of a lane is exactly its B operand for P . V.
template <int BITS, int G, int SL>
__global__ void __launch_bounds__(kThreads) decode_tc_kernel(const DecodeArgs a, const StageLayout L,
                                                             const __grid_constant__ CUtensorMap tm_k,
                                                             const __grid_constant__ CUtensorMap tm_v) {
  constexpr int HALF = kD / 2;
  constexpr int BK = 64 * SL;

  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t s_bar[kStages];
  __shared__ int s_abort;
  __shared__ float s_qp[G][kD];                          // q at q_pos, times sm_scale*log2(e)
  __shared__ __align__(16) uint2 s_qf[2][SL][8][8][4];   // [buf][slice][k-step][row][quarter] {a0, a2}
  __shared__ __align__(16) uint4 s_kp[2][8][4];          // [buf][k-step][quarter] {s01, s23, z01, z23} / 2
  __shared__ __align__(16) float2 s_vsz[2][BK][4];       // value (s, z) per token and group, fp32
  __shared__ __align__(16) uint4 s_rot[kWarps][2][4][32];  // R(j') of each lane's pairs {c, c, s, s}
  __shared__ float4 s_tok[kWarps][16];                   // per-token outlier data of one warp
  __shared__ float s_corr[kWarps][G][kD];                // fp32 P.V sums and value-outlier corrections
  __shared__ float s_z[kWarps][G][4];                    // zero-point sums per 32-channel block
  __shared__ float s_wm[kWarps][G], s_wl[kWarps][G];

  const Dims d = a.d;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g = lane >> 2, r = lane & 3;
  const int bh = blockIdx.y;
  const int b = bh / d.H_kv, hkv = bh % d.H_kv;
  const int split = blockIdx.x;
  const int units = a.n_full + (a.tail_len > 0 ? 1 : 0);
  const int u0 = (int)((long long)split * units / a.n_split);
  const int u1 = (int)((long long)(split + 1) * units / a.n_split);
  const int n_out = d.n_out, ng = d.ng, Gv = d.Gv;
  float* ws_base = a.ws + (((size_t)b * a.H_q + hkv * G) * a.S + split) * (kD + 2);
  const LaneOff lo = lane_offsets<BITS>(w, g, r);

  uint8_t* ring = dsmem + ((1024u - (smem_addr(dsmem) & 1023u)) & 1023u);
  const uint32_t ring_s = smem_addr(ring);

  auto issue = [&](int u, int stage) {
    const uint32_t bar = smem_addr(&s_bar[stage]);
    const uint32_t base = ring_s + stage * L.stage_bytes;
    const int t0 = u * BK;
    mbar_arrive_expect_tx(bar, L.tx_bytes);
    tma_load_3d(base + L.kc, &tm_k, 0, t0, bh, bar);
    tma_load_3d(base + L.vc, &tm_v, 0, t0, bh, bar);
    bulk_load(base + L.km, a.k_meta + ((size_t)bh * d.n_blk + u) * kD, L.km_bytes, bar);
    bulk_load(base + L.vm, a.v_meta + ((size_t)bh * d.T_max + t0) * ng, L.vm_bytes, bar);
    if (n_out > 0) {
      bulk_load(base + L.ko, a.k_outl + ((size_t)bh * d.T_max + t0) * n_out, L.outl_bytes, bar);
      bulk_load(base + L.vo, a.v_outl + ((size_t)bh * d.T_max + t0) * n_out, L.outl_bytes, bar);
    }
  };
  auto wait_unit = [&](int u) -> bool {
    const int k = u - u0;
    return mbar_wait(smem_addr(&s_bar[k % kStages]), (uint32_t)((k / kStages) & 1));
  };
  // Per-block tables shared by the warps: q rotated back to each slice start
  // (fp16, fragment order), the key scale/zero pairs (halved, fragment order)
  // and the value scale/zero per token and group (fp32).
  auto prep = [&](int u) {
    const int buf = (u - u0) & 1;
    const uint8_t* st = ring + ((u - u0) % kStages) * L.stage_bytes;
    for (int e = tid; e < SL * G * HALF; e += kThreads) {
      const int sl = e / (G * HALF), gg = (e / HALF) % G, i = e % HALF;
      float x = s_qp[gg][i], y = s_qp[gg][i + HALF];
      if (a.rope) {
        float2 rr = rope_block(a.rope, d, u, i);                             // R(t0)
        if (sl) rr = rot_compose(rr, rope_fine(a.rope, d, 64 * sl, i));       // R(t0 + 64 sl)
        const float x2 = fmaf(x, rr.x, y * rr.y), y2 = fmaf(y, rr.x, -x * rr.y);   // apply R(-.)
        x = x2;
        y = y2;
      }
      int rq, sq;
      chan_slot<BITS>(i & 15, rq, sq);
      reinterpret_cast<__half*>(&s_qf[buf][sl][i >> 4][gg][rq])[sq] = __float2half_rn(x);
      reinterpret_cast<__half*>(&s_qf[buf][sl][4 + (i >> 4)][gg][rq])[sq] = __float2half_rn(y);
    }
    if (u != a.n_full) {
      const uint32_t* km = reinterpret_cast<const uint32_t*>(st + L.km);
      for (int c = tid; c < kD; c += kThreads) {
        const uint32_t m = km[c];
        const int kq = (c < HALF) ? (c >> 4) : 4 + ((c - HALF) >> 4);
        int rq, sq;
        chan_slot<BITS>(c & 15, rq, sq);
        __half* e = reinterpret_cast<__half*>(&s_kp[buf][kq][rq]);
        e[sq] = __hmul(__ushort_as_half((uint16_t)(m & 0xFFFFu)), __float2half_rn(0.5f));
        e[4 + sq] = __hmul(__ushort_as_half((uint16_t)(m >> 16)), __float2half_rn(0.5f));
      }
    }
    const uint32_t* vm = reinterpret_cast<const uint32_t*>(st + L.vm);
    for (int e = tid; e < BK * ng; e += kThreads) {
      const uint32_t m = vm[e];
      s_vsz[buf][e / ng][e % ng] = make_float2(h2f((uint16_t)(m & 0xFFFFu)), h2f((uint16_t)(m >> 16)));
    }
  };
  auto abort_split = [&](int u) {
    // drain every copy still in flight, then report NaN for this split
    for (int x = u; x < u1 && x < u + kStages; ++x) wait_unit(x);
    for (int e = tid; e < G * (kD + 2); e += kThreads)
      ws_base[(size_t)(e / (kD + 2)) * a.S * (kD + 2) + e % (kD + 2)] = __int_as_float(0x7fffffff);
  };
  // fp16 block-rotated q of head gg at channel c (k-step order), for outlier weights
  auto q_at = [&](int buf, int sl, int gg, int c) -> float {
    int rq, sq;
    chan_slot<BITS>(c & 15, rq, sq);
    const int kq = (c < HALF) ? (c >> 4) : 4 + ((c - HALF) >> 4);
    return __half2float(reinterpret_cast<const __half*>(&s_qf[buf][sl][kq][gg][rq])[sq]);
  };

  // ---- prologue
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_addr(&s_bar[s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    s_abort = 0;
  }
  __syncthreads();
  if (tid == 0)
    for (int k = 0; k < kStages && u0 + k < u1; ++k) issue(u0 + k, k);
  for (int e = tid; e < G * HALF; e += kThreads) {
    const int gg = e / HALF, i = e % HALF;
    const __half* qh = a.q + ((size_t)b * a.H_q + hkv * G + gg) * kD;
    float x = __half2float(qh[i]), y = __half2float(qh[i + HALF]);
    if (a.rope) {
      const float2 rr = rot_compose(rope_block(a.rope, d, a.q_pos / BK, i), rope_fine(a.rope, d, a.q_pos % BK, i));
      const float x2 = fmaf(x, rr.x, -y * rr.y), y2 = fmaf(y, rr.x, x * rr.y);
      x = x2;
      y = y2;
    }
    s_qp[gg][i] = x * a.scale_log2;
    s_qp[gg][i + HALF] = y * a.scale_log2;
  }
  {
    uint32_t* z = reinterpret_cast<uint32_t*>(&s_qf[0][0][0][0][0]);
    for (int e = tid; e < (int)(sizeof(s_qf) / 4); e += kThreads) z[e] = 0u;
    for (int e = tid; e < kWarps * G * kD; e += kThreads) (&s_corr[0][0][0])[e] = 0.0f;
  }
  // in-block rotation R(j'), j' = 16 w + 8 nt + g, of the lane's channel pairs
  if (a.rope) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int j = 16 * w + 8 * nt + g;
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) {
        uint32_t cs[2], sn[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float2 c0 = rope_fine(a.rope, d, j, 16 * kq + chan_off<BITS>(r, 2 * h));
          const float2 c1 = rope_fine(a.rope, d, j, 16 * kq + chan_off<BITS>(r, 2 * h + 1));
          cs[h] = as_u32(__floats2half2_rn(c0.x, c1.x));
          sn[h] = as_u32(__floats2half2_rn(c0.y, c1.y));
        }
        s_rot[w][nt][kq][lane] = make_uint4(cs[0], cs[1], sn[0], sn[1]);
      }
    }
  }
  float o[8][4];     // P.V accumulators: 8 m-tiles of 16 channels x heads (2r, 2r+1)
#pragma unroll
  for (int n = 0; n < 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f;
  float zacc[4] = {0.f, 0.f, 0.f, 0.f};   // sum_t p z for head g, per 32-channel block
  __syncthreads();
  if (u0 < u1) {
    const bool ok = wait_unit(u0);
    if (__syncthreads_or(!ok)) {
      abort_split(u0);
      return;
    }
    prep(u0);
  }
  __syncthreads();

  const __half* k_tail = a.k_tail + (size_t)bh * BK * kD;

  // flush the P.V accumulators into the fp32 sums of heads 2r, 2r+1
  auto flush_o = [&]() {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int head = 2 * r + (e & 1);
        const int ch = 32 * (mt >> 1) + 4 * g + 2 * (mt & 1) + (e >> 1);
        if (head < G) s_corr[w][head][ch] = fmaf(o[mt][e], value_scale<BITS>(2 * (mt & 1) + (e >> 1)), s_corr[w][head][ch]);
        o[mt][e] = 0.0f;
      }
  };

  for (int u = u0; u < u1; ++u) {
    const int k = u - u0, stage = k % kStages, buf = k & 1;
    const bool is_tail = (u == a.n_full);
    const int ntok = is_tail ? a.tail_len : BK;
    const uint8_t* st = ring + stage * L.stage_bytes;
    const uint8_t* kc = st + L.kc;
    const uint8_t* vc = st + L.vc;
    const uint32_t* km = reinterpret_cast<const uint32_t*>(st + L.km);
    const uint32_t* ko = reinterpret_cast<const uint32_t*>(st + L.ko);
    const uint32_t* vo = reinterpret_cast<const uint32_t*>(st + L.vo);

    // ---- scores of the warp's tokens (rows = heads, 2 n-tiles per slice)
    float sc[SL][2][2];
#pragma unroll
    for (int sl = 0; sl < SL; ++sl) {
      // two accumulator chains per n-tile (first-half / partner k-steps)
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) {
        const uint2 qa = s_qf[buf][sl][kq][g][r];
        const uint2 qb = s_qf[buf][sl][kq + 4][g][r];
        uint4 kp = make_uint4(0u, 0u, 0u, 0u), kpp = kp;
        if (!is_tail) {
          kp = s_kp[buf][kq][r];
          kpp = s_kp[buf][kq + 4][r];
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int j = 64 * sl + 16 * w + 8 * nt + g;
          uint32_t kv[4];
          if (!is_tail) {
            uint32_t q[4];
            key_codes<BITS>(kc, lo, sl, nt, kq, q);
            kv[0] = as_u32(__hfma2(as_h2(q[0]), as_h2(kp.x), as_h2(kp.z)));
            kv[1] = as_u32(__hfma2(as_h2(q[1]), as_h2(kp.y), as_h2(kp.w)));
            kv[2] = as_u32(__hfma2(as_h2(q[2]), as_h2(kpp.x), as_h2(kpp.z)));
            kv[3] = as_u32(__hfma2(as_h2(q[3]), as_h2(kpp.y), as_h2(kpp.w)));
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c0 = 16 * kq + chan_off<BITS>(r, 2 * (e & 1)) + HALF * (e >> 1);
              const int c1 = 16 * kq + chan_off<BITS>(r, 2 * (e & 1) + 1) + HALF * (e >> 1);
              __half2 v = __floats2half2_rn(0.f, 0.f);
              if (j < ntok) {
                const __half* row = k_tail + (size_t)j * kD;
                v = __halves2half2(row[c0], row[c1]);
              }
              kv[e] = as_u32(__hmul2(v, as_h2(kHalf)));
            }
          }
          if (a.rope) {
            const uint4 rt = s_rot[w][nt][kq][lane];
            const uint32_t rcs[2] = {rt.x, rt.y}, rsn[2] = {rt.z, rt.w};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const __half2 x = as_h2(kv[h]), y = as_h2(kv[h + 2]);
              const __half2 c = as_h2(rcs[h]), s = as_h2(rsn[h]);
              kv[h] = as_u32(__hfma2(x, c, __hneg2(__hmul2(y, s))));
              kv[h + 2] = as_u32(__hfma2(y, c, __hmul2(x, s)));
            }
          }
          mma16816(acc[nt], qa.x, qa.y, kv[0], kv[1]);
          mma16816(acc2[nt], qb.x, qb.y, kv[2], kv[3]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sc[sl][nt][0] = 2.0f * (acc[nt][0] + acc2[nt][0]);
        sc[sl][nt][1] = 2.0f * (acc[nt][1] + acc2[nt][1]);
      }
      // dense-and-sparse keys: (x_out - x_dense) * <q, R(j') e_c> per outlier
      if (n_out > 0 && !is_tail) {
        for (int oi = 0; oi < n_out; ++oi) {
          if (lane < 16) {
            const int t = 64 * sl + 16 * w + lane;
            const uint32_t e = ko[t * n_out + oi];
            const int c = (int)(e & 0xFFFFu);
            const uint32_t m = km[c];
            const float xd = fmaf((float)tile_code<BITS>(kc, t, c), h2f((uint16_t)(m & 0xFFFFu)),
                                  h2f((uint16_t)(m >> 16)));
            float2 rot = make_float2(1.f, 0.f);
            if (a.rope) rot = rope_fine(a.rope, d, 16 * w + lane, c & (HALF - 1));
            s_tok[w][lane] = make_float4(h2f((uint16_t)(e >> 16)) - xd, __int_as_float(c), rot.x, rot.y);
          }
          __syncwarp();
          if (g < G) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float4 T = s_tok[w][8 * nt + 2 * r + e];
                const int c = __float_as_int(T.y), i = c & (HALF - 1);
                const float qx = q_at(buf, sl, g, i), qy = q_at(buf, sl, g, i + HALF);
                const float wgt = (c < HALF) ? fmaf(qx, T.z, qy * T.w) : fmaf(qy, T.z, -qx * T.w);
                sc[sl][nt][e] = fmaf(T.x, wgt, sc[sl][nt][e]);
              }
            }
          }
          __syncwarp();
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          if (64 * sl + 16 * w + 8 * nt + 2 * r + e >= ntok) sc[sl][nt][e] = -INFINITY;
    }

    // ---- online softmax of this warp's tokens (row g: head g; 4 lanes per row)
    float mb = -INFINITY;
#pragma unroll
    for (int sl = 0; sl < SL; ++sl)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) mb = fmaxf(mb, fmaxf(sc[sl][nt][0], sc[sl][nt][1]));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    const float m_new = fmaxf(m_run, mb);
    const float alpha = (m_new == -INFINITY) ? 1.0f : exp2f(m_run - m_new);
    float psum = 0.0f;
#pragma unroll
    for (int sl = 0; sl < SL; ++sl)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float p = (sc[sl][nt][e] == -INFINITY) ? 0.0f : exp2f(sc[sl][nt][e] - m_new);
          sc[sl][nt][e] = p;
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
      if (g < G)
        for (int c = r; c < kD; c += 4) s_corr[w][g][c] *= alpha;
      __syncwarp();
    }

    // ---- value outliers: p * (x_out - x_dense) into the warp's corrections
    if (n_out > 0) {
#pragma unroll
      for (int sl = 0; sl < SL; ++sl) {
        for (int oi = 0; oi < n_out; ++oi) {
          if (lane < 16) {
            const int t = 64 * sl + 16 * w + lane;
            float4 T = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < ntok) {
              const uint32_t e = vo[t * n_out + oi];
              const int c = (int)(e & 0xFFFFu);
              const float2 sz = s_vsz[buf][t][c / Gv];
              const float xd = fmaf((float)tile_code<BITS>(vc, t, c), sz.x, sz.y);
              T = make_float4(h2f((uint16_t)(e >> 16)) - xd, __int_as_float(c), 0.f, 0.f);
            }
            s_tok[w][lane] = T;
          }
          __syncwarp();
          if (g < G) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float4 T = s_tok[w][8 * nt + 2 * r + e];
                if (T.x != 0.0f) atomicAdd(&s_corr[w][g][__float_as_int(T.y)], sc[sl][nt][e] * T.x);
              }
          }
          __syncwarp();
        }
      }
    }

    // ---- P . V: A = value codes (16 channels x 16 tokens), B = p * s (fp16 hi + lo)
#pragma unroll
    for (int sl = 0; sl < SL; ++sl) {
      const int t0 = 64 * sl + 16 * w + 2 * r;         // tokens t0, t0+1, t0+8, t0+9
      const int tt[4] = {t0, t0 + 1, t0 + 8, t0 + 9};
      const float pp[4] = {sc[sl][0][0], sc[sl][0][1], sc[sl][1][0], sc[sl][1][1]};
      uint32_t bh0 = 0u, bh1 = 0u, bl0 = 0u, bl1 = 0u;
      int cur_gr = -1;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int gr = (32 * c4) / Gv;
        if (gr != cur_gr) {
          cur_gr = gr;
          float A[4], zs = 0.0f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            A[i] = 0.0f;
            if (tt[i] < ntok) {
              const float2 sz = s_vsz[buf][tt[i]][gr];
              A[i] = pp[i] * sz.x;
              zs = fmaf(pp[i], sz.y, zs);
            }
          }
          const __half2 h0 = __floats2half2_rn(A[0], A[1]), h1 = __floats2half2_rn(A[2], A[3]);
          const __half2 l0 = __floats2half2_rn(A[0] - __low2float(h0), A[1] - __high2float(h0));
          const __half2 l1 = __floats2half2_rn(A[2] - __low2float(h1), A[3] - __high2float(h1));
          bh0 = (g < G) ? as_u32(h0) : 0u;
          bh1 = (g < G) ? as_u32(h1) : 0u;
          bl0 = (g < G) ? as_u32(l0) : 0u;
          bl1 = (g < G) ? as_u32(l1) : 0u;
          zacc[c4] += zs;
        } else {
          zacc[c4] = zacc[c4 - 1];   // same value group: the two sums stay equal
        }
        uint32_t x0[4], x1[4];
        value_pair<BITS>(vc, lo, sl, 0, c4, x0);
        value_pair<BITS>(vc, lo, sl, 1, c4, x1);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          mma16816f(o[2 * c4 + mi], x0[2 * mi], x0[2 * mi + 1], x1[2 * mi], x1[2 * mi + 1], bh0, bh1);
          mma16816f(o[2 * c4 + mi], x0[2 * mi], x0[2 * mi + 1], x1[2 * mi], x1[2 * mi + 1], bl0, bl1);
        }
      }
    }

    // ---- every kFlush blocks move the P.V accumulators into the fp32 sums:
    // the tensor-core accumulation of many small positive products drifts
    // low when one accumulator runs over thousands of tokens
    if ((k + 1) % kFlush == 0) {
      __syncwarp();
      flush_o();
    }

    // ---- next block's tables; release this stage for the refill
    if (u + 1 < u1) {
      if (!wait_unit(u + 1)) s_abort = 1;
      prep(u + 1);
    }
    __syncthreads();
    if (s_abort) {
      abort_split(u + 1);
      return;
    }
    if (tid == 0 && u + kStages < u1) issue(u + kStages, stage);
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
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) s_z[w][g][c4] = zacc[c4];
  }
  __syncthreads();
  for (int e = tid; e < G * kD; e += kThreads) {
    const int gg = e / kD, ch = e % kD;
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, s_wm[ww][gg]);
    float sum = 0.0f, lsum = 0.0f;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) {
      const float f = (s_wm[ww][gg] == -INFINITY) ? 0.0f : exp2f(s_wm[ww][gg] - M);
      sum = fmaf(f, s_corr[ww][gg][ch] + s_z[ww][gg][ch >> 5], sum);
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

template <int BITS, int G, int SL>
cudaError_t launch_tc(const DecodeArgs& a, const tc::StageLayout& L, const CUtensorMap& tk,
                      const CUtensorMap& tv, size_t smem, cudaStream_t st);
template <int BITS, int G, int SL>
int tc_occupancy(size_t smem);

}  // namespace kvq
