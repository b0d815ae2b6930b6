// Fragment geometry of the tensor-core decode kernel (head_dim 128), shared
// by the kernel and by the RoPE table builder.
//
// q . k runs as mma.m16n8k16 with A = the block-rotated queries (rows = query
// heads) and B = dequantized, rotated keys (columns = 8 tokens of an n-tile).
// Lane (g, r) = (lane >> 2, lane & 3) holds, for the token in column g, the
// four channels of every k-step that sit at k = 2r, 2r+1 (b0) and 2r+8, 2r+9
// (b1). The k -> channel assignment is free as long as A uses the same one;
// it is chosen so that lane quarter r owns the 16 contiguous first-half
// channels [16r, 16r + 16) and their RoPE partners (+ D/2), so one row read
// per half gives a lane all its codes and the rotation never leaves the lane.
#pragma once

#include "kvq_common.cuh"

namespace kvq {
namespace tc {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kD = 128;

// Token of column n (0..7) of an 8-token n-tile, an involution chosen so the
// 64-bit code-row reads of lanes 0-15 and 16-31 fall in distinct banks under
// the 64 B TMA swizzle.
__host__ __device__ constexpr int tperm(int n) { return (n & 1) | ((n & 2) << 1) | ((n & 4) >> 1); }

// First-half channel of lane quarter r, k-step kq (0..3) and fragment slot s
// (0: b0.lo, 1: b0.hi, 2: b1.lo, 3: b1.hi). The slot order follows the order
// in which the magic-number extraction produces half2 pairs of codes.
template <int BITS>
__host__ __device__ constexpr int kchan(int r, int kq, int s) {
  return BITS == 4   ? 16 * r + 8 * (kq >> 1) + 2 * (kq & 1) + (s == 0 ? 0 : s == 1 ? 4 : s == 2 ? 1 : 5)
         : BITS == 2 ? 16 * r + 2 * kq + (s == 0 ? 0 : s == 1 ? 8 : s == 2 ? 1 : 9)
                     : 16 * r + 4 * kq + s;
}

// Inverse of kchan: first-half channel i (0..63) -> (r, kq, s).
template <int BITS>
__host__ __device__ inline void kslot(int i, int& r, int& kq, int& s) {
  r = i >> 4;
  const int o = i & 15;
  if (BITS == 4) {
    const int p = o & 7, bq = (p >> 1) & 1, rest = p - 2 * bq;
    kq = 2 * (o >> 3) + bq;
    s = rest == 0 ? 0 : rest == 4 ? 1 : rest == 1 ? 2 : 3;
  } else if (BITS == 2) {
    const int p = o & 7;
    kq = p >> 1;
    s = 2 * (p & 1) + (o >> 3);
  } else {
    kq = o >> 2;
    s = o & 3;
  }
}

// Byte offset of fragment slot s inside a {x, y, z, w} word quad whose x holds
// slots 0, 1 and y slots 2, 3 (z, w: the same slots of a second quantity).
__host__ __device__ constexpr int slot_byte(int s) { return (s >> 1) * 4 + (s & 1) * 2; }
// Byte offset of slot s inside an mma A quad {a0, a1, a2, a3}: slots 0, 1 in
// a0 (row g, k = 2r, 2r+1), slots 2, 3 in a2 (row g, k = 2r+8, 2r+9).
__host__ __device__ constexpr int aslot_byte(int s) { return (s >> 1) * 8 + (s & 1) * 2; }
// The same inside a pair {a0, a2} (a1 = a3 = 0 left out): slots 0, 1 in a0,
// slots 2, 3 in a2.
__host__ __device__ constexpr int aslot2_byte(int s) { return (s >> 1) * 4 + (s & 1) * 2; }

// In-block rotation table in fragment order, appended to the RoPE table for
// D = 128: uint4 {cos s0|s1, cos s2|s3, sin s0|s1, sin s2|s3} (fp16) of token
// j = 16 w + 8 nt + tperm(g) and channels kchan(r, kq, s), indexed
// [w][nt][kq][lane]. j < 64: slices of 128-token blocks reuse it.
constexpr int kRotFragQuads = kWarps * 2 * 4 * 32;
static_assert(kRotFragQuads == kRopeFragQuads, "RoPE buffer sizing");
__host__ __device__ inline int rot_frag_index(int w, int nt, int kq, int lane) {
  return ((w * 2 + nt) * 4 + kq) * 32 + lane;
}

}  // namespace tc
}  // namespace kvq
