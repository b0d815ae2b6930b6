// Internal definitions shared by the libkvq translation units (not installed).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq.h"

namespace kvq {

// Shape of one layer's cache as the kernels see it (derived from kvq_config).
struct Dims {
  int B, H_kv, D, T_max, bits, Bk, Gv;
  int n_out;      // outliers per vector
  int cb;         // code row bytes = D*bits/8
  int ng;         // value groups per token = D/Gv
  int n_blk;      // key blocks per stream = T_max/Bk
  int rope_n_hi;  // rows of the coarse RoPE table
  int flags;      // kvq_config.flags (KVQ_FLAG_*)
};

// Strides (elements of the buffer's own unit) of one (b, h_kv) stream.
__host__ __device__ inline size_t k_codes_stream(const Dims& d) { return (size_t)d.T_max * d.cb; }
__host__ __device__ inline size_t k_meta_stream(const Dims& d) { return (size_t)d.n_blk * d.D; }     // uint32 {s,z}
__host__ __device__ inline size_t k_tail_stream(const Dims& d) { return (size_t)d.Bk * d.D; }        // half
__host__ __device__ inline size_t outl_stream(const Dims& d) { return (size_t)d.T_max * d.n_out; }   // uint32 {idx,val}
__host__ __device__ inline size_t v_meta_stream(const Dims& d) { return (size_t)d.T_max * d.ng; }    // uint32 {s,z}

// RoPE table: three float2 {cos, sin} tables of rotate-half frequencies
// w_i = theta^(-2i/D), i < D/2:
//   fine   [D/2][Bk]     angle j * w_i,          j < Bk         (offset in a block)
//   coarse [256][D/2]    angle Bk * m * w_i,     m < 256        (block index, low byte)
//   hi     [n_hi][D/2]   angle 256 * Bk * m * w_i               (block index, high part)
// A position p = Bk * (256 * m_hi + m_lo) + j is R(p) = R_hi(m_hi) R_lo(m_lo) R_fine(j).
constexpr int kRopeLo = 256;
__host__ __device__ inline int rope_n_hi(int n_blk) { return (n_blk - 1) / kRopeLo + 1; }
__host__ __device__ inline size_t rope_fine_off(const Dims&) { return 0; }
__host__ __device__ inline size_t rope_lo_off(const Dims& d) { return (size_t)(d.D / 2) * d.Bk; }
__host__ __device__ inline size_t rope_hi_off(const Dims& d) { return rope_lo_off(d) + (size_t)kRopeLo * (d.D / 2); }
// For D = 128 a fourth table follows (16 B aligned): the in-block rotations of
// the tensor-core kernel in its fragment order, kRopeFragQuads uint4 of fp16
// {cos, cos, sin, sin} (see kvq_tc_geom.cuh).
constexpr int kRopeFragQuads = 1024;
__host__ __device__ inline size_t rope_frag_off(const Dims& d) {
  return (rope_hi_off(d) + (size_t)d.rope_n_hi * (d.D / 2) + 1) & ~(size_t)1;
}
__host__ __device__ inline size_t rope_entries(const Dims& d) {
  return d.D == 128 ? rope_frag_off(d) + 2 * (size_t)kRopeFragQuads
                    : rope_hi_off(d) + (size_t)d.rope_n_hi * (d.D / 2);
}

// Decode split-T scratch: per (b, h_q, split) the partial output o[D], then m, l.
// The workspace starts with the device status word (kWsHeaderBytes, of which
// the first 4 bytes are used); the partials follow.
constexpr int kMaxSplits = 256;
constexpr size_t kWsHeaderBytes = 256;
__host__ __device__ inline int max_splits(const Dims& d) {
  return d.n_blk + 1 < kMaxSplits ? d.n_blk + 1 : kMaxSplits;
}

// Devices the library's per-device tables cover (function attributes,
// occupancies, the allocation-free scratch address): ordinals 0 .. 63. A
// call on a device beyond them is refused with KVQ_ERR_UNSUPPORTED.
constexpr int kMaxDevices = 64;
inline int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return KVQ_ERR_CUDA;
  return (*dev >= 0 && *dev < kMaxDevices) ? KVQ_OK : KVQ_ERR_UNSUPPORTED;
}

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// cos/sin of the composed rotation R(a) R(b) = R(a + b).
__device__ __forceinline__ float2 rot_compose(float2 a, float2 b) {
  return make_float2(__fsub_rn(__fmul_rn(a.x, b.x), __fmul_rn(a.y, b.y)),
                     __fadd_rn(__fmul_rn(a.y, b.x), __fmul_rn(a.x, b.y)));
}

// Paged cache: physical key blocks of Bk tokens shared by the sequences
// through a block table, and per-sequence lengths on the device.
// block_table == nullptr selects the contiguous per-stream layout.
struct Paged {
  const int32_t* block_table = nullptr;  // [B][max_blocks]
  int32_t* seq_len = nullptr;            // [B]
  int max_blocks = 0;                    // T_max / Bk
  int n_blocks = 0;                      // physical blocks in the pools
  int max_len = 0;                       // host upper bound of every seq_len[b]
};

// Block index of key block u of stream (b, h) in the code, metadata and
// outlier buffers, seen as [block][Bk rows] (key metadata: [block][D]).
// Contiguous: (b H_kv + h) n_blk + u; paged: block_table[b][u] H_kv + h, a
// table entry outside [0, n_blocks) clamped so that every access stays inside
// the pools.
__device__ __forceinline__ size_t unit_block(const Dims& d, const int32_t* table, int max_blocks, int n_blocks,
                                             int b, int h, int u) {
  if (table) {
    int p = __ldg(table + (size_t)b * max_blocks + u);
    p = p < 0 ? 0 : (p >= n_blocks ? n_blocks - 1 : p);
    return (size_t)p * d.H_kv + h;
  }
  return ((size_t)b * d.H_kv + h) * d.n_blk + u;
}

// Launch helpers (defined in the kernel translation units).
cudaError_t launch_rope_init(const Dims& d, double theta, float2* tab, cudaStream_t st);
// pg: a paged cache (positions from pg->seq_len, advanced by n_new after the append).
// window_blocks > 0: key statistics over the last window_blocks key blocks,
// with every finished block's dense {min, max} per channel kept in k_bstat
// (the size of K_META). lv_mid: the 2^bits - 1 binary32 midpoints of a level
// table (host memory; non-uniform codes), NULL for the uniform grid.
cudaError_t launch_append(const Dims& d, const kvq_cache& c, const __half* k_new,
                          const __half* v_new, int n_new, cudaStream_t st, const Paged* pg = nullptr,
                          int window_blocks = 0, uint32_t* k_bstat = nullptr, const float* lv_mid = nullptr);
// split_cap > 0 bounds the T splits (and the workspace stride) below max_splits().
// pg: a paged cache (per-sequence lengths; q of sequence b at seq_len[b] - 1).
// ws: the workspace, status word first (kWsHeaderBytes), partials after it.
// tx_pad: diagnostics of the bounded waits (0: none). levels: the 16 levels
// of a non-uniform 4-bit cache (head_dim 128; NULL: uniform codes).
cudaError_t launch_decode(const Dims& d, const kvq_cache& c, const __half* q, int H_q, int q_pos,
                          const float2* rope, float sm_scale, __half* out, float* ws,
                          cudaStream_t st, int split_cap = 0, const Paged* pg = nullptr,
                          uint32_t tx_pad = 0, const float* levels = nullptr);

}  // namespace kvq
