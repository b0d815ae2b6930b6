// Non-uniform codes (KV Cache量化技术介绍, KVQuant "Non-Uniform KV Cache
// Quantization"): the codes of a group index a table of 2^b levels
// 0 = l_0 < l_1 < ... < l_L = 1 on the group's normalized range instead of the
// uniform grid k / L. Per group: z = the dense minimum (fp16, exact; -0 stored
// as +0), r = fp16_round_up(fp32(max) - fp32(min)) in the scale's slot, the
// code of x is the nearest level of u = fp32(fp32(x - z) / r) (the number of
// binary32 midpoints fp32(0.5 (l_k + l_k+1)) below u, ties to the lower
// level), x_hat = z + r * l_code. Groups, outliers, packing and buffers are
// those of the uniform cache.
//
// This file: the plain CUDA-core decode (split-T partials and their combine)
// for the calls the tensor-core kernel's level mode does not take (head_dim
// 64, precise scores). The append is the uniform
// append's kernel in its level-table mode (kvq_append.cu); the fp16 keys of an
// unfinished key block come from K_TAIL here as in the uniform decode.
#include "kvq_levels.cuh"

namespace kvq {
namespace {

constexpr int kLvThreads = 128;

__device__ __forceinline__ float hf(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// Code of channel c in a packed LSB-first row.
__device__ __forceinline__ uint32_t row_code(const uint8_t* row, int c, int bits) {
  const int bit = bits * c;
  uint32_t v = (uint32_t)row[bit >> 3] >> (bit & 7);
  if ((bit & 7) + bits > 8) v |= (uint32_t)row[(bit >> 3) + 1] << (8 - (bit & 7));
  return v & ((1u << bits) - 1u);
}

struct LvDecodeArgs {
  Dims d;
  const __half* k_tail;
  const uint8_t* k_codes;
  const uint32_t* k_meta;
  const uint32_t* k_outl;
  const uint8_t* v_codes;
  const uint32_t* v_meta;
  const uint32_t* v_outl;
  const __half* q;
  const float2* rope;   // NULL: no rotation
  float* ws;
  int T, H_q, q_pos, n_split, S;
  float sm_scale;
};

// cos/sin of position p for pair i from the RoPE table (block part composed
// with the in-block part).
__device__ __forceinline__ float2 rope_at(const float2* rope, const Dims& d, int p, int i) {
  const int half = d.D / 2, m = p / d.Bk, j = p - m * d.Bk;
  const float2 lo = __ldg(rope + rope_lo_off(d) + (size_t)(m % kRopeLo) * half + i);
  const float2 hi = __ldg(rope + rope_hi_off(d) + (size_t)(m / kRopeLo) * half + i);
  const float2 fine = __ldg(rope + rope_fine_off(d) + (size_t)i * d.Bk + j);
  return rot_compose(rot_compose(hi, lo), fine);
}

// Split-T partial attention of the G query heads of one kv head.
template <int G>
__global__ void __launch_bounds__(kLvThreads) decode_levels_kernel(const LvDecodeArgs a, const LevelTable t) {
  __shared__ float s_q[G][128];        // q rotated to q_pos, times sm_scale
  __shared__ float s_p[G][128];        // scores, then probabilities of the block's tokens
  __shared__ float s_m[G], s_l[G], s_alpha[G];
  __shared__ float s_lv[256];
  const Dims d = a.d;
  const int D = d.D, HALF = D / 2, Bk = d.Bk, bits = d.bits, n_out = d.n_out, ng = d.ng;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bh = blockIdx.y, b = bh / d.H_kv, hkv = bh - b * d.H_kv;
  const int split = blockIdx.x;
  const int n_full = a.T / Bk, tail_len = a.T - n_full * Bk;   // the last unit: fp16 keys of K_TAIL
  const int units = n_full + (tail_len > 0 ? 1 : 0);
  const int u0 = (int)((long long)split * units / a.n_split);
  const int u1 = (int)((long long)(split + 1) * units / a.n_split);

  for (int k = tid; k <= t.L; k += kLvThreads) s_lv[k] = t.lv[k];
  for (int e = tid; e < G * HALF; e += kLvThreads) {
    const int g = e / HALF, i = e - g * HALF;
    const __half* qh = a.q + ((size_t)b * a.H_q + hkv * G + g) * D;
    float x = __half2float(qh[i]), y = __half2float(qh[i + HALF]);
    if (a.rope) {
      const float2 r = rope_at(a.rope, d, a.q_pos, i);
      const float x2 = fmaf(x, r.x, -y * r.y), y2 = fmaf(y, r.x, x * r.y);
      x = x2;
      y = y2;
    }
    s_q[g][i] = x * a.sm_scale;
    s_q[g][i + HALF] = y * a.sm_scale;
  }
  if (tid < G) {
    s_m[tid] = -INFINITY;
    s_l[tid] = 0.0f;
  }
  float o[G];
#pragma unroll
  for (int g = 0; g < G; ++g) o[g] = 0.0f;
  __syncthreads();

  const size_t stream_row = (size_t)bh * d.T_max;
  for (int u = u0; u < u1; ++u) {
    const int t0 = u * Bk;
    const bool tail = u == n_full;
    const int ntok = tail ? tail_len : Bk;
    // scores: thread j takes token t0 + j
    for (int j = tid; j < Bk; j += kLvThreads) {
      if (j >= ntok) {
#pragma unroll
        for (int g = 0; g < G; ++g) s_p[g][j] = -INFINITY;
        continue;
      }
      const size_t row = stream_row + t0 + j;
      const __half* kt = a.k_tail + ((size_t)bh * Bk + j) * D;
      const uint8_t* kr = a.k_codes + row * d.cb;
      const uint32_t* km = a.k_meta + ((size_t)bh * d.n_blk + u) * D;
      float acc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) acc[g] = 0.0f;
      for (int i = 0; i < HALF; ++i) {
        float ka, kb;
        if (tail) {                                     // unfinished block: the fp16 keys
          ka = __half2float(kt[i]);
          kb = __half2float(kt[i + HALF]);
        } else {
          const uint32_t ma = __ldg(km + i), mb = __ldg(km + i + HALF);
          ka = fmaf(hf((uint16_t)(ma & 0xFFFFu)), s_lv[row_code(kr, i, bits)], hf((uint16_t)(ma >> 16)));
          kb = fmaf(hf((uint16_t)(mb & 0xFFFFu)), s_lv[row_code(kr, i + HALF, bits)], hf((uint16_t)(mb >> 16)));
        }
        for (int k = 0; k < (tail ? 0 : n_out); ++k) {   // dense-and-sparse: the outlier's own value
          const uint32_t e = __ldg(a.k_outl + row * n_out + k);
          const int c = (int)(e & 0xFFFFu);
          if (c == i) ka = hf((uint16_t)(e >> 16));
          if (c == i + HALF) kb = hf((uint16_t)(e >> 16));
        }
        float ra = ka, rb = kb;
        if (a.rope) {
          const float2 r = rope_at(a.rope, d, t0 + j, i);
          ra = fmaf(ka, r.x, -kb * r.y);
          rb = fmaf(kb, r.x, ka * r.y);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) acc[g] = fmaf(s_q[g][i], ra, fmaf(s_q[g][i + HALF], rb, acc[g]));
      }
#pragma unroll
      for (int g = 0; g < G; ++g) s_p[g][j] = acc[g];
    }
    __syncthreads();
    // online softmax: a warp per head
    for (int g = warp; g < G; g += kLvThreads / 32) {
      float mb = -INFINITY;
      for (int j = lane; j < Bk; j += 32) mb = fmaxf(mb, s_p[g][j]);
      for (int off = 16; off; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
      const float m_new = fmaxf(s_m[g], mb);
      float sum = 0.0f;
      for (int j = lane; j < Bk; j += 32) {
        const float p = expf(s_p[g][j] - m_new);
        s_p[g][j] = p;
        sum += p;
      }
      for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      if (lane == 0) {
        const float alpha = (s_m[g] == -INFINITY) ? 0.0f : expf(s_m[g] - m_new);
        s_alpha[g] = alpha;
        s_l[g] = fmaf(s_l[g], alpha, sum);
        s_m[g] = m_new;
      }
    }
    __syncthreads();
    // values: thread c takes channel c
    if (tid < D) {
      const int c = tid;
#pragma unroll
      for (int g = 0; g < G; ++g) o[g] *= s_alpha[g];
      for (int j = 0; j < ntok; ++j) {
        const size_t row = stream_row + t0 + j;
        const uint32_t m = __ldg(a.v_meta + row * ng + c / d.Gv);
        float v = fmaf(hf((uint16_t)(m & 0xFFFFu)), s_lv[row_code(a.v_codes + row * d.cb, c, bits)],
                       hf((uint16_t)(m >> 16)));
        for (int k = 0; k < n_out; ++k) {
          const uint32_t e = __ldg(a.v_outl + row * n_out + k);
          if ((int)(e & 0xFFFFu) == c) v = hf((uint16_t)(e >> 16));
        }
#pragma unroll
        for (int g = 0; g < G; ++g) o[g] = fmaf(s_p[g][j], v, o[g]);
      }
    }
    __syncthreads();
  }
  // partial (o[D], m, l) of each head for this split
  for (int g = 0; g < G; ++g) {
    float* p = a.ws + (((size_t)b * a.H_q + hkv * G + g) * a.S + split) * (D + 2);
    if (tid < D) p[tid] = o[g];
    if (tid == 0) {
      p[D] = s_m[g];
      p[D + 1] = s_l[g];
    }
  }
}

// out = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s over the splits.
__global__ void combine_levels_kernel(const float* __restrict__ ws, __half* __restrict__ out, int D, int n_split,
                                      int S) {
  const int bhq = blockIdx.x, c = threadIdx.x;
  const float* p = ws + (size_t)bhq * S * (D + 2);
  float M = -INFINITY;
  for (int s = 0; s < n_split; ++s) M = fmaxf(M, p[(size_t)s * (D + 2) + D]);
  float Lsum = 0.0f, acc = 0.0f;
  for (int s = 0; s < n_split; ++s) {
    const float* ps = p + (size_t)s * (D + 2);
    if (ps[D] == -INFINITY) continue;                    // split without tokens
    const float w = expf(ps[D] - M);
    Lsum = fmaf(w, ps[D + 1], Lsum);
    if (c < D) acc = fmaf(w, ps[c], acc);
  }
  if (c < D) out[(size_t)bhq * D + c] = __float2half_rn(Lsum > 0.0f ? acc / Lsum : 0.0f);
}

}  // namespace

cudaError_t launch_decode_levels(const Dims& d, const kvq_cache& c, const __half* q, int H_q, int q_pos,
                                 const float2* rope, float sm_scale, __half* out, float* ws,
                                 const LevelTable& t, cudaStream_t st) {
  LvDecodeArgs a;
  a.d = d;
  a.k_tail = static_cast<const __half*>(c.k_tail);
  a.k_codes = static_cast<const uint8_t*>(c.k_codes);
  a.k_meta = static_cast<const uint32_t*>(c.k_meta);
  a.k_outl = static_cast<const uint32_t*>(c.k_outl);
  a.v_codes = static_cast<const uint8_t*>(c.v_codes);
  a.v_meta = static_cast<const uint32_t*>(c.v_meta);
  a.v_outl = static_cast<const uint32_t*>(c.v_outl);
  a.q = q;
  a.rope = rope;
  ws += kWsHeaderBytes / sizeof(float);   // the partials follow the status word
  a.ws = ws;
  a.T = c.T_cur;
  a.H_q = H_q;
  a.q_pos = q_pos;
  a.S = max_splits(d);
  a.sm_scale = sm_scale;
  int dev = 0, sms = 0;
  if (current_device(&dev) != KVQ_OK) return cudaErrorInvalidDevice;   // the API checked it first
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int units = (a.T + d.Bk - 1) / d.Bk, streams = d.B * d.H_kv;
  int n = (4 * sms + streams - 1) / streams;               // about four CTAs per SM
  if (n > units) n = units;
  if (n > a.S) n = a.S;
  a.n_split = n < 1 ? 1 : n;
  const dim3 grid(a.n_split, streams);
  switch (H_q / d.H_kv) {
    case 1: decode_levels_kernel<1><<<grid, kLvThreads, 0, st>>>(a, t); break;
    case 2: decode_levels_kernel<2><<<grid, kLvThreads, 0, st>>>(a, t); break;
    case 4: decode_levels_kernel<4><<<grid, kLvThreads, 0, st>>>(a, t); break;
    default: decode_levels_kernel<8><<<grid, kLvThreads, 0, st>>>(a, t); break;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  combine_levels_kernel<<<d.B * H_q, 128, 0, st>>>(ws, out, d.D, a.n_split, a.S);
  return cudaGetLastError();
}

}  // namespace kvq
