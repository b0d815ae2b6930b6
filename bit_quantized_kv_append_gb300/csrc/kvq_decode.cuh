// kvq_decode_attn kernels: split-T flash-decode over the packed cache.
//
// KV Cache量化技术介绍 (developer.horizon.auto/blog/13163):
//   KVQuant "Pre-RoPE Key Quantization": keys are dequantized, then rotated
//     to their position before q . k;
//   Quanto step 3 (实时反量化访问): the cache is dequantized in registers at
//     read time, never written back in full precision.
// Partial kernel: one CTA per (T split, (b, h_kv) stream) serves the G query
// heads of that kv head. For every key block of its split it
//   1. rotates the query (already at q_pos) back by the block start t0, so a
//      key at t0 + j only needs the in-block rotation R(j) (two-level tables);
//   2. scores: each thread dequantizes its token's key codes (x = q*s + z with
//      the block's per-channel s, z), rotates pairs (i, i + D/2) by R(j), dots
//      with the G queries; outliers correct the score by
//      (x_out - x_dense) * <q, R(j) e_c>;
//   3. online softmax per head (running max m, sum l, rescale alpha), base 2;
//   4. values: each thread owns a channel pair and accumulates p * x_hat for the
//      G heads, outliers replacing their element.
// It writes (o[D], m, l) per head and split; the combine kernel merges splits
// with weights 2^(m_s - max m).
#pragma once

#include <type_traits>

#include "kvq_common.cuh"

namespace kvq {

constexpr int kDecThreads = 128;

struct DecodeArgs {
  Dims d;
  const uint8_t* k_codes;
  const uint32_t* k_meta;
  const __half* k_tail;
  const uint32_t* k_outl;
  const uint8_t* v_codes;
  const uint32_t* v_meta;
  const uint32_t* v_outl;
  const __half* q;
  const float2* rope;  // NULL: no rotation
  float* ws;
  int T, n_full, tail_len, H_q, q_pos, n_split, S;
  float scale_log2;    // sm_scale * log2(e)
  const int32_t* block_table;  // paged cache (NULL: contiguous streams)
  const int32_t* seq_len;      // paged: tokens of each sequence
  int max_blocks, n_blocks;
  uint32_t* status;            // device status word: KVQ_STATUS_* bits are ORed in
  uint32_t tx_pad;             // diagnostics: bytes each ring stage expects beyond its copies (0)
  float lv[256];               // level table of non-uniform codes (tensor-core mode 2)
};

// Tokens, full key blocks, tail length and query position of sequence b.
struct SeqExtent {
  int T, n_full, tail_len, q_pos;
};
__device__ __forceinline__ SeqExtent seq_extent(const DecodeArgs& a, int b) {
  SeqExtent e;
  if (a.block_table) {
    const int cap = a.max_blocks * a.d.Bk;
    const int t = __ldg(a.seq_len + b);
    e.T = t < 0 ? 0 : (t > cap ? cap : t);
    e.q_pos = e.T > 0 ? e.T - 1 : 0;
  } else {
    e.T = a.T;
    e.q_pos = a.q_pos;
  }
  e.n_full = e.T / a.d.Bk;
  e.tail_len = e.T - e.n_full * a.d.Bk;
  return e;
}

template <int N, int I = 0, typename F>
__device__ __forceinline__ void static_for(F&& f) {
  if constexpr (I < N) {
    f(std::integral_constant<int, I>{});
    static_for<N, I + 1>(f);
  }
}

// Whole code row of one token in registers (CB bytes, CB/4 words).
template <int CB>
struct Row {
  uint32_t w[CB / 4];
  __device__ __forceinline__ void load(const uint8_t* p) {
    if constexpr (CB % 16 == 0) {
#pragma unroll
      for (int k = 0; k < CB / 16; ++k) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p) + k);
        w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < CB / 8; ++k) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(p) + k);
        w[2 * k] = v.x; w[2 * k + 1] = v.y;
      }
    }
  }
  // Code of channel C (compile-time) in the LSB-first bitstream.
  template <int BITS, int C>
  __device__ __forceinline__ uint32_t code() const {
    constexpr int bit = BITS * C, wi = bit >> 5, off = bit & 31;
    constexpr uint32_t mask = (1u << BITS) - 1u;
    uint32_t v = w[wi] >> off;
    if constexpr (off + BITS > 32) v |= w[wi + 1] << (32 - off);
    return v & mask;
  }
};

// Code of a runtime channel read from global memory (outlier corrections).
template <int BITS>
__device__ __forceinline__ uint32_t code_at(const uint8_t* row, int c) {
  const int bit = BITS * c;
  uint32_t v = (uint32_t)__ldg(row + (bit >> 3)) >> (bit & 7);
  if ((bit & 7) + BITS > 8) v |= (uint32_t)__ldg(row + (bit >> 3) + 1) << (8 - (bit & 7));
  return v & ((1u << BITS) - 1u);
}

// cos/sin of the angle Bk*m*w_i of key block m, from the coarse tables.
__device__ __forceinline__ float2 rope_block(const float2* rope, const Dims& d, int m, int i) {
  const int half = d.D / 2;
  const float2 lo = __ldg(rope + rope_lo_off(d) + (size_t)(m % kRopeLo) * half + i);
  const float2 hi = __ldg(rope + rope_hi_off(d) + (size_t)(m / kRopeLo) * half + i);
  return rot_compose(hi, lo);
}

__device__ __forceinline__ float2 rope_fine(const float2* rope, const Dims& d, int j, int i) {
  return __ldg(rope + rope_fine_off(d) + (size_t)i * d.Bk + j);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One rotated key pair (ka, kb) at in-block offset j, dotted with G queries.
template <int D, int G>
__device__ __forceinline__ void dot_pair(float ka, float kb, int i, int j, const float2* rope,
                                         const Dims& d, const float (*qb)[D], float (&acc)[G]) {
  constexpr int HALF = D / 2;
  float ra = ka, rb = kb;
  if (rope) {
    const float2 r = rope_fine(rope, d, j, i);
    ra = fmaf(ka, r.x, -kb * r.y);
    rb = fmaf(kb, r.x, ka * r.y);
  }
#pragma unroll
  for (int g = 0; g < G; ++g) acc[g] = fmaf(qb[g][i], ra, fmaf(qb[g][i + HALF], rb, acc[g]));
}

// Dense scores of pairs [I0, I0 + NPP) of one quantized key row.
template <int BITS, int D, int G, int I0, int NPP, int CB>
__device__ __forceinline__ void score_quant(const Row<CB>& row, const float* ks, const float* kz,
                                            const float (*qb)[D], const float2* rope,
                                            const Dims& d, int j, float (&acc)[G]) {
  constexpr int HALF = D / 2;
  static_for<NPP>([&](auto kk) {
    constexpr int i = I0 + decltype(kk)::value;
    const float ka = fmaf((float)row.template code<BITS, i>(), ks[i], kz[i]);
    const float kb = fmaf((float)row.template code<BITS, i + HALF>(), ks[i + HALF], kz[i + HALF]);
    dot_pair<D, G>(ka, kb, i, j, rope, d, qb, acc);
  });
}

// Scores of pairs [I0, I0 + NPP) of one fp16 tail key row.
template <int D, int G, int I0, int NPP>
__device__ __forceinline__ void score_tail(const __half* krow, const float (*qb)[D],
                                           const float2* rope, const Dims& d, int j,
                                           float (&acc)[G]) {
  constexpr int HALF = D / 2;
#pragma unroll 8
  for (int k = 0; k < NPP; ++k) {
    const int i = I0 + k;
    dot_pair<D, G>(__half2float(krow[i]), __half2float(krow[i + HALF]), i, j, rope, d, qb, acc);
  }
}

template <int BITS, int D, int G>
__global__ void __launch_bounds__(kDecThreads) decode_partial_kernel(const DecodeArgs a) {
  constexpr int NT = kDecThreads;
  constexpr int HALF = D / 2;
  constexpr int CB = D * BITS / 8;
  constexpr int NTP = NT / HALF;       // token phases of the value step
  __shared__ float s_qp[G][D];          // q rotated to q_pos, times sm_scale*log2(e)
  __shared__ float s_qb[G][D];          // s_qp rotated back by the block start
  __shared__ float s_ks[D], s_kz[D];    // key scale/zero of the block
  __shared__ float s_sc[2][G][128];     // partial scores (two pair halves when Bk = 64)
  __shared__ float s_p[G][128];         // probabilities of the block
  __shared__ float s_m[G], s_l[G], s_alpha[G];

  const Dims d = a.d;
  const int Bk = d.Bk;
  const int tid = threadIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / d.H_kv, hkv = bh % d.H_kv;
  const int split = blockIdx.x;
  const SeqExtent ex = seq_extent(a, b);
  const int units = ex.n_full + (ex.tail_len > 0 ? 1 : 0);
  const int u0 = (int)((long long)split * units / a.n_split);
  const int u1 = (int)((long long)(split + 1) * units / a.n_split);
  const int n_out = d.n_out;

  // ---- query: rotate to q_pos, scale
  for (int e = tid; e < G * HALF; e += NT) {
    const int g = e / HALF, i = e % HALF;
    const __half* qh = a.q + ((size_t)b * a.H_q + hkv * G + g) * D;
    float u = __half2float(qh[i]), v = __half2float(qh[i + HALF]);
    if (a.rope) {
      const float2 r = rot_compose(rope_block(a.rope, d, ex.q_pos / Bk, i),
                                   rope_fine(a.rope, d, ex.q_pos % Bk, i));
      const float u2 = fmaf(u, r.x, -v * r.y);
      const float v2 = fmaf(v, r.x, u * r.y);
      u = u2;
      v = v2;
    }
    s_qp[g][i] = u * a.scale_log2;
    s_qp[g][i + HALF] = v * a.scale_log2;
  }
  if (tid < G) {
    s_m[tid] = -INFINITY;
    s_l[tid] = 0.0f;
  }

  // value step: thread owns channels (2cp, 2cp + 1), tokens j = tp mod NTP
  const int cp = tid % HALF, tp = tid / HALF;
  const int c0 = 2 * cp;
  const int vgroup = c0 / d.Gv;
  float o[G][2];
#pragma unroll
  for (int g = 0; g < G; ++g) o[g][0] = o[g][1] = 0.0f;


  for (int u = u0; u < u1; ++u) {
    const bool is_tail = (u == ex.n_full);
    const size_t kblk = unit_block(d, a.block_table, a.max_blocks, a.n_blocks, b, hkv, u);
    const size_t row0 = kblk * Bk;     // row of the block's first token
    const int t0 = u * Bk;
    const int ntok = is_tail ? ex.tail_len : Bk;
    __syncthreads();  // previous block's shared data fully consumed

    // ---- 1. query back-rotated by t0; key params
    for (int e = tid; e < G * HALF; e += NT) {
      const int g = e / HALF, i = e % HALF;
      const float u_ = s_qp[g][i], v_ = s_qp[g][i + HALF];
      if (a.rope) {
        const float2 r = rope_block(a.rope, d, u, i);          // R(t0); apply R(-t0)
        s_qb[g][i] = fmaf(u_, r.x, v_ * r.y);
        s_qb[g][i + HALF] = fmaf(v_, r.x, -u_ * r.y);
      } else {
        s_qb[g][i] = u_;
        s_qb[g][i + HALF] = v_;
      }
    }
    if (!is_tail) {
      for (int c = tid; c < D; c += NT) {
        const uint32_t w = __ldg(a.k_meta + kblk * D + c);
        s_ks[c] = h2f((uint16_t)(w & 0xFFFF));
        s_kz[c] = h2f((uint16_t)(w >> 16));
      }
    }
    __syncthreads();

    // ---- 2. scores
    {
      const int ph = (Bk == 64) ? (tid >> 6) : 0;
      const int j = (Bk == 64) ? (tid & 63) : tid;
      float acc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) acc[g] = 0.0f;
      if (j < ntok) {
        const int t = t0 + j;
        if (!is_tail) {
          const uint8_t* rowp = a.k_codes + (row0 + j) * CB;
          Row<CB> row;
          row.load(rowp);
          if (Bk == 128) {
            score_quant<BITS, D, G, 0, HALF>(row, s_ks, s_kz, s_qb, a.rope, d, j, acc);
          } else if (ph == 0) {
            score_quant<BITS, D, G, 0, HALF / 2>(row, s_ks, s_kz, s_qb, a.rope, d, j, acc);
          } else {
            score_quant<BITS, D, G, HALF / 2, HALF / 2>(row, s_ks, s_kz, s_qb, a.rope, d, j, acc);
          }
          if (ph == 0) {
            // dense-and-sparse: replace the dense value at each outlier channel
            for (int k = 0; k < n_out; ++k) {
              const uint32_t e = __ldg(a.k_outl + (row0 + j) * n_out + k);
              const int c = (int)(e & 0xFFFF);
              const float xo = h2f((uint16_t)(e >> 16));
              const float xd = fmaf((float)code_at<BITS>(rowp, c), s_ks[c], s_kz[c]);
              const float delta = xo - xd;
              const int i = c % HALF;
              float2 r = make_float2(1.0f, 0.0f);
              if (a.rope) r = rope_fine(a.rope, d, j, i);
#pragma unroll
              for (int g = 0; g < G; ++g) {
                // <q, R(j) e_c>: e_i -> (cos, sin) on (i, i+HALF); e_{i+HALF} -> (-sin, cos)
                const float wgt = (c < HALF) ? fmaf(s_qb[g][i], r.x, s_qb[g][i + HALF] * r.y)
                                             : fmaf(s_qb[g][i + HALF], r.x, -s_qb[g][i] * r.y);
                acc[g] = fmaf(delta, wgt, acc[g]);
              }
            }
          }
        } else {
          const __half* krow = a.k_tail + ((size_t)bh * Bk + j) * D;
          if (Bk == 128) {
            score_tail<D, G, 0, HALF>(krow, s_qb, a.rope, d, j, acc);
          } else if (ph == 0) {
            score_tail<D, G, 0, HALF / 2>(krow, s_qb, a.rope, d, j, acc);
          } else {
            score_tail<D, G, HALF / 2, HALF / 2>(krow, s_qb, a.rope, d, j, acc);
          }
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) s_sc[ph][g][j] = acc[g];
    }
    __syncthreads();

    // ---- 3. online softmax (log2 domain)
    {
      const int warp = tid >> 5, lane = tid & 31;
      for (int g = warp; g < G; g += NT / 32) {
        float sv[4];
        float mloc = -INFINITY;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int jj = lane + 32 * k;
          float s = -INFINITY;
          if (jj < ntok) s = s_sc[0][g][jj] + (Bk == 64 ? s_sc[1][g][jj] : 0.0f);
          sv[k] = s;
          mloc = fmaxf(mloc, s);
        }
        mloc = warp_max(mloc);
        const float m_old = s_m[g];
        const float m_new = fmaxf(m_old, mloc);
        float psum = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int jj = lane + 32 * k;
          const float p = exp2f(sv[k] - m_new);
          if (jj < 128) s_p[g][jj] = p;
          psum += p;
        }
        psum = warp_sum(psum);
        if (lane == 0) {
          const float alpha = exp2f(m_old - m_new);
          s_alpha[g] = alpha;
          s_l[g] = fmaf(s_l[g], alpha, psum);
          s_m[g] = m_new;
        }
      }
    }
    __syncthreads();

    // ---- 4. values
#pragma unroll
    for (int g = 0; g < G; ++g) {
      o[g][0] *= s_alpha[g];
      o[g][1] *= s_alpha[g];
    }
    for (int jj = tp; jj < ntok; jj += NTP) {
      const size_t t = row0 + jj;
      const uint8_t* rowp = a.v_codes + t * CB;
      uint32_t q0, q1;
      if constexpr (BITS == 4) {
        const uint32_t byte = __ldg(rowp + cp);
        q0 = byte & 15u;
        q1 = byte >> 4;
      } else {
        q0 = code_at<BITS>(rowp, c0);
        q1 = code_at<BITS>(rowp, c0 + 1);
      }
      const uint32_t msz = __ldg(a.v_meta + t * d.ng + vgroup);
      const float s = h2f((uint16_t)(msz & 0xFFFF)), z = h2f((uint16_t)(msz >> 16));
      float vx = fmaf((float)q0, s, z), vy = fmaf((float)q1, s, z);
      for (int k = 0; k < n_out; ++k) {
        const uint32_t e = __ldg(a.v_outl + t * n_out + k);
        const int c = (int)(e & 0xFFFF);
        const float xo = h2f((uint16_t)(e >> 16));
        if (c == c0) vx = xo;
        if (c == c0 + 1) vy = xo;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float p = s_p[g][jj];
        o[g][0] = fmaf(p, vx, o[g][0]);
        o[g][1] = fmaf(p, vy, o[g][1]);
      }
    }
  }
  __syncthreads();

  // ---- partial results: reduce the NTP token phases, write (o, m, l)
  float* red = &s_sc[0][0][0];   // [NTP][G][D] (fits: NTP * D = 256)
#pragma unroll
  for (int g = 0; g < G; ++g) {
    red[(tp * G + g) * D + c0] = o[g][0];
    red[(tp * G + g) * D + c0 + 1] = o[g][1];
  }
  __syncthreads();
  for (int e = tid; e < G * D; e += NT) {
    const int g = e / D, c = e % D;
    float sum = 0.0f;
#pragma unroll
    for (int k = 0; k < NTP; ++k) sum += red[(k * G + g) * D + c];
    float* dst = a.ws + (((size_t)b * a.H_q + hkv * G + g) * a.S + split) * (D + 2);
    dst[c] = sum;
    if (c == 0) {
      dst[D] = s_m[g];
      dst[D + 1] = s_l[g];
    }
  }
}

template <int BITS, int D, int G>
cudaError_t launch_partial(const DecodeArgs& a, cudaStream_t st);
template <int BITS, int D, int G>
int partial_occupancy();

}  // namespace kvq
