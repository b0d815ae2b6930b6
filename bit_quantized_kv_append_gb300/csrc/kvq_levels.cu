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
// Plain CUDA-core kernels (a per-element division and table lookups; the
// tensor-core kernels serve the uniform grid), for caches filled in whole key
// blocks: an append kernel (one CTA per key block, stream and {K, V}), a
// split-T decode kernel and its combine.
#include "kvq_levels.cuh"

namespace kvq {
namespace {

constexpr int kLvThreads = 128;

__device__ __forceinline__ uint16_t hbits16(__half h) { return __half_as_ushort(h); }
__device__ __forceinline__ float hf(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// Range and zero of a group from the binary32 min/max of its dense elements;
// any = false: every element is an outlier (r = z = 0). Returns {r, z} as fp16
// bits (low, high) and the binary32 values.
__device__ uint32_t range_zero(float mn, float mx, bool any, float* r_out, float* z_out) {
  if (!any) {
    *r_out = 0.0f;
    *z_out = 0.0f;
    return 0u;
  }
  const __half rh = __float2half_ru(__fsub_rn(mx, mn));
  const float z = (mn == 0.0f) ? 0.0f : mn;     // -0 stored as +0; mn is an fp16 value: exact
  *r_out = __half2float(rh);
  *z_out = z;
  return (uint32_t)hbits16(rh) | ((uint32_t)hbits16(__float2half_rn(z)) << 16);
}

// Nearest level of u = fp32(fp32(x - z) / r); 0 when r = 0.
__device__ uint32_t level_code(float x, float z, float r, const LevelTable& t) {
  if (!(r > 0.0f)) return 0u;
  const float u = __fdiv_rn(__fsub_rn(x, z), r);
  uint32_t q = 0;
  for (int k = 0; k < t.L; ++k) q += (u > t.mid[k]) ? 1u : 0u;
  return q;
}

// Code of channel c in a packed LSB-first row.
__device__ __forceinline__ uint32_t row_code(const uint8_t* row, int c, int bits) {
  const int bit = bits * c;
  uint32_t v = (uint32_t)row[bit >> 3] >> (bit & 7);
  if ((bit & 7) + bits > 8) v |= (uint32_t)row[(bit >> 3) + 1] << (8 - (bit & 7));
  return v & ((1u << bits) - 1u);
}

struct LvAppendArgs {
  Dims d;
  uint8_t* k_codes;
  uint32_t* k_meta;
  uint32_t* k_outl;
  uint8_t* v_codes;
  uint32_t* v_meta;
  uint32_t* v_outl;
  const __half* k_new;
  const __half* v_new;
  int T_cur, n_new;
};

// One key block of one stream: keys (blockIdx.z = 1) or the block's values.
__global__ void __launch_bounds__(kLvThreads) append_levels_kernel(const LvAppendArgs a, const LevelTable t) {
  extern __shared__ __align__(16) unsigned char smem[];
  const Dims d = a.d;
  const int D = d.D, Bk = d.Bk, n_out = d.n_out, bits = d.bits, ng = d.ng;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bh = blockIdx.y;
  const bool isK = blockIdx.z != 0;
  const int t0 = a.T_cur + (int)blockIdx.x * Bk;          // first token of the block
  const int wpr = D / 32;                                  // outlier-mask words per row
  __half* sX = reinterpret_cast<__half*>(smem);                                   // [Bk][D]
  uint32_t* sEx = reinterpret_cast<uint32_t*>(sX + (size_t)Bk * D);               // [Bk][D/32]
  const int np = D > Bk * ng ? D : Bk * ng;
  float* sR = reinterpret_cast<float*>(sEx + (size_t)Bk * wpr);                   // keys [D], values [Bk][ng]
  float* sZ = sR + np;

  // 1. stage the block's rows; clear the outlier marks
  const __half* src = (isK ? a.k_new : a.v_new) + ((size_t)bh * a.n_new + (t0 - a.T_cur)) * D;
  for (int i = tid; i < Bk * D / 8; i += kLvThreads)
    reinterpret_cast<uint4*>(sX)[i] = __ldg(reinterpret_cast<const uint4*>(src) + i);
  for (int i = tid; i < Bk * wpr; i += kLvThreads) sEx[i] = 0u;
  __syncthreads();

  // 2. outliers: per row the n_out largest |x| (fp16 magnitude bits order like
  // |x|), ties to the lower channel: keys (|x| bits << 8) | (255 - channel)
  const size_t row0 = (size_t)bh * d.T_max + t0;           // row of the block's first token
  uint32_t* gout = isK ? a.k_outl : a.v_outl;
  const int E = D / 32;                                    // elements per lane (2 or 4)
  for (int r = warp; r < Bk; r += kLvThreads / 32) {
    uint32_t key[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = lane * E + e;
      key[e] = (e < E) ? (((uint32_t)(hbits16(sX[r * D + c]) & 0x7FFFu) << 8) | (uint32_t)(255 - c)) : 0u;
    }
    for (int k = 0; k < n_out; ++k) {
      uint32_t best = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) best = max(best, key[e]);
      best = __reduce_max_sync(0xffffffffu, best);
#pragma unroll
      for (int e = 0; e < 4; ++e) key[e] = (key[e] == best) ? 0u : key[e];
      const int c = 255 - (int)(best & 0xFFu);
      if (lane == 0) {
        gout[(row0 + r) * n_out + k] = (uint32_t)c | ((uint32_t)hbits16(sX[r * D + c]) << 16);
        sEx[r * wpr + (c >> 5)] |= 1u << (c & 31);
      }
    }
  }
  __syncthreads();

  // 3. range and zero: values per (token, group), keys per channel over the block
  if (!isK) {
    for (int it = tid; it < Bk * ng; it += kLvThreads) {
      const int r = it / ng, g = it - r * ng;
      float mn = INFINITY, mx = -INFINITY;
      bool any = false;
      for (int c = g * d.Gv; c < (g + 1) * d.Gv; ++c) {
        if ((sEx[r * wpr + (c >> 5)] >> (c & 31)) & 1u) continue;
        const float x = __half2float(sX[r * D + c]);
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
        any = true;
      }
      a.v_meta[(row0 + r) * ng + g] = range_zero(mn, mx, any, &sR[it], &sZ[it]);
    }
  } else {
    for (int c = tid; c < D; c += kLvThreads) {
      float mn = INFINITY, mx = -INFINITY;
      bool any = false;
      for (int r = 0; r < Bk; ++r) {
        if ((sEx[r * wpr + (c >> 5)] >> (c & 31)) & 1u) continue;
        const float x = __half2float(sX[r * D + c]);
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
        any = true;
      }
      a.k_meta[((size_t)bh * d.n_blk + t0 / Bk) * D + c] = range_zero(mn, mx, any, &sR[c], &sZ[c]);
    }
  }
  __syncthreads();

  // 4. codes of every element (outlier positions too), packed LSB-first, one row per thread
  for (int r = tid; r < Bk; r += kLvThreads) {
    uint32_t w[32];                                       // a row is at most 128 bytes
    for (int i = 0; i < 32; ++i) w[i] = 0u;
    for (int c = 0; c < D; ++c) {
      const int gi = isK ? c : r * ng + c / d.Gv;
      const uint32_t q = level_code(__half2float(sX[r * D + c]), sZ[gi], sR[gi], t);
      const int bit = bits * c, wi = bit >> 5, sh = bit & 31;
      w[wi] |= q << sh;
      if (sh + bits > 32) w[wi + 1] |= q >> (32 - sh);
    }
    uint32_t* dst = reinterpret_cast<uint32_t*>((isK ? a.k_codes : a.v_codes) + (row0 + r) * d.cb);
    for (int i = 0; i < d.cb / 4; ++i) dst[i] = w[i];
  }
}

struct LvDecodeArgs {
  Dims d;
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
  const int units = a.T / Bk;
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
    // scores: thread j takes token t0 + j
    for (int j = tid; j < Bk; j += kLvThreads) {
      const size_t row = stream_row + t0 + j;
      const uint8_t* kr = a.k_codes + row * d.cb;
      const uint32_t* km = a.k_meta + ((size_t)bh * d.n_blk + u) * D;
      float acc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) acc[g] = 0.0f;
      for (int i = 0; i < HALF; ++i) {
        const uint32_t ma = __ldg(km + i), mb = __ldg(km + i + HALF);
        float ka = fmaf(hf((uint16_t)(ma & 0xFFFFu)), s_lv[row_code(kr, i, bits)], hf((uint16_t)(ma >> 16)));
        float kb = fmaf(hf((uint16_t)(mb & 0xFFFFu)), s_lv[row_code(kr, i + HALF, bits)], hf((uint16_t)(mb >> 16)));
        for (int k = 0; k < n_out; ++k) {               // dense-and-sparse: the outlier's own value
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
      for (int j = 0; j < Bk; ++j) {
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

cudaError_t launch_append_levels(const Dims& d, const kvq_cache& c, const __half* k_new, const __half* v_new,
                                 int n_new, const LevelTable& t, cudaStream_t st) {
  LvAppendArgs a;
  a.d = d;
  a.k_codes = static_cast<uint8_t*>(c.k_codes);
  a.k_meta = static_cast<uint32_t*>(c.k_meta);
  a.k_outl = static_cast<uint32_t*>(c.k_outl);
  a.v_codes = static_cast<uint8_t*>(c.v_codes);
  a.v_meta = static_cast<uint32_t*>(c.v_meta);
  a.v_outl = static_cast<uint32_t*>(c.v_outl);
  a.k_new = k_new;
  a.v_new = v_new;
  a.T_cur = c.T_cur;
  a.n_new = n_new;
  const int np = d.D > d.Bk * d.ng ? d.D : d.Bk * d.ng;
  const size_t smem = (size_t)d.Bk * d.D * sizeof(__half) + (size_t)d.Bk * (d.D / 32) * sizeof(uint32_t) +
                      2 * (size_t)np * sizeof(float);
  const dim3 grid(n_new / d.Bk, d.B * d.H_kv, 2);
  append_levels_kernel<<<grid, kLvThreads, smem, st>>>(a, t);
  return cudaGetLastError();
}

cudaError_t launch_decode_levels(const Dims& d, const kvq_cache& c, const __half* q, int H_q, int q_pos,
                                 const float2* rope, float sm_scale, __half* out, float* ws,
                                 const LevelTable& t, cudaStream_t st) {
  LvDecodeArgs a;
  a.d = d;
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
  const int units = a.T / d.Bk, streams = d.B * d.H_kv;
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
