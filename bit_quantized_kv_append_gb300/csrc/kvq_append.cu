// kvq_append: quantize new keys and values into the packed cache.
//
// KV Cache量化技术介绍 (developer.horizon.auto/blog/13163):
//   KVQuant "Per-Vector Dense-and-Sparse Quantization" -> step B (outliers);
//   KVQuant "Per-Channel Key Quantization"             -> step C, keys;
//   Quanto steps 1-2 (block scale and zero_point)       -> step C, values;
//   codes and LSB-first packing                         -> step D.
// One CTA per (key block touched by the append, (b, h_kv) stream). The CTA
// stages the block's new value rows, and the block's keys when the append
// completes it, in shared memory, then runs the steps in the method's order.
// All rounding follows the library's stated arithmetic: binary32 RN subtract
// and divide, fp16 round-up for the scale, round-half-even codes.
#include "kvq_common.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxGroups = 4;  // D / Gv <= 128 / 32

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
};

__device__ __forceinline__ uint16_t hbits(__half h) { return __half_as_ushort(h); }

// clamp(rint((x - z) / s), 0, L) in binary32 round-to-nearest; 0 when s = 0.
// Clamping r to [0, L] before rounding gives the same integer as clamping after.
__device__ __forceinline__ uint32_t quant_code(float x, float z, float s, float Lf) {
  if (s == 0.0f) return 0u;
  float r = __fdiv_rn(__fsub_rn(x, z), s);
  r = fminf(fmaxf(r, 0.0f), Lf);
  return (uint32_t)__float2int_rn(r);
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

template <int BITS>
__device__ __forceinline__ void pack32(const uint32_t (&q)[32], uint32_t (&w)[BITS]) {
#pragma unroll
  for (int k = 0; k < BITS; ++k) w[k] = 0u;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const int bit = e * BITS;
    w[bit >> 5] |= q[e] << (bit & 31);
    if ((bit & 31) + BITS > 32) w[(bit >> 5) + 1] |= q[e] >> (32 - (bit & 31));
  }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) append_kernel(const AppendArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const Dims d = a.d;
  const int D = d.D, Bk = d.Bk, n_out = d.n_out;
  const int bh = blockIdx.y;
  const int blk = a.first_blk + blockIdx.x;
  const int t_blk0 = blk * Bk;
  const int t_end = a.T_cur + a.n_new;
  const int t_lo = max(t_blk0, a.T_cur);
  const int t_hi = min(t_blk0 + Bk, t_end);
  const int nv = t_hi - t_lo;                      // new tokens in this block, >= 1
  const bool complete = t_blk0 + Bk <= t_end;
  const float Lf = (float)((1 << BITS) - 1);

  __half* sV = reinterpret_cast<__half*>(smem);                       // [Bk][D]
  __half* sK = sV + Bk * D;                                            // [Bk][D]
  uint16_t* sVo = reinterpret_cast<uint16_t*>(sK + Bk * D);           // [Bk][MAX_OUT]
  uint16_t* sKo = sVo + Bk * KVQ_MAX_OUTLIERS;                         // [Bk][MAX_OUT]
  float2* sVsz = reinterpret_cast<float2*>(sKo + Bk * KVQ_MAX_OUTLIERS);  // [Bk][4]
  float2* sKsz = sVsz + Bk * kMaxGroups;                               // [D]

  // ---- A. stage rows in shared memory (16-byte vectors)
  const int vpr = D / 8;
  const __half* v_src = a.v_new + ((size_t)bh * a.n_new + (t_lo - a.T_cur)) * D;
  for (int i = threadIdx.x; i < nv * vpr; i += kThreads) {
    const int r = i / vpr, c = i % vpr;
    reinterpret_cast<uint4*>(sV + r * D)[c] =
        __ldg(reinterpret_cast<const uint4*>(v_src + (size_t)r * D) + c);
  }
  __half* tail = a.k_tail + (size_t)bh * Bk * D;
  if (complete) {
    for (int i = threadIdx.x; i < Bk * vpr; i += kThreads) {
      const int j = i / vpr, c = i % vpr;
      const int t = t_blk0 + j;
      const __half* src = (t < a.T_cur) ? tail + (size_t)j * D
                                        : a.k_new + ((size_t)bh * a.n_new + (t - a.T_cur)) * D;
      reinterpret_cast<uint4*>(sK + j * D)[c] = reinterpret_cast<const uint4*>(src)[c];
    }
  } else if (a.tail_in_kernel) {
    // unfinished block: keep the new keys as fp16 rows t % Bk of the tail
    for (int i = threadIdx.x; i < nv * vpr; i += kThreads) {
      const int r = i / vpr, c = i % vpr;
      const int t = t_lo + r;
      reinterpret_cast<uint4*>(tail + (size_t)(t - t_blk0) * D)[c] = __ldg(
          reinterpret_cast<const uint4*>(a.k_new + ((size_t)bh * a.n_new + (t - a.T_cur)) * D) + c);
    }
  }
  __syncthreads();

  // ---- B. dense-and-sparse split: per vector, the n_out largest |x|
  if (n_out > 0) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = D >> 5;                          // elements per lane (2 or 4)
    const int nrows = nv + (complete ? Bk : 0);
    for (int r = warp; r < nrows; r += kThreads / 32) {
      const bool isV = r < nv;
      const int row = isV ? r : r - nv;
      const __half* x = (isV ? sV : sK) + row * D;
      uint16_t* so = (isV ? sVo : sKo) + row * KVQ_MAX_OUTLIERS;
      const int t = isV ? t_lo + row : t_blk0 + row;
      uint32_t* gout = (isV ? a.v_outl : a.k_outl) + ((size_t)bh * d.T_max + t) * n_out;
      // key = |x| bits (15) above (255 - channel): the max is the largest |x|,
      // lowest channel on ties; keys of distinct channels never coincide
      uint32_t key[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = lane * E + e;
        key[e] = (e < E) ? (((uint32_t)(hbits(x[c]) & 0x7FFF) << 8) | (uint32_t)(255 - c)) : 0u;
      }
      for (int k = 0; k < n_out; ++k) {
        uint32_t best = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) best = max(best, key[e]);
        best = __reduce_max_sync(0xffffffffu, best);
#pragma unroll
        for (int e = 0; e < 4; ++e) key[e] = (key[e] == best) ? 0u : key[e];
        if (lane == 0) {
          const int c = 255 - (int)(best & 0xFF);
          so[k] = (uint16_t)c;
          gout[k] = (uint32_t)c | ((uint32_t)hbits(x[c]) << 16);
        }
      }
    }
  }
  __syncthreads();

  // ---- C. statistics: values per (token, group), keys per channel over the block
  {
    const int Gv = d.Gv, ng = d.ng;
    const int nVi = nv * ng;
    const int nKi = complete ? D : 0;
    for (int it = threadIdx.x; it < nVi + nKi; it += kThreads) {
      float mn = INFINITY, mx = -INFINITY;
      bool any = false;
      if (it < nVi) {
        const int r = it / ng, g = it % ng;
        const __half* x = sV + r * D + g * Gv;
        const uint16_t* so = sVo + r * KVQ_MAX_OUTLIERS;
        for (int k = 0; k < Gv; ++k) {
          const int cc = (k + threadIdx.x) & (Gv - 1);   // staggered start spreads banks
          const int c = g * Gv + cc;
          bool ex = false;
          for (int o = 0; o < n_out; ++o) ex |= (so[o] == c);
          if (!ex) {
            const float v = __half2float(x[cc]);
            mn = fminf(mn, v);
            mx = fmaxf(mx, v);
            any = true;
          }
        }
        float2 sz;
        const uint32_t packed = group_params(mn, mx, any, Lf, &sz);
        a.v_meta[((size_t)bh * d.T_max + (t_lo + r)) * ng + g] = packed;
        sVsz[r * kMaxGroups + g] = sz;
      } else {
        const int c = it - nVi;
        for (int j = 0; j < Bk; ++j) {
          const uint16_t* so = sKo + j * KVQ_MAX_OUTLIERS;
          bool ex = false;
          for (int o = 0; o < n_out; ++o) ex |= (so[o] == c);
          if (!ex) {
            const float v = __half2float(sK[j * D + c]);
            mn = fminf(mn, v);
            mx = fmaxf(mx, v);
            any = true;
          }
        }
        float2 sz;
        const uint32_t packed = group_params(mn, mx, any, Lf, &sz);
        a.k_meta[((size_t)bh * d.n_blk + blk) * D + c] = packed;
        sKsz[c] = sz;
      }
    }
  }
  __syncthreads();

  // ---- D. codes for every element (outlier positions included), packed
  {
    const int nch = D / 32;
    const int nVc = nv * nch;
    const int nKc = complete ? Bk * nch : 0;
    for (int it = threadIdx.x; it < nVc + nKc; it += kThreads) {
      const bool isV = it < nVc;
      const int k = isV ? it : it - nVc;
      const int r = k / nch, ch = k % nch;
      const __half* x = (isV ? sV : sK) + r * D + ch * 32;
      uint32_t q[32];
      if (isV) {
        const float2 sz = sVsz[r * kMaxGroups + (ch * 32) / d.Gv];
#pragma unroll
        for (int e = 0; e < 32; ++e) q[e] = quant_code(__half2float(x[e]), sz.y, sz.x, Lf);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float2 sz = sKsz[ch * 32 + e];
          q[e] = quant_code(__half2float(x[e]), sz.y, sz.x, Lf);
        }
      }
      uint32_t w[BITS];
      pack32<BITS>(q, w);
      const int t = isV ? t_lo + r : t_blk0 + r;
      uint8_t* base = isV ? a.v_codes : a.k_codes;
      uint32_t* dst = reinterpret_cast<uint32_t*>(base + ((size_t)bh * d.T_max + t) * d.cb) + ch * BITS;
#pragma unroll
      for (int b = 0; b < BITS; ++b) dst[b] = w[b];
    }
  }
}

// Keys of the last, unfinished block of a multi-block append whose first block
// read the old tail: written after the main launch so the two never overlap.
__global__ void tail_copy_kernel(__half* __restrict__ k_tail, const __half* __restrict__ k_new,
                                 int Bk, int D, int n_new, int T_cur, int t_from, int t_to) {
  const int bh = blockIdx.y;
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
  return (size_t)2 * d.Bk * d.D * sizeof(__half) + (size_t)2 * d.Bk * KVQ_MAX_OUTLIERS * sizeof(uint16_t) +
         (size_t)d.Bk * kMaxGroups * sizeof(float2) + (size_t)d.D * sizeof(float2);
}

template <int BITS>
cudaError_t launch_bits(const AppendArgs& a, dim3 grid, size_t smem, cudaStream_t st) {
  static bool attr_set = false;  // per device the attribute is idempotent
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(append_kernel<BITS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  append_kernel<BITS><<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(const Dims& d, const kvq_cache& c, const __half* k_new,
                          const __half* v_new, int n_new, cudaStream_t st) {
  const int T_cur = c.T_cur, t_end = T_cur + n_new;
  const int first = T_cur / d.Bk, last = (t_end - 1) / d.Bk;
  const bool last_unfinished = (t_end % d.Bk) != 0;
  const bool first_reads_tail = (T_cur % d.Bk) != 0;
  const bool defer_tail = last_unfinished && first != last && first_reads_tail;

  AppendArgs a;
  a.d = d;
  a.k_codes = static_cast<uint8_t*>(c.k_codes);
  a.k_meta = static_cast<uint32_t*>(c.k_meta);
  a.k_tail = static_cast<__half*>(c.k_tail);
  a.k_outl = static_cast<uint32_t*>(c.k_outl);
  a.v_codes = static_cast<uint8_t*>(c.v_codes);
  a.v_meta = static_cast<uint32_t*>(c.v_meta);
  a.v_outl = static_cast<uint32_t*>(c.v_outl);
  a.k_new = k_new;
  a.v_new = v_new;
  a.T_cur = T_cur;
  a.n_new = n_new;
  a.first_blk = first;
  a.tail_in_kernel = defer_tail ? 0 : 1;

  const dim3 grid(last - first + 1, d.B * d.H_kv);
  const size_t smem = append_smem(d);
  cudaError_t e;
  switch (d.bits) {
    case 2: e = launch_bits<2>(a, grid, smem, st); break;
    case 3: e = launch_bits<3>(a, grid, smem, st); break;
    default: e = launch_bits<4>(a, grid, smem, st); break;
  }
  if (e != cudaSuccess || !defer_tail) return e;
  const int rows = t_end - last * d.Bk;
  const int blocks = (rows * (d.D / 8) + 255) / 256;
  tail_copy_kernel<<<dim3(blocks, d.B * d.H_kv), 256, 0, st>>>(
      static_cast<__half*>(c.k_tail), k_new, d.Bk, d.D, n_new, T_cur, last * d.Bk, t_end);
  return cudaGetLastError();
}

}  // namespace kvq
