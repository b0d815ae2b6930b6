// Plain CPU oracle for low-bit KV-cache quantization and decode attention.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product library links, loads or
// calls this file; only the tests, the smoke check and the benchmark's CPU
// baseline do. It shares no code, header or table with the CUDA path.
//
// What it computes (step by step, in the order the method states it):
//   KV Cache量化技术介绍 (developer.horizon.auto/blog/13163), KVQuant section:
//     "Per-Channel Key Quantization"  -> keys get one scale/zero per channel
//                                         over a block of tokens;
//     "Pre-RoPE Key Quantization"     -> keys are quantized before RoPE, and
//                                         RoPE is applied after dequantization;
//     "Per-Vector Dense-and-Sparse Quantization" -> each vector's largest
//                                         |x| elements are kept apart (sparse)
//                                         and the rest is quantized (dense).
//   Same page, Quanto section, steps 1-2: block-wise quantization where each
//     block keeps a scale and a zero_point used to restore the values.
//   Readings taken where the page is silent or its formula image was lost:
//   unsigned codes q in [0, L], L = 2^b - 1;
//   zero z = the block minimum (fp16, exact); scale s = (max - min) / L in fp32,
//   stored in fp16 rounded toward +infinity; q = clamp(rint((x - z) / s), 0, L)
//   with fp32 round-to-nearest arithmetic and round-half-to-even; x_hat =
//   q * s + z; outlier slots hold (index, fp16 value) ordered by descending
//   |x| then ascending index; a group with max == min has s = 0 and codes 0; a
//   group whose every element is an outlier has s = 0, z = 0.
//
//   Page mlqm.cn/news/1064729 ("UltraQuant ..."), §3.2, sliding-window
//     statistics: the scale and zero of a key block may come from the most
//     recent W tokens (W a multiple of the block, e.g. 1024) instead of the
//     block alone. Reading: for key block b and channel c, (s, z) are the
//     group parameters of the dense elements of channel c in tokens
//     [max(0, (b + 1) Bk - W), (b + 1) Bk); the block's codes use them (the
//     clamp of the code rule never binds for the block's own elements, which
//     lie inside the window). W = Bk is the per-block rule.
//
//   Same page, KVQuant "Non-Uniform KV Cache Quantization": codes may instead
//     index a calibrated table of levels (a non-uniform grid). Reading: 2^b
//     sorted levels 0 = l_0 < ... < l_L = 1 on the group's normalized range;
//     r = fp16_round_up(fp32(max) - fp32(min)) (the range) takes the scale's
//     slot; u = fp32(fp32(x - z) / r); the code is the nearest level (the
//     number of binary32 midpoints fp32(0.5 (l_k + l_k+1)) below u; ties to the
//     lower level); x_hat = z + r * l_code. The table is fitted offline by
//     one-dimensional k-means (Lloyd) on normalized calibration values with the
//     end levels held at 0 and 1 (the pages' sensitivity weighting needs
//     gradients of a model and is left out).
//
// Build: g++ -O2 -ffp-contract=off -fPIC -shared (no fast-math, no SIMD
// intrinsics), so every float operation below is one IEEE-754 binary32 or
// binary64 operation rounded to nearest.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------- binary16
// IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.

double half_to_double(uint16_t h) {
  const int sign = h >> 15;
  const int e = (h >> 10) & 0x1F;
  const int f = h & 0x3FF;
  double v;
  if (e == 0) {
    v = std::ldexp(static_cast<double>(f), -24);           // subnormal
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = std::ldexp(static_cast<double>(f | 0x400), e - 25);  // 1.f * 2^(e-15)
  }
  return sign ? -v : v;
}

// Every binary16 value is exactly a binary32 value.
float half_to_float(uint16_t h) { return static_cast<float>(half_to_double(h)); }

// Encode a non-negative double that is exactly a binary16 value.
uint16_t encode_exact_half(double v) {
  if (v == 0.0) return 0;
  if (v >= 65536.0) return 0x7C00;
  if (v < std::ldexp(1.0, -14)) {
    return static_cast<uint16_t>(std::ldexp(v, 24));        // f * 2^-24
  }
  int k;
  std::frexp(v, &k);                                          // v in [2^(k-1), 2^k)
  const int e = k - 1;                                        // unbiased exponent
  const double frac = std::ldexp(v, -e) - 1.0;                // in [0, 1)
  const int f = static_cast<int>(std::ldexp(frac, 10));
  return static_cast<uint16_t>(((e + 15) << 10) | f);
}

// Smallest binary16 value >= x, for finite x >= 0 (round toward +infinity).
uint16_t float_to_half_up(float x) {
  const double v = static_cast<double>(x);
  if (v <= 0.0) return 0;
  if (v > 65504.0) return 0x7C00;
  double ulp;
  if (v < std::ldexp(1.0, -14)) {
    ulp = std::ldexp(1.0, -24);
  } else {
    int k;
    std::frexp(v, &k);
    ulp = std::ldexp(1.0, (k - 1) - 10);
  }
  const double m = std::ceil(v / ulp);                        // exact: ulp is 2^n
  return encode_exact_half(m * ulp);
}

// Round half to even, for the finite binary32 quotient of the code step.
double rint_half_even(float r) {
  const double x = static_cast<double>(r);
  const double fl = std::floor(x);
  const double fr = x - fl;                                   // exact
  if (fr > 0.5) return fl + 1.0;
  if (fr < 0.5) return fl;
  return (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

// ---------------------------------------------------------------- method steps

// Dense-and-sparse split of one vector: the n_out indices with the largest
// |x|; ties go to the lower index; slots ordered by descending |x| then index.
void select_outliers(const uint16_t* x, int D, int n_out, uint16_t* idx, uint16_t* val) {
  std::vector<int> order(D);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
    return half_to_double(x[a] & 0x7FFF) > half_to_double(x[b] & 0x7FFF);
  });
  for (int k = 0; k < n_out; ++k) {
    idx[k] = static_cast<uint16_t>(order[k]);
    val[k] = x[order[k]];
  }
}

// Scale and zero-point of one block (Quanto steps 1-2), over the elements that
// are not outliers. Returns binary16 bit patterns.
void group_params(const std::vector<uint16_t>& elems, int bits, uint16_t* s_out, uint16_t* z_out) {
  if (elems.empty()) {  // every element of the group is an outlier
    *s_out = 0;
    *z_out = 0;
    return;
  }
  double mn = INFINITY, mx = -INFINITY;
  for (uint16_t e : elems) {
    const double v = half_to_double(e);
    mn = std::min(mn, v);
    mx = std::max(mx, v);
  }
  const int L = (1 << bits) - 1;
  // z is the minimum itself; -0 is stored as +0.
  uint16_t zb = 0;
  for (uint16_t e : elems) {
    if (half_to_double(e) == mn) { zb = e; break; }
  }
  if (mn == 0.0) zb = 0;
  const float range = static_cast<float>(mx) - static_cast<float>(mn);  // binary32, RN
  const float q = range / static_cast<float>(L);                        // binary32, RN
  *s_out = float_to_half_up(q);
  *z_out = zb;
}

// Integer code of one element: clamp(rint((x - z) / s), 0, L).
int quantize_one(uint16_t x, uint16_t s, uint16_t z, int bits) {
  const int L = (1 << bits) - 1;
  if ((s & 0x7FFF) == 0) return 0;
  const float d = half_to_float(x) - half_to_float(z);       // binary32, RN
  const float r = d / half_to_float(s);                      // binary32, RN
  if (!(r > 0.0f)) return 0;
  if (r >= static_cast<float>(L)) return L;
  const double n = rint_half_even(r);
  return static_cast<int>(std::min<double>(n, L));
}

// ---------------------------------------------------------------- non-uniform codes
// Range and zero of one group for a level table: r = fp16_round_up(max - min)
// in binary32, z = min (fp16, -0 stored as +0); an all-outlier group has r = z = 0.
void group_params_nuq(const std::vector<uint16_t>& elems, uint16_t* r_out, uint16_t* z_out) {
  if (elems.empty()) {
    *r_out = 0;
    *z_out = 0;
    return;
  }
  double mn = INFINITY, mx = -INFINITY;
  for (uint16_t e : elems) {
    const double v = half_to_double(e);
    mn = std::min(mn, v);
    mx = std::max(mx, v);
  }
  uint16_t zb = 0;
  for (uint16_t e : elems) {
    if (half_to_double(e) == mn) { zb = e; break; }
  }
  if (mn == 0.0) zb = 0;
  *r_out = float_to_half_up(static_cast<float>(mx) - static_cast<float>(mn));   // binary32, RN, then up
  *z_out = zb;
}

// Binary32 midpoints between consecutive levels.
std::vector<float> level_mids(const float* levels, int L) {
  std::vector<float> mids(L);
  for (int k = 0; k < L; ++k) mids[k] = (levels[k] + levels[k + 1]) * 0.5f;
  return mids;
}

// Code of one element against a level table: the nearest level of
// u = fp32(fp32(x - z) / r), i.e. the number of midpoints below u.
int quantize_nuq(uint16_t x, uint16_t r, uint16_t z, const std::vector<float>& mids) {
  if ((r & 0x7FFF) == 0) return 0;
  const float d = half_to_float(x) - half_to_float(z);       // binary32, RN
  const float u = d / half_to_float(r);                      // binary32, RN
  int q = 0;
  for (float m : mids)
    if (u > m) ++q;
  return q;
}

// One-dimensional k-means (Lloyd) of samples u in [0, 1] into 2^b levels,
// starting from the uniform grid k / L; the end levels stay at 0 and 1, an
// interior level moves to the mean of the samples nearest to it (a level
// with no samples stays). binary64 throughout; the result is rounded to binary32.
void nuq_fit(const double* u, size_t n, int bits, int iters, float* levels_out) {
  const int L = (1 << bits) - 1;
  std::vector<double> lv(L + 1);
  for (int k = 0; k <= L; ++k) lv[k] = static_cast<double>(k) / L;
  std::vector<double> sum(L + 1), cnt(L + 1), mids(L);
  for (int it = 0; it < iters; ++it) {
    for (int k = 0; k < L; ++k) mids[k] = 0.5 * (lv[k] + lv[k + 1]);
    std::fill(sum.begin(), sum.end(), 0.0);
    std::fill(cnt.begin(), cnt.end(), 0.0);
    for (size_t i = 0; i < n; ++i) {
      int q = 0;
      while (q < L && u[i] > mids[q]) ++q;                      // the nearest level, ties to the lower
      sum[q] += u[i];
      cnt[q] += 1.0;
    }
    for (int k = 1; k < L; ++k)
      if (cnt[k] > 0) lv[k] = sum[k] / cnt[k];
  }
  for (int k = 0; k <= L; ++k) levels_out[k] = static_cast<float>(lv[k]);
}

// LSB-first bit packing of one row: element d occupies bits [b*d, b*d + b).
void pack_row(const int* codes, int D, int bits, uint8_t* out) {
  const int nbytes = D * bits / 8;
  std::memset(out, 0, nbytes);
  for (int d = 0; d < D; ++d) {
    for (int k = 0; k < bits; ++k) {
      if ((codes[d] >> k) & 1) {
        const int bit = bits * d + k;
        out[bit / 8] = static_cast<uint8_t>(out[bit / 8] | (1u << (bit % 8)));
      }
    }
  }
}

int unpack_one(const uint8_t* row, int d, int bits) {
  int q = 0;
  for (int k = 0; k < bits; ++k) {
    const int bit = bits * d + k;
    q |= ((row[bit / 8] >> (bit % 8)) & 1) << k;
  }
  return q;
}

struct Shape {
  int T, D, bits, Bk, Gv, n_out;
  int row_bytes() const { return D * bits / 8; }
  int n_full() const { return T / Bk; }
};

bool is_outlier(const uint16_t* idx, int n_out, int c) {
  for (int k = 0; k < n_out; ++k)
    if (idx[k] == c) return true;
  return false;
}

// Encode one (batch, kv-head) stream of T tokens.
// levels: a level table (non-uniform codes) or nullptr (uniform grid).
// window: tokens of the key statistics window (a multiple of Bk; Bk or 0:
// the block alone).
void encode_stream(const Shape& sh, const uint16_t* K, const uint16_t* V,
                   uint8_t* k_codes, uint16_t* k_meta, uint16_t* k_tail, uint16_t* k_outl,
                   uint8_t* v_codes, uint16_t* v_meta, uint16_t* v_outl, const float* levels,
                   int window) {
  const int D = sh.D, T = sh.T, n_out = sh.n_out, bits = sh.bits;
  const std::vector<float> mids = levels ? level_mids(levels, (1 << bits) - 1) : std::vector<float>();
  auto params = [&](const std::vector<uint16_t>& dense, uint16_t* s, uint16_t* z) {
    if (levels) group_params_nuq(dense, s, z);
    else group_params(dense, bits, s, z);
  };
  auto code = [&](uint16_t x, uint16_t s, uint16_t z) {
    return levels ? quantize_nuq(x, s, z, mids) : quantize_one(x, s, z, bits);
  };
  const int rb = sh.row_bytes();
  const int ng = D / sh.Gv;
  std::vector<uint16_t> oi(std::max(n_out, 1)), ov(std::max(n_out, 1));
  std::vector<int> codes(D);

  // Values: per token, per group of Gv channels.
  for (int t = 0; t < T; ++t) {
    const uint16_t* x = V + static_cast<size_t>(t) * D;
    select_outliers(x, D, n_out, oi.data(), ov.data());
    for (int k = 0; k < n_out; ++k) {
      v_outl[(static_cast<size_t>(t) * n_out + k) * 2 + 0] = oi[k];
      v_outl[(static_cast<size_t>(t) * n_out + k) * 2 + 1] = ov[k];
    }
    for (int g = 0; g < ng; ++g) {
      std::vector<uint16_t> dense;
      for (int c = g * sh.Gv; c < (g + 1) * sh.Gv; ++c)
        if (!is_outlier(oi.data(), n_out, c)) dense.push_back(x[c]);
      uint16_t s, z;
      params(dense, &s, &z);
      v_meta[(static_cast<size_t>(t) * ng + g) * 2 + 0] = s;
      v_meta[(static_cast<size_t>(t) * ng + g) * 2 + 1] = z;
      for (int c = g * sh.Gv; c < (g + 1) * sh.Gv; ++c) codes[c] = code(x[c], s, z);
    }
    pack_row(codes.data(), D, bits, v_codes + static_cast<size_t>(t) * rb);
  }

  // Keys: per channel over each completed block of Bk tokens.
  const int nb = sh.n_full();
  // outlier channels of every key vector of the finished blocks
  std::vector<uint16_t> win_idx(static_cast<size_t>(nb) * sh.Bk * std::max(n_out, 1));
  for (int b = 0; b < nb; ++b) {
    const int t0 = b * sh.Bk;
    for (int j = 0; j < sh.Bk; ++j) {
      const int t = t0 + j;
      const uint16_t* x = K + static_cast<size_t>(t) * D;
      select_outliers(x, D, n_out, oi.data(), ov.data());
      for (int k = 0; k < n_out; ++k) {
        win_idx[static_cast<size_t>(t) * n_out + k] = oi[k];
        k_outl[(static_cast<size_t>(t) * n_out + k) * 2 + 0] = oi[k];
        k_outl[(static_cast<size_t>(t) * n_out + k) * 2 + 1] = ov[k];
      }
    }
    std::vector<uint16_t> s_c(D), z_c(D);
    // the statistics window: this block, or the last `window` tokens up to its end
    const int w0 = (window > sh.Bk) ? std::max(0, t0 + sh.Bk - window) : t0;
    for (int c = 0; c < D; ++c) {
      std::vector<uint16_t> dense;
      for (int t = w0; t < t0 + sh.Bk; ++t)
        if (!is_outlier(&win_idx[static_cast<size_t>(t) * n_out], n_out, c))
          dense.push_back(K[static_cast<size_t>(t) * D + c]);
      params(dense, &s_c[c], &z_c[c]);
      k_meta[(static_cast<size_t>(b) * D + c) * 2 + 0] = s_c[c];
      k_meta[(static_cast<size_t>(b) * D + c) * 2 + 1] = z_c[c];
    }
    for (int j = 0; j < sh.Bk; ++j) {
      const int t = t0 + j;
      for (int c = 0; c < D; ++c)
        codes[c] = code(K[static_cast<size_t>(t) * D + c], s_c[c], z_c[c]);
      pack_row(codes.data(), D, bits, k_codes + static_cast<size_t>(t) * rb);
    }
  }
  // Tokens of the unfinished block stay as fp16 keys.
  for (int t = nb * sh.Bk; t < T; ++t)
    std::memcpy(k_tail + static_cast<size_t>(t - nb * sh.Bk) * D, K + static_cast<size_t>(t) * D,
                sizeof(uint16_t) * D);
}

// x_hat = q * s + z (binary64; with a level table z + r * l_q), outlier
// positions restored, tail keys as fp16.
void dequant_stream(const Shape& sh, const uint8_t* k_codes, const uint16_t* k_meta,
                    const uint16_t* k_tail, const uint16_t* k_outl, const uint8_t* v_codes,
                    const uint16_t* v_meta, const uint16_t* v_outl, double* Kh, double* Vh,
                    const float* levels) {
  auto value = [&](int q, double s, double z) {
    return levels ? z + s * static_cast<double>(levels[q]) : q * s + z;
  };
  const int D = sh.D, T = sh.T, n_out = sh.n_out, bits = sh.bits;
  const int rb = sh.row_bytes();
  const int ng = D / sh.Gv;
  const int nb = sh.n_full();
  for (int t = 0; t < T; ++t) {
    const uint8_t* vr = v_codes + static_cast<size_t>(t) * rb;
    for (int c = 0; c < D; ++c) {
      const int g = c / sh.Gv;
      const double s = half_to_double(v_meta[(static_cast<size_t>(t) * ng + g) * 2 + 0]);
      const double z = half_to_double(v_meta[(static_cast<size_t>(t) * ng + g) * 2 + 1]);
      Vh[static_cast<size_t>(t) * D + c] = value(unpack_one(vr, c, bits), s, z);
    }
    for (int k = 0; k < n_out; ++k) {
      const uint16_t i = v_outl[(static_cast<size_t>(t) * n_out + k) * 2 + 0];
      const uint16_t v = v_outl[(static_cast<size_t>(t) * n_out + k) * 2 + 1];
      Vh[static_cast<size_t>(t) * D + i] = half_to_double(v);
    }
    if (t < nb * sh.Bk) {
      const int b = t / sh.Bk;
      const uint8_t* kr = k_codes + static_cast<size_t>(t) * rb;
      for (int c = 0; c < D; ++c) {
        const double s = half_to_double(k_meta[(static_cast<size_t>(b) * D + c) * 2 + 0]);
        const double z = half_to_double(k_meta[(static_cast<size_t>(b) * D + c) * 2 + 1]);
        Kh[static_cast<size_t>(t) * D + c] = value(unpack_one(kr, c, bits), s, z);
      }
      for (int k = 0; k < n_out; ++k) {
        const uint16_t i = k_outl[(static_cast<size_t>(t) * n_out + k) * 2 + 0];
        const uint16_t v = k_outl[(static_cast<size_t>(t) * n_out + k) * 2 + 1];
        Kh[static_cast<size_t>(t) * D + i] = half_to_double(v);
      }
    } else {
      for (int c = 0; c < D; ++c)
        Kh[static_cast<size_t>(t) * D + c] =
            half_to_double(k_tail[static_cast<size_t>(t - nb * sh.Bk) * D + c]);
    }
  }
}

// Rotary embedding, rotate-half pairing (i, i + D/2), angle pos * theta^(-2i/D).
void rope(const double* x, int D, double pos, double theta, double* y) {
  const int h = D / 2;
  for (int i = 0; i < h; ++i) {
    const double phi = pos * std::pow(theta, -2.0 * i / D);
    const double c = std::cos(phi), s = std::sin(phi);
    y[i] = x[i] * c - x[i + h] * s;
    y[i + h] = x[i + h] * c + x[i] * s;
  }
}

// Exact (binary64) softmax attention of G query heads over one stream.
void attention_stream(int T, int D, int G, const double* Kh, const double* Vh, const uint16_t* q,
                      double q_pos, double pos_offset, double theta, double sm_scale, double* out) {
  std::vector<double> qr(D), kr(D), sc(T), qd(D);
  std::vector<double> Krot(static_cast<size_t>(T) * D);
  for (int t = 0; t < T; ++t) {
    if (theta > 0.0)
      rope(Kh + static_cast<size_t>(t) * D, D, t + pos_offset, theta, &Krot[static_cast<size_t>(t) * D]);
    else
      std::memcpy(&Krot[static_cast<size_t>(t) * D], Kh + static_cast<size_t>(t) * D, sizeof(double) * D);
  }
  for (int h = 0; h < G; ++h) {
    for (int d = 0; d < D; ++d) qd[d] = half_to_double(q[static_cast<size_t>(h) * D + d]);
    if (theta > 0.0)
      rope(qd.data(), D, q_pos + pos_offset, theta, qr.data());
    else
      qr = qd;
    double mx = -INFINITY;
    for (int t = 0; t < T; ++t) {
      double acc = 0.0;
      for (int d = 0; d < D; ++d) acc += qr[d] * Krot[static_cast<size_t>(t) * D + d];
      sc[t] = sm_scale * acc;
      mx = std::max(mx, sc[t]);
    }
    double den = 0.0;
    for (int t = 0; t < T; ++t) {
      sc[t] = std::exp(sc[t] - mx);
      den += sc[t];
    }
    for (int d = 0; d < D; ++d) {
      double acc = 0.0;
      for (int t = 0; t < T; ++t) acc += sc[t] * Vh[static_cast<size_t>(t) * D + d];
      out[static_cast<size_t>(h) * D + d] = acc / den;
    }
  }
}

template <typename F>
void parallel_for(int n, int nthreads, F f) {
  if (nthreads <= 1 || n <= 1) {
    for (int i = 0; i < n; ++i) f(i);
    return;
  }
  std::vector<std::thread> pool;
  const int nt = std::min(n, nthreads);
  for (int w = 0; w < nt; ++w)
    pool.emplace_back([=, &f]() {
      for (int i = w; i < n; i += nt) f(i);
    });
  for (auto& th : pool) th.join();
}

bool shape_ok(int T, int D, int bits, int Bk, int Gv, int n_out) {
  if (T < 0 || D <= 0 || D % 2 || Bk <= 0 || Gv <= 0 || D % Gv) return false;
  if (bits < 1 || bits > 8 || (D * bits) % 8) return false;
  if (n_out < 0 || n_out > D) return false;
  return true;
}

}  // namespace

extern "C" {

int kvqo_encode_levels(int P, int T, int D, int bits, int Bk, int Gv, int n_out, const uint16_t* K,
                       const uint16_t* V, uint8_t* k_codes, uint16_t* k_meta, uint16_t* k_tail,
                       uint16_t* k_outl, uint8_t* v_codes, uint16_t* v_meta, uint16_t* v_outl,
                       const float* levels, int nthreads);
int kvqo_dequant_levels(int P, int T, int D, int bits, int Bk, int Gv, int n_out, const uint8_t* k_codes,
                        const uint16_t* k_meta, const uint16_t* k_tail, const uint16_t* k_outl,
                        const uint8_t* v_codes, const uint16_t* v_meta, const uint16_t* v_outl,
                        double* Kh, double* Vh, const float* levels, int nthreads);

int kvqo_encode(int P, int T, int D, int bits, int Bk, int Gv, int n_out, const uint16_t* K,
                const uint16_t* V, uint8_t* k_codes, uint16_t* k_meta, uint16_t* k_tail,
                uint16_t* k_outl, uint8_t* v_codes, uint16_t* v_meta, uint16_t* v_outl,
                int nthreads) {
  return kvqo_encode_levels(P, T, D, bits, Bk, Gv, n_out, K, V, k_codes, k_meta, k_tail, k_outl, v_codes,
                            v_meta, v_outl, nullptr, nthreads);
}

int kvqo_encode_window(int P, int T, int D, int bits, int Bk, int Gv, int n_out, int window,
                       const uint16_t* K, const uint16_t* V, uint8_t* k_codes, uint16_t* k_meta,
                       uint16_t* k_tail, uint16_t* k_outl, uint8_t* v_codes, uint16_t* v_meta,
                       uint16_t* v_outl, const float* levels, int nthreads);

// levels: 2^bits sorted binary32 levels (non-uniform codes) or NULL (uniform).
int kvqo_encode_levels(int P, int T, int D, int bits, int Bk, int Gv, int n_out, const uint16_t* K,
                       const uint16_t* V, uint8_t* k_codes, uint16_t* k_meta, uint16_t* k_tail,
                       uint16_t* k_outl, uint8_t* v_codes, uint16_t* v_meta, uint16_t* v_outl,
                       const float* levels, int nthreads) {
  return kvqo_encode_window(P, T, D, bits, Bk, Gv, n_out, Bk, K, V, k_codes, k_meta, k_tail, k_outl, v_codes,
                            v_meta, v_outl, levels, nthreads);
}

// window: key statistics over the last `window` tokens (a positive multiple
// of Bk; Bk is the per-block rule); uniform grid only when window > Bk.
int kvqo_encode_window(int P, int T, int D, int bits, int Bk, int Gv, int n_out, int window,
                       const uint16_t* K, const uint16_t* V, uint8_t* k_codes, uint16_t* k_meta,
                       uint16_t* k_tail, uint16_t* k_outl, uint8_t* v_codes, uint16_t* v_meta,
                       uint16_t* v_outl, const float* levels, int nthreads) {
  if (!shape_ok(T, D, bits, Bk, Gv, n_out) || P < 0) return 1;
  if (window < Bk || window % Bk || (levels && window != Bk)) return 1;
  const Shape sh{T, D, bits, Bk, Gv, n_out};
  const size_t td = static_cast<size_t>(T) * D;
  const size_t rows = static_cast<size_t>(T) * sh.row_bytes();
  const size_t km = static_cast<size_t>(sh.n_full()) * D * 2;
  const size_t kt = static_cast<size_t>(Bk) * D;
  const size_t ol = static_cast<size_t>(T) * n_out * 2;
  const size_t vm = static_cast<size_t>(T) * (D / Gv) * 2;
  parallel_for(P, nthreads, [&](int p) {
    std::memset(k_codes + p * rows, 0, rows);
    std::memset(k_outl + p * ol, 0, ol * sizeof(uint16_t));
    std::memset(k_tail + p * kt, 0, kt * sizeof(uint16_t));
    encode_stream(sh, K + p * td, V + p * td, k_codes + p * rows, k_meta + p * km, k_tail + p * kt,
                  k_outl + p * ol, v_codes + p * rows, v_meta + p * vm, v_outl + p * ol, levels, window);
  });
  return 0;
}

int kvqo_dequant(int P, int T, int D, int bits, int Bk, int Gv, int n_out, const uint8_t* k_codes,
                 const uint16_t* k_meta, const uint16_t* k_tail, const uint16_t* k_outl,
                 const uint8_t* v_codes, const uint16_t* v_meta, const uint16_t* v_outl,
                 double* Kh, double* Vh, int nthreads) {
  return kvqo_dequant_levels(P, T, D, bits, Bk, Gv, n_out, k_codes, k_meta, k_tail, k_outl, v_codes, v_meta,
                             v_outl, Kh, Vh, nullptr, nthreads);
}

int kvqo_dequant_levels(int P, int T, int D, int bits, int Bk, int Gv, int n_out, const uint8_t* k_codes,
                        const uint16_t* k_meta, const uint16_t* k_tail, const uint16_t* k_outl,
                        const uint8_t* v_codes, const uint16_t* v_meta, const uint16_t* v_outl,
                        double* Kh, double* Vh, const float* levels, int nthreads) {
  if (!shape_ok(T, D, bits, Bk, Gv, n_out) || P < 0) return 1;
  const Shape sh{T, D, bits, Bk, Gv, n_out};
  const size_t td = static_cast<size_t>(T) * D;
  const size_t rows = static_cast<size_t>(T) * sh.row_bytes();
  const size_t km = static_cast<size_t>(sh.n_full()) * D * 2;
  const size_t kt = static_cast<size_t>(Bk) * D;
  const size_t ol = static_cast<size_t>(T) * n_out * 2;
  const size_t vm = static_cast<size_t>(T) * (D / Gv) * 2;
  parallel_for(P, nthreads, [&](int p) {
    dequant_stream(sh, k_codes + p * rows, k_meta + p * km, k_tail + p * kt, k_outl + p * ol,
                   v_codes + p * rows, v_meta + p * vm, v_outl + p * ol, Kh + p * td, Vh + p * td, levels);
  });
  return 0;
}

int kvqo_attention(int P, int T, int D, int G, const double* Kh, const double* Vh,
                   const uint16_t* q, double q_pos, double pos_offset, double theta,
                   double sm_scale, double* out, int nthreads) {
  if (P < 0 || T <= 0 || D <= 0 || D % 2 || G <= 0) return 1;
  const size_t td = static_cast<size_t>(T) * D;
  const size_t gd = static_cast<size_t>(G) * D;
  parallel_for(P, nthreads, [&](int p) {
    attention_stream(T, D, G, Kh + p * td, Vh + p * td, q + p * gd, q_pos, pos_offset, theta,
                     sm_scale, out + p * gd);
  });
  return 0;
}

// Single-step entry points, used by the pins.
int kvqo_select_outliers(int D, const uint16_t* x, int n_out, uint16_t* idx, uint16_t* val) {
  if (D <= 0 || n_out < 0 || n_out > D) return 1;
  select_outliers(x, D, n_out, idx, val);
  return 0;
}

int kvqo_group_params(int n, const uint16_t* x, const uint8_t* excluded, int bits, uint16_t* s,
                      uint16_t* z) {
  std::vector<uint16_t> dense;
  for (int i = 0; i < n; ++i)
    if (!excluded || !excluded[i]) dense.push_back(x[i]);
  group_params(dense, bits, s, z);
  return 0;
}

int kvqo_quantize(int n, const uint16_t* x, uint16_t s, uint16_t z, int bits, int* codes) {
  for (int i = 0; i < n; ++i) codes[i] = quantize_one(x[i], s, z, bits);
  return 0;
}

int kvqo_group_params_levels(int n, const uint16_t* x, const uint8_t* excluded, uint16_t* r, uint16_t* z) {
  std::vector<uint16_t> dense;
  for (int i = 0; i < n; ++i)
    if (!excluded || !excluded[i]) dense.push_back(x[i]);
  group_params_nuq(dense, r, z);
  return 0;
}

int kvqo_quantize_levels(int n, const uint16_t* x, uint16_t r, uint16_t z, int bits, const float* levels,
                         int* codes) {
  const std::vector<float> mids = level_mids(levels, (1 << bits) - 1);
  for (int i = 0; i < n; ++i) codes[i] = quantize_nuq(x[i], r, z, mids);
  return 0;
}

int kvqo_fit_levels(size_t n, const double* u, int bits, int iters, float* levels) {
  if (bits < 1 || bits > 8 || iters < 0) return 1;
  nuq_fit(u, n, bits, iters, levels);
  return 0;
}

uint16_t kvqo_half_up(float x) { return float_to_half_up(x); }

double kvqo_half_to_double(uint16_t h) { return half_to_double(h); }

int kvqo_pack_row(int D, const int* codes, int bits, uint8_t* out) {
  if ((D * bits) % 8) return 1;
  pack_row(codes, D, bits, out);
  return 0;
}

int kvqo_rope(int D, const double* x, double pos, double theta, double* y) {
  if (D % 2) return 1;
  rope(x, D, pos, theta, y);
  return 0;
}

}  // extern "C"
