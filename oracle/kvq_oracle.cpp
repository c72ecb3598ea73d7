// kvq_oracle.cpp -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, CPU restatement of what the compressed-KV decode path
// computes.  Only the test suite, the smoke check and the benchmark's CPU
// baseline leg may load this library; the product library never does, and
// this file shares no code, header or table with it.
//
// Sources (the four pages the method is described on):
//   [VKQ]  "VLM_KV_Quantization" (nuiw.github.io): intro checklist, §1
//          (what was measured: FP16/INT8/INT4/INT2 on the historical cache,
//          Visual/Text and K/V split), §2 (cache shape [B, H_kv, T, D],
//          K stored after RoPE, GQA 28/4), §4 (K and V quantised
//          independently with the same token set, bits and group size).
//   [HG]   HeadGuard news brief (jiinsi.com, "KV 캐시 양자화의 딜레마"):
//          bullet list of the key ideas -- about 1/8 of the physical KV heads
//          keep their image K (and, as needed, V) in bf16; composable with any
//          low-bit KV quantiser.
//   [WSVD] gist.science summary of WSVD, §2.라 (fused kernel): reconstruct
//          K/V on chip and feed QK, softmax and PV directly.
//
// Readings taken where the pages are silent:
//   * the quantiser is group-wise asymmetric min-max along D with a float
//     zero equal to the group minimum, scale = (max-min)/(2^b-1), both
//     stored as IEEE binary16;
//   * a group minimum of -0 is taken as +0 (signed zeros compare equal);
//   * codes are computed with the STORED fp16 scale and zero, in fp32:
//     u = (x - z) / s (separate round-to-nearest subtraction and IEEE
//     division), code = clamp(rint_half_even(u), 0, 2^b-1); a group whose
//     stored scale is 0 gets all-zero codes;
//   * packing: a sequence of codes goes to 32-bit words little-endian, code
//     j to word j / (32/b) at bit offset b * (j mod (32/b)); bits == 16
//     means the row is kept as bf16;
//   * storage order (the cache layout of this library, not a page's): a
//     packed K or V row holds element d at sequence slot sigma(d), defined
//     in include/kvq.h and restated in oracle_code_slot below; the stored
//     scale/zero row is [z_0 .. z_{D/G-1}, s_0 .. s_{D/G-1}];
//   * a position is quantised iff it lies in the visual range, its KV head
//     is not protected and the tensor's bit-width is below 16;
//   * query head hq reads KV head hq / (H_q / H_kv);
//   * attention is exact softmax(scale * q . k) . v in fp64 over the
//     dequantised cache (dequantised value = code * s + z in fp64).
//
// Everything floating point below is plain IEEE arithmetic; the library is
// compiled with -ffp-contract=off so that no multiply-add is fused.
//
// ORACLE_PLANT (default 0) selects one deliberate mistake; non-zero values are
// built only by the test that checks each pin catches a plausible error.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>
#include <limits>

#if defined(__linux__)
#include <sched.h>
#endif

#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

namespace {

uint32_t float_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}

float bits_float(uint32_t u) {
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------

// bfloat16 -> float: the bf16 pattern is the upper half of the binary32 one.
float oracle_bf16_to_f32(uint16_t b) { return bits_float(static_cast<uint32_t>(b) << 16); }

// binary16 -> float, exact (every binary16 value is a binary32 value).
float oracle_f16_to_f32(uint16_t h) {
  const uint32_t sign = (h & 0x8000u) ? 1u : 0u;
  const int e = (h >> 10) & 0x1f;
  const uint32_t m = h & 0x3ffu;
  float mag;
  if (e == 0x1f) {
    mag = m ? std::numeric_limits<float>::quiet_NaN() : std::numeric_limits<float>::infinity();
  } else if (e == 0) {
    mag = std::ldexp(static_cast<float>(m), -24);  // subnormal: m * 2^-24
  } else {
    mag = std::ldexp(static_cast<float>(m | 0x400u), e - 25);  // (1.m) * 2^(e-15)
  }
  return sign ? -mag : mag;
}

// float -> binary16 with round-to-nearest, ties to even (IEEE 754 default),
// including gradual underflow and overflow to infinity.
uint16_t oracle_f32_to_f16(float x) {
  const uint32_t u = float_bits(x);
  const uint16_t sign = static_cast<uint16_t>((u >> 16) & 0x8000u);
  const uint32_t a = u & 0x7fffffffu;
  if (a >= 0x7f800000u) {  // inf / nan
    return static_cast<uint16_t>(sign | 0x7c00u | (a > 0x7f800000u ? 0x200u : 0u));
  }
  // 65520 = 0x477ff000 is the midpoint between 65504 (odd mantissa) and 2^16:
  // ties go to even, i.e. to 2^16, which is infinity in binary16.
  if (a >= 0x477ff000u) return static_cast<uint16_t>(sign | 0x7c00u);
  const int e = static_cast<int>(a >> 23) - 127;
  if (e >= -14) {  // normal binary16
    uint32_t h = (static_cast<uint32_t>(e + 15) << 10) | ((a & 0x7fffffu) >> 13);
    const uint32_t rest = a & 0x1fffu;
#if ORACLE_PLANT == 7
    (void)rest;  // planted: truncate instead of rounding
#else
    if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1;  // carry may bump the exponent
#endif
    return static_cast<uint16_t>(sign | h);
  }
  if (a < 0x00800000u) return sign;  // binary32 subnormal: far below 2^-25
  // subnormal binary16: result = round(|x| / 2^-24)
  const uint32_t mant = (a & 0x7fffffu) | 0x800000u;  // |x| = mant * 2^(e-23)
  const int shift = -(e + 1);                          // |x| / 2^-24 = mant >> shift
  if (shift > 24) return sign;
  uint32_t q = mant >> shift;
  const uint32_t rest = mant & ((1u << shift) - 1u);
  const uint32_t half = 1u << (shift - 1);
  if (rest > half || (rest == half && (q & 1u))) q += 1;
  return static_cast<uint16_t>(sign | q);
}

// ---------------------------------------------------------------------------
// The quantiser ([VKQ] §1/§4: INT8/INT4/INT2 with a group size; K and V each
// with their own bit-width).
// ---------------------------------------------------------------------------

// Quantise one row of D bf16 values in groups of G consecutive elements.
// codes[D]: one code per element; s_bits/z_bits[D/G]: binary16 scale and zero.
// Returns 0 on success, -1 on bad arguments.
int oracle_quantize_row(const uint16_t* x, int D, int G, int bits, uint8_t* codes,
                        uint16_t* s_bits, uint16_t* z_bits) {
  if (!x || !codes || !s_bits || !z_bits) return -1;
  if (!(bits == 2 || bits == 4 || bits == 8)) return -1;
  if (G <= 0 || D <= 0 || D % G != 0) return -1;
#if ORACLE_PLANT == 9
  const int qmax = (1 << bits);  // planted: wrong number of steps
#else
  const int qmax = (1 << bits) - 1;
#endif
  for (int g = 0; g < D / G; ++g) {
    float mn = oracle_bf16_to_f32(x[g * G]);
    float mx = mn;
    for (int i = 1; i < G; ++i) {
      const float v = oracle_bf16_to_f32(x[g * G + i]);
      if (v < mn) mn = v;
      if (v > mx) mx = v;
    }
    // Signed zeros compare equal, so "the minimum" of a group holding both
    // -0 and +0 has no defined sign; adding +0 maps -0 to +0 and leaves every
    // other value unchanged, so the stored zero never depends on scan order.
    mn = mn + 0.0f;
    const float range = mx - mn;                              // fp32, round to nearest
    const float s32 = range / static_cast<float>(qmax);       // fp32 IEEE division
    const uint16_t sh = oracle_f32_to_f16(s32);
    const uint16_t zh = oracle_f32_to_f16(mn);
    s_bits[g] = sh;
    z_bits[g] = zh;
    const float sf = oracle_f16_to_f32(sh);
    const float zf = oracle_f16_to_f32(zh);
    for (int i = 0; i < G; ++i) {
      int c = 0;
      if (sf != 0.0f) {
        const float v = oracle_bf16_to_f32(x[g * G + i]);
        const float diff = v - zf;           // fp32 subtraction
        const float u = diff / sf;           // fp32 IEEE division
#if ORACLE_PLANT == 2
        float r = std::floor(u);             // planted: truncation
#else
        float r = std::nearbyint(u);         // default rounding mode: half to even
#endif
        if (r < 0.0f) r = 0.0f;
        if (r > static_cast<float>(qmax)) r = static_cast<float>(qmax);
        c = static_cast<int>(r);
      }
      codes[g * G + i] = static_cast<uint8_t>(c);
    }
  }
  return 0;
}

// Pack D codes of `bits` bits into 32-bit words: element d -> word d/(32/bits),
// bit offset bits*(d mod (32/bits)).  words must hold D*bits/32 entries.
int oracle_pack_row(const uint8_t* codes, int D, int bits, uint32_t* words) {
  if (!codes || !words) return -1;
  if (!(bits == 2 || bits == 4 || bits == 8)) return -1;
  const int per = 32 / bits;
  if (D % per != 0) return -1;
  for (int w = 0; w < D / per; ++w) words[w] = 0;
  for (int d = 0; d < D; ++d) {
#if ORACLE_PLANT == 4
    words[d / per] |= static_cast<uint32_t>(codes[d]) << (bits * (per - 1 - d % per));  // planted
#else
    words[d / per] |= static_cast<uint32_t>(codes[d]) << (bits * (d % per));
#endif
  }
  return 0;
}

// Many rows at once: quantise + pack n_rows rows of D values.
// words[n_rows][D*bits/32], s_bits/z_bits[n_rows][D/G].
int oracle_quantize_pack_rows(const uint16_t* x, int64_t n_rows, int D, int G, int bits,
                              uint32_t* words, uint16_t* s_bits, uint16_t* z_bits) {
  std::vector<uint8_t> codes(D);
  const int W = D * bits / 32;
  for (int64_t r = 0; r < n_rows; ++r) {
    if (oracle_quantize_row(x + r * D, D, G, bits, codes.data(), s_bits + r * (D / G),
                            z_bits + r * (D / G)) != 0)
      return -1;
    if (oracle_pack_row(codes.data(), D, bits, words + r * W) != 0) return -1;
  }
  return 0;
}

// Storage slot of element d (D = 128) in a packed row of the cache, kind 0
// = K, 1 = V (the layout documented in include/kvq.h, restated here from
// that definition).  K: d = 32P + 8t + 4e + i with P, t, i in [0,4) and e in
// {0,1};  V: d = 16m + 8r + n with m, n in [0,8) and r in {0,1}.  Returns -1
// for an unsupported argument.
int oracle_code_slot(int kind, int bits, int d) {
  if (d < 0 || d >= 128 || !(bits == 2 || bits == 4 || bits == 8)) return -1;
  if (kind == 1) {
    const int m = d / 16, r = (d / 8) % 2, n = d % 8;
    return 16 * n + 2 * m + r;
  }
  if (kind != 0) return -1;
  const int P = d / 32, t = (d / 8) % 4, e = (d / 4) % 2, i = d % 4;
  if (bits == 2) {
    // crumb of register (P, i mod 2) inside its half-word
    static const int crumb[4][2] = {{4, 7}, {3, 6}, {2, 5}, {0, 1}};
#if ORACLE_PLANT == 10
    return 32 * t + 16 * (i / 2) + 8 * e + crumb[P][(i + 1) % 2];  // planted: members swapped
#else
    return 32 * t + 16 * (i / 2) + 8 * e + crumb[P][i % 2];
#endif
  }
  if (bits == 4) return 32 * t + 8 * i + 4 * e + P;
  return 32 * t + 4 * (2 * P + i / 2) + 2 * e + i % 2;
}

// Quantise and pack n_rows rows of D = 128 values in the cache's storage
// order: words[n_rows][D*bits/32] (slot sequence of oracle_code_slot) and the
// stored scale/zero rows sz[n_rows][2*D/G] = [z_0.., s_0..].
int oracle_quantize_pack_rows_stored(const uint16_t* x, int64_t n_rows, int D, int G, int bits,
                                     int kind, uint32_t* words, uint16_t* sz) {
  if (D != 128 || G <= 0 || D % G != 0) return -1;
  std::vector<uint8_t> codes(D), slotted(D);
  std::vector<uint16_t> s(D / G), z(D / G);
  const int W = D * bits / 32, ng = D / G;
  for (int64_t r = 0; r < n_rows; ++r) {
    if (oracle_quantize_row(x + r * D, D, G, bits, codes.data(), s.data(), z.data()) != 0) return -1;
    for (int d = 0; d < D; ++d) {
      const int j = oracle_code_slot(kind, bits, d);
      if (j < 0) return -1;
      slotted[j] = codes[d];
    }
    if (oracle_pack_row(slotted.data(), D, bits, words + r * W) != 0) return -1;
    for (int g = 0; g < ng; ++g) {
      sz[r * 2 * ng + g] = z[g];
      sz[r * 2 * ng + ng + g] = s[g];
    }
  }
  return 0;
}

// Dequantise in fp64: x_hat = code * s + z.
void oracle_dequant_row(const uint8_t* codes, const uint16_t* s_bits, const uint16_t* z_bits,
                        int D, int G, double* out) {
  for (int d = 0; d < D; ++d) {
    const double s = static_cast<double>(oracle_f16_to_f32(s_bits[d / G]));
    const double z = static_cast<double>(oracle_f16_to_f32(z_bits[d / G]));
#if ORACLE_PLANT == 1
    (void)z;
    out[d] = static_cast<double>(codes[d]) * s;  // planted: zero term dropped
#else
    out[d] = static_cast<double>(codes[d]) * s + z;
#endif
  }
}

// Which positions are quantised ([VKQ] intro checklist and §1: only the
// historical visual block; [HG]: protected heads stay bf16).
int oracle_is_packed(int p, int vis_start, int vis_end, int head_protected, int bits) {
#if ORACLE_PLANT == 5
  (void)head_protected;
  return (p >= vis_start && p < vis_end && bits < 16) ? 1 : 0;  // planted: protection ignored
#elif ORACLE_PLANT == 6
  return (p >= vis_start && p <= vis_end && !head_protected && bits < 16) ? 1 : 0;  // planted
#else
  return (p >= vis_start && p < vis_end && !head_protected && bits < 16) ? 1 : 0;
#endif
}

// Reconstruct what the decode step reads for one tensor (K or V):
// x bf16 [B, H, T, D] -> out fp64 [B, H, T, D].  Packed positions go
// through quantise -> dequantise, all others are the bf16 value widened.
// prot[H]: 1 = protected head.  Also reports the number of packed rows.
int oracle_reconstruct(const uint16_t* x, int B, int H, int T, int D, int vis_start,
                       int vis_end, const uint8_t* prot, int bits, int G, double* out,
                       int64_t* n_packed_rows) {
  if (!x || !out || !prot) return -1;
  if (bits != 16 && (D % G != 0)) return -1;
  std::vector<uint8_t> codes(D);
  std::vector<uint16_t> s(D), z(D);
  int64_t packed = 0;
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h)
      for (int t = 0; t < T; ++t) {
        const int64_t row = ((static_cast<int64_t>(b) * H + h) * T + t) * D;
        if (oracle_is_packed(t, vis_start, vis_end, prot[h], bits)) {
          if (oracle_quantize_row(x + row, D, G, bits, codes.data(), s.data(), z.data()) != 0)
            return -1;
          oracle_dequant_row(codes.data(), s.data(), z.data(), D, G, out + row);
          ++packed;
        } else {
          for (int d = 0; d < D; ++d) out[row + d] = static_cast<double>(oracle_bf16_to_f32(x[row + d]));
        }
      }
  if (n_packed_rows) *n_packed_rows = packed;
  return 0;
}

// Number of host threads this process may run on.
int oracle_online_cores(void) {
#if defined(__linux__)
  cpu_set_t set;
  CPU_ZERO(&set);
  if (sched_getaffinity(0, sizeof(set), &set) == 0) {
    const int n = CPU_COUNT(&set);
    if (n > 0) return n;
  }
#endif
  const unsigned n = std::thread::hardware_concurrency();
  return n ? static_cast<int>(n) : 1;
}

// Exact softmax attention in fp64 for one decode query per sequence.
//   q     bf16 [B, Hq, D]
//   khat  fp64 [B, Hkv, T, D]  (dequantised cache, e.g. from oracle_reconstruct)
//   vhat  fp64 [B, Hkv, T, D]
//   out   fp64 [B, Hq, D];  lse fp64 [B, Hq] (natural log), may be null
// Query head hq uses KV head hq / (Hq / Hkv).  threads <= 0: all online cores.
int oracle_attention(const uint16_t* q, const double* khat, const double* vhat, int B, int Hq,
                     int Hkv, int T, int D, double scale, double* out, double* lse, int threads) {
  if (!q || !khat || !vhat || !out) return -1;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || T <= 0 || D <= 0) return -1;
  const int g = Hq / Hkv;
  const int64_t jobs = static_cast<int64_t>(B) * Hq;
  if (threads <= 0) threads = oracle_online_cores();
  if (threads > jobs) threads = static_cast<int>(jobs > 0 ? jobs : 1);

  auto one = [&](int64_t job) {
    const int b = static_cast<int>(job / Hq);
    const int hq = static_cast<int>(job % Hq);
#if ORACLE_PLANT == 3
    const int h = hq % Hkv;  // planted: interleaved instead of contiguous grouping
    (void)g;
#else
    const int h = hq / g;
#endif
    const uint16_t* qv = q + (static_cast<int64_t>(b) * Hq + hq) * D;
    const double* K = khat + (static_cast<int64_t>(b) * Hkv + h) * T * D;
    const double* V = vhat + (static_cast<int64_t>(b) * Hkv + h) * T * D;
    std::vector<double> qd(D), sc(T);
    for (int d = 0; d < D; ++d) qd[d] = static_cast<double>(oracle_bf16_to_f32(qv[d]));
    double m = -std::numeric_limits<double>::infinity();
    for (int t = 0; t < T; ++t) {
      double acc = 0.0;
      for (int d = 0; d < D; ++d) acc += qd[d] * K[static_cast<int64_t>(t) * D + d];
#if ORACLE_PLANT == 8
      sc[t] = acc;  // planted: softmax scale dropped
#else
      sc[t] = scale * acc;
#endif
      if (sc[t] > m) m = sc[t];
    }
    double den = 0.0;
    for (int t = 0; t < T; ++t) {
      sc[t] = std::exp(sc[t] - m);
      den += sc[t];
    }
    double* o = out + (static_cast<int64_t>(b) * Hq + hq) * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int t = 0; t < T; ++t) {
      const double w = sc[t] / den;
      for (int d = 0; d < D; ++d) o[d] += w * V[static_cast<int64_t>(t) * D + d];
    }
    if (lse) lse[static_cast<int64_t>(b) * Hq + hq] = m + std::log(den);
  };

  if (threads <= 1) {
    for (int64_t j = 0; j < jobs; ++j) one(j);
    return 0;
  }
  std::vector<std::thread> pool;
  for (int w = 0; w < threads; ++w) {
    pool.emplace_back([&, w]() {
      for (int64_t j = w; j < jobs; j += threads) one(j);
    });
  }
  for (auto& th : pool) th.join();
  return 0;
}

// Softmax weights of one (b, hq) query, for the sum-to-one pin.
int oracle_attention_weights(const uint16_t* q, const double* khat, int Hq, int Hkv, int T,
                             int D, int hq, double scale, double* w) {
  if (!q || !khat || !w || Hq % Hkv != 0 || hq < 0 || hq >= Hq || T <= 0) return -1;
  const int h = hq / (Hq / Hkv);
  const uint16_t* qv = q + static_cast<int64_t>(hq) * D;
  const double* K = khat + static_cast<int64_t>(h) * T * D;
  double m = -std::numeric_limits<double>::infinity();
  for (int t = 0; t < T; ++t) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d)
      acc += static_cast<double>(oracle_bf16_to_f32(qv[d])) * K[static_cast<int64_t>(t) * D + d];
    w[t] = scale * acc;
    if (w[t] > m) m = w[t];
  }
  double den = 0.0;
  for (int t = 0; t < T; ++t) {
    w[t] = std::exp(w[t] - m);
    den += w[t];
  }
  for (int t = 0; t < T; ++t) w[t] /= den;
  return 0;
}

}  // extern "C"
