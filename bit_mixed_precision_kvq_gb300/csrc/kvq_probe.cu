// kvq_probe.cu -- kvq_sensitivity_probe: how far quantising K or V moves
// attention, measured on one layer's cache.
//
// "VLM_KV_Quantization" (nuiw.github.io), sections 3-4: quantisation damage
// is read as the KL divergence of the distribution after quantisation from
// the unquantised one, with visual K or visual V quantised alone (same
// tokens, bits, group size).  Restated without a model, per (b, hq):
//   kl_attn = D_KL(p || p_hat): softmax weights over positions, from the raw
//             bf16 K (p) and from K as the decode reads it (p_hat);
//   kl_out  = D_KL(P || P_hat): P = softmax(R o), o the attention output
//             over the raw K/V, P_hat the same over the cache, R a readout
//             matrix given by the caller (it stands for the layers after
//             attention);
//   err     = ||o_hat - o||_2.
// "As the decode reads it" = the dequantised value code * s + z of a packed
// row (the fp16 scale/zero widened), or the bf16 row of the side store.
//
// Everything is fp64.  With p_t = e^{s_t - lse}:
//   D_KL(p || p_hat) = sum_t p_t (s_t - s_hat_t) - lse + lse_hat,
// so one pass over the positions keeps, for both score streams, an online
// softmax state (max m, sum l, output o) plus A = sum e^{s - m} (s - s_hat).
//
// Two kernels.  probe_partial: grid (S, rows); each of a CTA's 4 warps
// takes every 4th batch of 32 positions of the CTA's slice of the row's
// positions (lane j scores position j of a batch; the output sums run with
// lane l owning elements 4l .. 4l + 3) and writes its own partial state.
// probe_finish: one CTA per row merges the row's 4 S partials and evaluates
// the divergences, the error and the readout.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "kvq_device.cuh"

namespace kvq {
namespace {

constexpr int kProbeWarps = 4;
constexpr int kProbeThreads = 32 * kProbeWarps;
constexpr int kProbeMaxOut = 2048;     // readout rows (fp64 logits of both sides in shared memory)
constexpr int kProbeCTAsTarget = 608;  // 4 CTAs of 128 threads per SM on 152 SMs
constexpr int kProbeMinPos = 128;      // positions per CTA at least (one batch of 32 per warp)

// One warp's partial state: m, l, A (exact side), m_hat, l_hat, then o[kD]
// and o_hat[kD].
constexpr int kPartDoubles = 8 + 2 * kD;

struct ProbeArgs {
  Params p;
  const uint16_t* kin;  // raw bf16 K and V, element strides sb, sh, st
  const uint16_t* vin;
  int64_t sb, sh, st;
  int32_t T, S;
  double scale;
  const float* R;  // readout [n_out][kD]
  int32_t n_out;
  double* part;    // [rows][S * kProbeWarps][kPartDoubles]
  double* result;  // [rows][3]
};

// Storage slot of element d in a packed row (the order include/kvq.h
// documents).  K: d = 32P + 8t + 4e + i; V: d = 16m + 8r + n.
__device__ __forceinline__ int stored_slot(bool is_v, int bits, int d) {
  if (is_v) return 16 * (d & 7) + 2 * (d >> 4) + ((d >> 3) & 1);
  const int P = d >> 5, t = (d >> 3) & 3, e = (d >> 2) & 1, i = d & 3;
  if (bits == 2) {  // crumb c of the pair: (4, 7), (3, 6), (2, 5), (0, 1) for P = 0 .. 3
    const int c = (i & 1) ? (P < 3 ? 7 - P : 1) : (P < 3 ? 4 - P : 0);
    return 32 * t + 16 * (i >> 1) + 8 * e + c;
  }
  if (bits == 4) return 32 * t + 8 * i + 4 * e + P;
  return 32 * t + 4 * (2 * P + (i >> 1)) + 2 * e + (i & 1);
}

// bf16 -> fp64 by assembling the fp64 bit pattern with integer operations
// (GB300 issues fp64 arithmetic and conversions at 1/64 of the fp32 rate):
// sign, exponent rebiased by 1023 - 127, mantissa shifted; zero, infinity
// and NaN keep their meaning; a bf16 subnormal takes the conversion path.
__device__ __forceinline__ double bf16d(uint16_t h) {
  const uint32_t e = (h >> 7) & 0xffu, m = h & 0x7fu;
  if (e == 0u && m != 0u) return static_cast<double>(__uint_as_float(static_cast<uint32_t>(h) << 16));
  const uint32_t ed = e == 0u ? 0u : (e == 0xffu ? 0x7ffu : e + 896u);
  const uint32_t hi = (static_cast<uint32_t>(h & 0x8000u) << 16) | (ed << 20) | (m << 13);
  return __hiloint2double(static_cast<int>(hi), 0);
}
__device__ __forceinline__ double f16d(uint16_t h) {
  return static_cast<double>(__half2float(__ushort_as_half(h)));
}

// 4 consecutive bf16 values d0 .. d0 + 3 of a row.
__device__ __forceinline__ void load4_bf16(const uint8_t* row, int d0, double (&x)[4]) {
  const uint2 w = *reinterpret_cast<const uint2*>(row + 2 * d0);
  x[0] = bf16d(static_cast<uint16_t>(w.x & 0xffffu));
  x[1] = bf16d(static_cast<uint16_t>(w.x >> 16));
  x[2] = bf16d(static_cast<uint16_t>(w.y & 0xffffu));
  x[3] = bf16d(static_cast<uint16_t>(w.y >> 16));
}

// Elements d0 .. d0 + 3 of a packed row: code * s + z (ctab[c] = c as fp64,
// a shared-memory table).
__device__ __forceinline__ void load4_packed(const uint8_t* codes, const uint8_t* sz, bool is_v, int bits,
                                             int G, int d0, const double* ctab, double (&x)[4]) {
  const int per_word = 32 / bits;
  const uint32_t mask = (1u << bits) - 1u;
  const uint16_t* szh = reinterpret_cast<const uint16_t*>(sz);
  const int ng = kD / G;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int d = d0 + j;
    const int s = stored_slot(is_v, bits, d);
    const uint32_t w = reinterpret_cast<const uint32_t*>(codes)[s / per_word];
    const uint32_t c = (w >> (bits * (s % per_word))) & mask;
    const int g = d / G;
    x[j] = ctab[c] * f16d(szh[ng + g]) + f16d(szh[g]);
  }
}

// Elements 4 lane .. 4 lane + 3 of K (is_v = false) or V at position t of
// (b, h), as the decode reads them.
__device__ __forceinline__ void load4_cached(const Params& p, bool is_v, int b, int h, int t, int lane,
                                             const double* ctab, double (&x)[4]) {
  const int d0 = 4 * lane;
  if (t < p.vs || t >= p.ve) {
    const int tr = t < p.vs ? t : t - p.Tv;
    const int64_t row = (static_cast<int64_t>(b) * p.Hkv + h) * p.T_text + tr;
    load4_bf16(p.seg[is_v ? KVQ_SEG_TEXT_V : KVQ_SEG_TEXT_K] + row * (2 * kD), d0, x);
    return;
  }
  const int mode = p.prot[h], slot = p.slot[h], r = t - p.vs;
  if (!is_v && mode != 0) {
    const int64_t row = prot_k_row(p, b, mode == 1 ? kClsProt : kClsKonly, slot) * p.Tv + r;
    load4_bf16(p.seg[KVQ_SEG_PROT_K] + row * (2 * kD), d0, x);
    return;
  }
  if (is_v && mode == 1) {
    const int64_t row = (static_cast<int64_t>(b) * p.n_prot + slot) * p.Tv + r;
    load4_bf16(p.seg[KVQ_SEG_PROT_V] + row * (2 * kD), d0, x);
    return;
  }
  const int64_t row = is_v ? packed_v_row(p, b, mode == 2 ? kClsKonly : kClsPacked, slot) * p.Tv_pad + r
                           : (static_cast<int64_t>(b) * p.n_packed + slot) * p.Tv_pad + r;
  const int bits = is_v ? p.vb : p.kb;
  const uint8_t* codes = p.seg[is_v ? KVQ_SEG_V_CODES : KVQ_SEG_K_CODES] + row * (is_v ? p.vrow : p.krow);
  if (bits == 16) {
    load4_bf16(codes, d0, x);
    return;
  }
  const uint8_t* sz = p.seg[is_v ? KVQ_SEG_V_SZ : KVQ_SEG_K_SZ] + row * (is_v ? p.vszrow : p.kszrow);
  load4_packed(codes, sz, is_v, bits, p.G, d0, ctab, x);
}

__device__ __forceinline__ double warp_sum(double x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// q . x for a bf16 row x (16-byte aligned), with four independent partial
// sums (a single chain of dependent fp64 FMAs would leave the FP64 pipe idle
// for most of its latency).
__device__ __forceinline__ double dot_bf16_row(const double* sq, const uint8_t* row) {
  double acc[4] = {0.0, 0.0, 0.0, 0.0};
#pragma unroll 2
  for (int d0 = 0; d0 < kD; d0 += 8) {
    const uint4 w = *reinterpret_cast<const uint4*>(row + 2 * d0);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc[e] = fma(sq[d0 + 2 * e], bf16d(static_cast<uint16_t>(ws[e] & 0xffffu)), acc[e]);
      acc[e] = fma(sq[d0 + 2 * e + 1], bf16d(static_cast<uint16_t>(ws[e] >> 16)), acc[e]);
    }
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// Scores of one position for the lane that owns it: s = q . k (raw bf16 K
// row) and s_hat = q . k_hat (K as the decode reads it), both unscaled.
// A packed K row is summed per group as s_g * sum_g q c + z_g * sum_g q.
__device__ __forceinline__ void position_scores(const Params& p, const double* sq, const double* sQ,
                                                const double* ctab, const uint16_t* kraw, int b, int h, int t,
                                                double& s, double& sh) {
  s = dot_bf16_row(sq, reinterpret_cast<const uint8_t*>(kraw));
  // where the decode reads this K row
  const uint8_t* bf = nullptr;
  if (t < p.vs || t >= p.ve) {
    const int tr = t < p.vs ? t : t - p.Tv;
    bf = p.seg[KVQ_SEG_TEXT_K] + ((static_cast<int64_t>(b) * p.Hkv + h) * p.T_text + tr) * (2 * kD);
  } else if (p.prot[h] != 0) {
    const int64_t row = prot_k_row(p, b, p.prot[h] == 1 ? kClsProt : kClsKonly, p.slot[h]) * p.Tv + (t - p.vs);
    bf = p.seg[KVQ_SEG_PROT_K] + row * (2 * kD);
  }
  const int64_t prow = (static_cast<int64_t>(b) * p.n_packed + p.slot[h]) * p.Tv_pad + (t - p.vs);
  if (!bf && p.kb == 16) bf = p.seg[KVQ_SEG_K_CODES] + prow * p.krow;
  if (bf) {
    sh = dot_bf16_row(sq, bf);
    return;
  }
  const int bits = p.kb, per_word = 32 / bits, ng = kD / p.G;
  const uint32_t mask = (1u << bits) - 1u;
  const uint32_t* codes = reinterpret_cast<const uint32_t*>(p.seg[KVQ_SEG_K_CODES] + prow * p.krow);
  const uint16_t* sz = reinterpret_cast<const uint16_t*>(p.seg[KVQ_SEG_K_SZ] + prow * p.kszrow);
  sh = 0.0;
  for (int g = 0; g < ng; ++g) {
    double pg[4] = {0.0, 0.0, 0.0, 0.0};
    for (int d = g * p.G; d < (g + 1) * p.G; d += 4) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int sl = stored_slot(false, bits, d + e);
        const uint32_t c = (codes[sl / per_word] >> (bits * (sl % per_word))) & mask;
        pg[e] = fma(sq[d + e], ctab[c], pg[e]);
      }
    }
    sh += f16d(sz[ng + g]) * ((pg[0] + pg[1]) + (pg[2] + pg[3])) + f16d(sz[g]) * sQ[g];
  }
}

__device__ __forceinline__ double warp_max(double x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = fmax(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}

__global__ void __launch_bounds__(kProbeThreads) probe_partial(const __grid_constant__ ProbeArgs a) {
  __shared__ double sq[kD];      // q of the row
  __shared__ double sQ[kD / 32]; // its group sums (G >= 32)
  __shared__ double ctab[256];   // code -> fp64
  const Params& p = a.p;
  const int row = blockIdx.y;  // b * Hq + hq
  const int b = row / p.Hq, hq = row - (row / p.Hq) * p.Hq;
  const int h = hq / p.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = (a.T + a.S - 1) / a.S;
  const int t_begin = blockIdx.x * chunk, t_end = min(a.T, t_begin + chunk);
  sq[threadIdx.x] = bf16d(p.q[static_cast<int64_t>(row) * kD + threadIdx.x]);  // kProbeThreads == kD
  ctab[threadIdx.x] = static_cast<double>(threadIdx.x);
  ctab[threadIdx.x + kProbeThreads] = static_cast<double>(threadIdx.x + kProbeThreads);
  __syncthreads();
  if (threadIdx.x < kD / p.G) {
    double x = 0.0;
    for (int d = threadIdx.x * p.G; d < (threadIdx.x + 1) * p.G; ++d) x += sq[d];
    sQ[threadIdx.x] = x;
  }
  __syncthreads();

  // Batches of 32 positions per warp: lane j scores position tb + j, the
  // online softmax takes the batch at once (one exp per lane and side), and
  // the output sums run with lane l owning elements 4l .. 4l + 3.
  double m = -INFINITY, l = 0.0, A = 0.0, mh = -INFINITY, lh = 0.0;
  double o[4] = {0.0, 0.0, 0.0, 0.0}, oh[4] = {0.0, 0.0, 0.0, 0.0};
  for (int tb = t_begin + 32 * warp; tb < t_end; tb += 32 * kProbeWarps) {
    const int t = tb + lane;
    const bool valid = t < t_end;
    double s = -INFINITY, sh = -INFINITY;
    if (valid) {
      position_scores(p, sq, sQ, ctab, a.kin + b * a.sb + h * a.sh + t * a.st, b, h, t, s, sh);
      s *= a.scale;
      sh *= a.scale;
    }
    const double mn = fmax(m, warp_max(s)), mhn = fmax(mh, warp_max(sh));
    const double c = exp(m - mn), ch = exp(mh - mhn);  // m = -inf: 0
    const double w = valid ? exp(s - mn) : 0.0, wh = valid ? exp(sh - mhn) : 0.0;
    l = l * c + warp_sum(w);
    A = A * c + warp_sum(valid ? w * (s - sh) : 0.0);
    lh = lh * ch + warp_sum(wh);
    m = mn;
    mh = mhn;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      o[e] *= c;
      oh[e] *= ch;
    }
    const int nb = min(32, t_end - tb);
    for (int j = 0; j < nb; ++j) {
      const double wj = __shfl_sync(0xffffffffu, w, j), whj = __shfl_sync(0xffffffffu, wh, j);
      const int tj = tb + j;
      double v[4], vh[4];
      load4_bf16(reinterpret_cast<const uint8_t*>(a.vin + b * a.sb + h * a.sh + tj * a.st), 4 * lane, v);
      load4_cached(p, true, b, h, tj, lane, ctab, vh);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o[e] += wj * v[e];
        oh[e] += whj * vh[e];
      }
    }
  }
  double* out = a.part + (static_cast<int64_t>(row) * a.S * kProbeWarps + blockIdx.x * kProbeWarps + warp) *
                             kPartDoubles;
  if (lane == 0) {
    out[0] = m;
    out[1] = l;
    out[2] = A;
    out[3] = mh;
    out[4] = lh;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    out[8 + 4 * lane + e] = o[e];
    out[8 + kD + 4 * lane + e] = oh[e];
  }
}

// Block-wide sum / max over the 128 threads (every thread gets the result).
template <bool kMax>
__device__ __forceinline__ double block_reduce(double x, double* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const double y = __shfl_xor_sync(0xffffffffu, x, off);
    x = kMax ? fmax(x, y) : x + y;
  }
  __syncthreads();  // red[] may still be read by a previous reduction
  if (lane == 0) red[warp] = x;
  __syncthreads();
  double r = red[0];
#pragma unroll
  for (int w = 1; w < kProbeWarps; ++w) r = kMax ? fmax(r, red[w]) : r + red[w];
  return r;
}

__global__ void __launch_bounds__(kProbeThreads) probe_finish(const __grid_constant__ ProbeArgs a) {
  extern __shared__ double zbuf[];  // z[n_out], z_hat[n_out]
  __shared__ double so[kD], soh[kD];
  __shared__ double red[kProbeWarps];
  const int row = blockIdx.x;
  const int d = threadIdx.x;  // one output element per thread (kD == 128 threads)
  const int np = a.S * kProbeWarps;
  const double* part = a.part + static_cast<int64_t>(row) * np * kPartDoubles;
  double M = -INFINITY, Mh = -INFINITY;
  for (int j = 0; j < np; ++j) {
    M = fmax(M, part[j * kPartDoubles + 0]);
    Mh = fmax(Mh, part[j * kPartDoubles + 3]);
  }
  double L = 0.0, A = 0.0, O = 0.0, Lh = 0.0, Oh = 0.0;
  for (int j = 0; j < np; ++j) {
    const double* q = part + j * kPartDoubles;
    if (q[0] != -INFINITY) {
      const double c = exp(q[0] - M);
      L += q[1] * c;
      A += q[2] * c;
      O += q[8 + d] * c;
    }
    if (q[3] != -INFINITY) {
      const double c = exp(q[3] - Mh);
      Lh += q[4] * c;
      Oh += q[8 + kD + d] * c;
    }
  }
  O /= L;
  Oh /= Lh;
  so[d] = O;
  soh[d] = Oh;
  const double kl_attn = A / L - (M + log(L)) + (Mh + log(Lh));
  const double err2 = block_reduce<false>((Oh - O) * (Oh - O), red);  // also publishes so / soh
  // readout logits z = R o, z_hat = R o_hat
  double zmax = -INFINITY, zhmax = -INFINITY;
  for (int i = threadIdx.x; i < a.n_out; i += kProbeThreads) {
    const float* r = a.R + static_cast<int64_t>(i) * kD;
    double za[2] = {0.0, 0.0}, zha[2] = {0.0, 0.0};  // two chains per side (FP64 latency)
#pragma unroll 4
    for (int e = 0; e < kD; e += 2) {
      const float2 w2 = *reinterpret_cast<const float2*>(r + e);
      za[0] = fma(static_cast<double>(w2.x), so[e], za[0]);
      za[1] = fma(static_cast<double>(w2.y), so[e + 1], za[1]);
      zha[0] = fma(static_cast<double>(w2.x), soh[e], zha[0]);
      zha[1] = fma(static_cast<double>(w2.y), soh[e + 1], zha[1]);
    }
    const double z = za[0] + za[1], zh = zha[0] + zha[1];
    zbuf[i] = z;
    zbuf[a.n_out + i] = zh;
    zmax = fmax(zmax, z);
    zhmax = fmax(zhmax, zh);
  }
  zmax = block_reduce<true>(zmax, red);
  zhmax = block_reduce<true>(zhmax, red);
  double se = 0.0, seh = 0.0;
  for (int i = threadIdx.x; i < a.n_out; i += kProbeThreads) {
    se += exp(zbuf[i] - zmax);
    seh += exp(zbuf[a.n_out + i] - zhmax);
  }
  const double lse = zmax + log(block_reduce<false>(se, red));
  const double lseh = zhmax + log(block_reduce<false>(seh, red));
  double acc = 0.0;
  for (int i = threadIdx.x; i < a.n_out; i += kProbeThreads) {
    const double z = zbuf[i], zh = zbuf[a.n_out + i];
    acc += exp(z - lse) * (z - zh);
  }
  const double kl_out = block_reduce<false>(acc, red) - lse + lseh;
  if (threadIdx.x == 0) {
    a.result[3 * static_cast<int64_t>(row) + 0] = kl_attn;
    a.result[3 * static_cast<int64_t>(row) + 1] = kl_out;
    a.result[3 * static_cast<int64_t>(row) + 2] = sqrt(err2);
  }
}

// Splits per row: enough CTAs to fill the GPU, at least kProbeMinPos
// positions each.
int probe_splits(int64_t rows, int32_t T) {
  int64_t s = (kProbeCTAsTarget + rows - 1) / rows;
  const int64_t cap = (T + kProbeMinPos - 1) / kProbeMinPos;
  if (s > cap) s = cap;
  if (s < 1) s = 1;
  return static_cast<int>(s);
}

}  // namespace
}  // namespace kvq

extern "C" size_t kvq_probe_workspace_bytes(const kvq_layout* L, int32_t T) {
  if (kvq_check_layout(L) != KVQ_OK || T < 1) return 0;
  const int64_t rows = static_cast<int64_t>(L->d.B) * L->d.H_q;
  return static_cast<size_t>(rows * kvq::probe_splits(rows, T) * kvq::kProbeWarps * kvq::kPartDoubles * 8);
}

extern "C" kvq_status kvq_sensitivity_probe(const kvq_layout* L, const void* cache, const void* q_bf16,
                                            const void* k_bf16, const void* v_bf16, int64_t stride_b,
                                            int64_t stride_h, int64_t stride_t, int32_t T,
                                            float softmax_scale, const float* readout, int32_t n_out,
                                            double* result, void* workspace, size_t ws_bytes,
                                            void* stream) {
  const kvq_status st = kvq_check_layout(L);
  if (st != KVQ_OK) return st;
  if (L->d.D != kvq::kD) return KVQ_ERR_UNSUPPORTED;
  if (!cache || !q_bf16 || !k_bf16 || !v_bf16 || !readout || !result || !workspace)
    return KVQ_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(cache) % 256 || reinterpret_cast<uintptr_t>(q_bf16) % 16 ||
      reinterpret_cast<uintptr_t>(k_bf16) % 16 || reinterpret_cast<uintptr_t>(v_bf16) % 16 ||
      reinterpret_cast<uintptr_t>(readout) % 8 || reinterpret_cast<uintptr_t>(result) % 8 ||
      reinterpret_cast<uintptr_t>(workspace) % 16)
    return KVQ_ERR_INVALID_ARG;
  if (stride_b % 8 || stride_h % 8 || stride_t % 8 || stride_b < 0 || stride_h < 0 || stride_t < 0)
    return KVQ_ERR_INVALID_ARG;
  if (T < 1 || T > L->d.T_cap) return KVQ_ERR_INVALID_ARG;
  if (n_out < 1 || n_out > kvq::kProbeMaxOut) return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  if (ws_bytes < kvq_probe_workspace_bytes(L, T)) return KVQ_ERR_CAPACITY;
  static kvq::ProbeArgs a;  // large (Params): off the host stack
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  a = kvq::ProbeArgs{};
  kvq_fill_params(L, &a.p);
  const uint8_t* base = static_cast<const uint8_t*>(cache);
  for (int s = 0; s < KVQ_NSEG; ++s) a.p.seg[s] = base + L->off[s];
  a.p.q = static_cast<const uint16_t*>(q_bf16);
  a.kin = static_cast<const uint16_t*>(k_bf16);
  a.vin = static_cast<const uint16_t*>(v_bf16);
  a.sb = stride_b;
  a.sh = stride_h;
  a.st = stride_t;
  a.T = T;
  const int64_t rows = static_cast<int64_t>(L->d.B) * L->d.H_q;
  a.S = kvq::probe_splits(rows, T);
  a.scale = static_cast<double>(softmax_scale);
  a.R = readout;
  a.n_out = n_out;
  a.part = static_cast<double*>(workspace);
  a.result = result;
  if (rows == 0) return KVQ_OK;
  if (rows > 65535) return KVQ_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  kvq::probe_partial<<<dim3(a.S, static_cast<unsigned>(rows)), kvq::kProbeThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return kvq_cuda_fail(e);
  kvq::probe_finish<<<static_cast<unsigned>(rows), kvq::kProbeThreads, 2 * n_out * sizeof(double), s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return kvq_cuda_fail(e);
  return KVQ_OK;
}
