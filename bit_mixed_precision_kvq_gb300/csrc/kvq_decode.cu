// kvq_decode.cu -- kvq_decode_attention: split-KV flash decoding over the
// mixed-precision cache, plus the cross-split log-sum-exp combine.
//
// Method sources: WSVD summary (gist.science 2604.02570), section 2.라 --
// K/V are rebuilt on chip inside a flash-decoding pipeline and used at once
// for QK, softmax and PV, with no reconstructed tensor written back to
// device memory; "VLM_KV_Quantization", section 2 -- GQA cache
// [B, H_kv, T, D] read by H_q / H_kv query heads per KV head.
//
// Softmax runs in base 2: q is pre-multiplied by softmax_scale * log2(e), so
// a partial holds m = max score (log2 units), l = sum 2^(s - m) and
// o = sum 2^(s - m) v.  The combine merges partials with the usual rescaling
// and reports lse = ln(2) * (M + log2 L).
#include <cuda_runtime.h>

#include <cmath>

#include "kvq_device.cuh"

namespace kvq {

// ---------------------------------------------------------------------------
// Combine: one CTA per (b, hq), one thread per d.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) combine_kernel(Params p) {
  const int bq = blockIdx.x;
  const int b = bq / p.Hq;
  const int hq = bq - b * p.Hq;
  const int h = hq / p.g;
  const int r = hq - h * p.g;
  const int hc = r / kNH;
  const int j = r - hc * kNH;
  const int u = unit_of(p, b, h, hc);
  int cf, cl;
  plan_unit_chunks(p.plan, u, &cf, &cl);
  const int d = threadIdx.x;
  float M = -INFINITY;
  for (int c = cf; c <= cl; ++c) M = fmaxf(M, p.ws_ml[(static_cast<int64_t>(u + c) * kNH + j) * 2]);
  float L = 0.0f, O = 0.0f;
  for (int c = cf; c <= cl; ++c) {
    const int64_t s = static_cast<int64_t>(u + c) * kNH + j;
    const float m = p.ws_ml[s * 2];
    if (m == -INFINITY) continue;
    const float w = exp2f(m - M);
    L = fmaf(w, p.ws_ml[s * 2 + 1], L);
    O = fmaf(w, p.ws_o[s * kD + d], O);
  }
  p.out[static_cast<int64_t>(bq) * kD + d] = f32_to_bf16_bits(O / L);
  if (d == 0 && p.lse) p.lse[bq] = 0.69314718055994531f * (M + log2f(L));
}

namespace {

// ---------------------------------------------------------------------------
// Simple split kernel: 8 warps, one position per warp per step, lanes over D.
// ---------------------------------------------------------------------------

// Lane's 4 elements (d = 4*lane .. 4*lane+3) of one K or V row, as fp32.
__device__ __forceinline__ void load4(const uint8_t* row, const uint8_t* sz, int bits, int G, int lane,
                                      float out[4]) {
  if (bits == 16) {
    const uint2 w = *reinterpret_cast<const uint2*>(row + 8 * lane);
    out[0] = bf16_lo(w.x);
    out[1] = bf16_hi(w.x);
    out[2] = bf16_lo(w.y);
    out[3] = bf16_hi(w.y);
    return;
  }
  const int d0 = 4 * lane;
  const uint32_t word = reinterpret_cast<const uint32_t*>(row)[(d0 * bits) >> 5];
  const int shift = (d0 * bits) & 31;
  const __half2 szv = reinterpret_cast<const __half2*>(sz)[d0 / G];
  const float s = __low2float(szv), z = __high2float(szv);
  const uint32_t mask = (1u << bits) - 1u;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t c = (word >> (shift + i * bits)) & mask;
    out[i] = fmaf(static_cast<float>(c), s, z);
  }
}

constexpr int kWarpsSimple = 8;

__global__ void __launch_bounds__(256) split_simple_kernel(Params p) {
  __shared__ float sm_ml[kWarpsSimple][kNH][2];
  __shared__ float sm_o[kWarpsSimple][kNH][kD];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int c = blockIdx.x;
  const Cut a = plan_cut(p.plan, c);
  const Cut e = plan_cut(p.plan, c + 1);
  const int u_last = e.u < p.plan.U ? e.u : p.plan.U - 1;
  for (int u = a.u; u <= u_last; ++u) {
    const int ps = (u == a.u) ? a.p : 0;
    const int pe = (u == e.u) ? e.p : p.plan.T;
    const UnitInfo ui = unit_info(p, u);
    const int hq0 = ui.h * p.g + ui.hc * kNH;
    const int nh = min(kNH, p.g - ui.hc * kNH);
    float q[kNH][4];
#pragma unroll
    for (int j = 0; j < kNH; ++j) {
      if (j < nh) {
        const uint2 w = *reinterpret_cast<const uint2*>(
            p.q + (static_cast<int64_t>(ui.b) * p.Hq + hq0 + j) * kD + 4 * lane);
        q[j][0] = bf16_lo(w.x) * p.scale_log2;
        q[j][1] = bf16_hi(w.x) * p.scale_log2;
        q[j][2] = bf16_lo(w.y) * p.scale_log2;
        q[j][3] = bf16_hi(w.y) * p.scale_log2;
      } else {
        q[j][0] = q[j][1] = q[j][2] = q[j][3] = 0.0f;
      }
    }
    float m[kNH], l[kNH], o[kNH][4];
#pragma unroll
    for (int j = 0; j < kNH; ++j) {
      m[j] = -INFINITY;
      l[j] = 0.0f;
      o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;
    }
    for (int pos = ps + warp; pos < pe; pos += kWarpsSimple) {
      const RowRef rr = row_ref(p, ui, pos);
      float k[4], v[4];
      load4(rr.k, rr.ksz, rr.kbits, p.G, lane, k);
      load4(rr.v, rr.vsz, rr.vbits, p.G, lane, v);
#pragma unroll
      for (int j = 0; j < kNH; ++j) {
        if (j >= nh) break;
        float s = q[j][0] * k[0] + q[j][1] * k[1] + q[j][2] * k[2] + q[j][3] * k[3];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        const float mn = fmaxf(m[j], s);
        const float corr = exp2f(m[j] - mn);
        const float pj = exp2f(s - mn);
        l[j] = fmaf(l[j], corr, pj);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[j][i] = fmaf(o[j][i], corr, pj * v[i]);
        m[j] = mn;
      }
    }
#pragma unroll
    for (int j = 0; j < kNH; ++j) {
      if (lane == 0) {
        sm_ml[warp][j][0] = m[j];
        sm_ml[warp][j][1] = l[j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) sm_o[warp][j][4 * lane + i] = o[j][i];
    }
    __syncthreads();
    const int64_t slot = static_cast<int64_t>(u) + c;
    for (int idx = threadIdx.x; idx < nh * kD; idx += blockDim.x) {
      const int j = idx / kD, d = idx - j * kD;
      float M = -INFINITY;
      for (int w = 0; w < kWarpsSimple; ++w) M = fmaxf(M, sm_ml[w][j][0]);
      float L = 0.0f, O = 0.0f;
      if (M != -INFINITY) {
        for (int w = 0; w < kWarpsSimple; ++w) {
          const float sc = exp2f(sm_ml[w][j][0] - M);
          L = fmaf(sm_ml[w][j][1], sc, L);
          O = fmaf(sm_o[w][j][d], sc, O);
        }
      }
      p.ws_o[(slot * kNH + j) * kD + d] = O;
      if (d == 0) {
        p.ws_ml[(slot * kNH + j) * 2] = M;
        p.ws_ml[(slot * kNH + j) * 2 + 1] = L;
      }
    }
    __syncthreads();
  }
}

}  // namespace
}  // namespace kvq

extern "C" kvq_status kvq_decode_attention(const kvq_layout* L, const void* cache, const void* q_bf16,
                                           int32_t T, float softmax_scale, void* out_bf16, float* lse,
                                           void* workspace, size_t ws_bytes, void* stream) {
  const kvq_status st = kvq_check_layout(L);
  if (st != KVQ_OK) return st;
  if (!cache || !q_bf16 || !out_bf16 || !workspace) return KVQ_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(cache) % 256 || reinterpret_cast<uintptr_t>(workspace) % 256 ||
      reinterpret_cast<uintptr_t>(q_bf16) % 16 || reinterpret_cast<uintptr_t>(out_bf16) % 16 ||
      reinterpret_cast<uintptr_t>(lse) % 4)
    return KVQ_ERR_INVALID_ARG;
  if (T < 1 || T > L->d.T_cap) return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  if (ws_bytes < static_cast<size_t>(L->workspace_bytes)) return KVQ_ERR_CAPACITY;
  int n_sm = 0;
  if (kvq_device_sm_count(&n_sm) != 0) return KVQ_ERR_CUDA;

  kvq::Params p;
  kvq_fill_params(L, &p);
  const uint8_t* base = static_cast<const uint8_t*>(cache);
  for (int s = 0; s < KVQ_NSEG; ++s) p.seg[s] = base + L->off[s];
  p.T = T;
  p.q = static_cast<const uint16_t*>(q_bf16);
  p.out = static_cast<uint16_t*>(out_bf16);
  p.lse = lse;
  const int64_t slots = static_cast<int64_t>(L->units) + KVQ_MAX_CTAS - 1;
  p.ws_o = static_cast<float*>(workspace);
  const int64_t o_bytes = (slots * kvq::kNH * kvq::kD * 4 + 255) / 256 * 256;
  p.ws_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + o_bytes);
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.plan = kvq_make_plan(L, T, 2 * n_sm);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  kvq::split_simple_kernel<<<p.plan.C, 256, 0, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  kvq::combine_kernel<<<L->d.B * L->d.H_q, kvq::kD, 0, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}
