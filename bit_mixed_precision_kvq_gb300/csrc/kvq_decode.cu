// kvq_decode.cu -- kvq_decode_attention: host launcher for the split-KV
// partial kernel (kvq_split.cuh) and the cross-split log-sum-exp combine.
//
// Method sources: WSVD summary (gist.science 2604.02570), section 2.라 --
// K/V are rebuilt on chip inside a flash-decoding pipeline and used at once
// for QK, softmax and PV, with no reconstructed tensor written back to
// device memory; "VLM_KV_Quantization", section 2 -- GQA cache
// [B, H_kv, T, D] read by H_q / H_kv query heads per KV head.
//
// Softmax runs in base 2: scores are scaled by softmax_scale * log2(e), so a
// partial holds m = max score (log2 units), l = sum 2^(s - m) and
// o = sum 2^(s - m) v.  The combine merges partials with the usual rescaling
// and reports lse = ln(2) * (M + log2 L).
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "kvq_device.cuh"
#include "kvq_ptx.cuh"
#include "kvq_split.cuh"

namespace kvq {

const void* split_kernel_k2(int vb, int G);
const void* split_kernel_k4(int vb, int G);
const void* split_kernel_k8(int vb, int G);
const void* split_kernel_k16(int vb, int G);

constexpr int kCombineWarps = 16;

// ---------------------------------------------------------------------------
// Combine: one CTA per (b, hq).  16 warps fold the unit's partial slots with
// an online rescaling; the warp states are merged in shared memory.  Lane l
// owns d = 4l .. 4l+3.  A NaN partial max (a failed wait in the split kernel)
// turns the output into NaN.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const __grid_constant__ Params p) {
  __shared__ float sm_ml[kCombineWarps][2];
  __shared__ float4 sm_o[kCombineWarps][32];
  __shared__ int sm_bad;
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bq = blockIdx.x;
  const int b = bq / p.Hq;
  const int hq = bq - b * p.Hq;
  const int h = hq / p.g;
  const int r = hq - h * p.g;
  const int hc = r / kNH;
  const int j = r - hc * kNH;
  const int u = unit_of(p, b, h, hc);
  int cf, cl;
  plan_unit_chunks(p.plan, p.cuts, u, &cf, &cl);
  if (threadIdx.x == 0) sm_bad = 0;
  __syncthreads();
  float M = -INFINITY, L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  bool bad = false;
  // Warp w folds slots cf + 8w + {0..7}, then the next 8 * kCombineWarps;
  // the eight loads of a batch are issued before any of them is used.
  for (int c0 = cf + 8 * warp; c0 <= cl; c0 += 8 * kCombineWarps) {
    float mb[8], lb[8];
    float4 ob[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      mb[k] = -INFINITY;
      lb[k] = 0.f;
      ob[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c0 + k <= cl) {
        const int64_t s = static_cast<int64_t>(u + c0 + k) * kNH + j;
        mb[k] = p.ws_ml[s * 2];
        lb[k] = p.ws_ml[s * 2 + 1];
        ob[k] = reinterpret_cast<const float4*>(p.ws_o + s * kD)[lane];
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float m = mb[k];
      if (m != m) bad = true;
      if (m == -INFINITY || m != m) continue;
      const float Mn = fmaxf(M, m);
      const float a = exp2f(M - Mn), w = exp2f(m - Mn);
      L = L * a + lb[k] * w;
      O.x = O.x * a + ob[k].x * w;
      O.y = O.y * a + ob[k].y * w;
      O.z = O.z * a + ob[k].z * w;
      O.w = O.w * a + ob[k].w * w;
      M = Mn;
    }
  }
  if (bad) sm_bad = 1;
  if (lane == 0) {
    sm_ml[warp][0] = M;
    sm_ml[warp][1] = L;
  }
  sm_o[warp][lane] = O;
  __syncthreads();
  if (warp != 0) return;
  float Mt = -INFINITY;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) Mt = fmaxf(Mt, sm_ml[w][0]);
  float Lt = 0.f;
  float4 Ot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) {
    if (sm_ml[w][0] == -INFINITY) continue;
    const float sc = exp2f(sm_ml[w][0] - Mt);
    Lt = fmaf(sm_ml[w][1], sc, Lt);
    const float4 o = sm_o[w][lane];
    Ot.x = fmaf(o.x, sc, Ot.x);
    Ot.y = fmaf(o.y, sc, Ot.y);
    Ot.z = fmaf(o.z, sc, Ot.z);
    Ot.w = fmaf(o.w, sc, Ot.w);
  }
  float inv = 1.0f / Lt;
  if (sm_bad) inv = __int_as_float(0x7fffffff);
  uint2 packed;
  packed.x = static_cast<uint32_t>(f32_to_bf16_bits(Ot.x * inv)) |
             (static_cast<uint32_t>(f32_to_bf16_bits(Ot.y * inv)) << 16);
  packed.y = static_cast<uint32_t>(f32_to_bf16_bits(Ot.z * inv)) |
             (static_cast<uint32_t>(f32_to_bf16_bits(Ot.w * inv)) << 16);
  reinterpret_cast<uint2*>(p.out + static_cast<int64_t>(bq) * kD)[lane] = packed;
  if (lane == 0 && p.lse) p.lse[bq] = sm_bad ? inv : 0.69314718055994531f * (Mt + log2f(Lt));
}

}  // namespace kvq

namespace {

// Positions per packed tile and its sub-buffer offsets inside one stage.
void packed_tile_geometry(kvq::Params* p) {
  const int w = p->krow + p->kszrow + p->vrow + p->vszrow;
  int tt = ((kvq::kStageBytes - 4 * 128) / w) / 32 * 32;  // whole 32-position blocks
  if (tt > 512) tt = 512;
  auto r128 = [](int x) { return (x + 127) / 128 * 128; };
  p->tt_pk = tt;
  p->pk_off_vc = r128(tt * p->krow);
  p->pk_off_ksz = p->pk_off_vc + r128(tt * p->vrow);
  p->pk_off_vsz = p->pk_off_ksz + r128(tt * p->kszrow);
}

const void* split_kernel_for(int kb, int vb, int G) {
  switch (kb) {
    case 2: return kvq::split_kernel_k2(vb, G);
    case 4: return kvq::split_kernel_k4(vb, G);
    case 8: return kvq::split_kernel_k8(vb, G);
    case 16: return kvq::split_kernel_k16(vb, G);
  }
  return nullptr;
}

// One CTA per SM: the stage ring, merge buffers and barriers must fit the
// 227 KiB a CTA may use.
constexpr size_t kSplitSmemBytes = sizeof(kvq::SplitSmem);
static_assert(kSplitSmemBytes <= 232448, "split kernel shared memory exceeds one CTA's limit");

}  // namespace

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
  const void* split = split_kernel_for(L->d.k_bits, L->d.v_bits, L->d.group_size);
  if (!split) return KVQ_ERR_UNSUPPORTED;
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
  packed_tile_geometry(&p);
  p.plan = kvq_make_plan(L, T, n_sm);  // one CTA per SM
  for (int c = 0; c <= p.plan.C; ++c) p.cuts[c] = kvq::plan_cut(p.plan, c);

  // Opt each split kernel into >48 KB of dynamic shared memory, once.
  static std::mutex mu;
  static bool smem_set[17][17][3] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    bool& done = smem_set[L->d.k_bits][L->d.v_bits][L->d.group_size == 32 ? 0 : (L->d.group_size == 64 ? 1 : 2)];
    if (!done) {
      const cudaError_t e = cudaFuncSetAttribute(split, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(kSplitSmemBytes));
      if (e != cudaSuccess) return kvq_cuda_fail(e);
      cudaFuncAttributes fa;
      const cudaError_t e2 = cudaFuncGetAttributes(&fa, split);
      if (e2 != cudaSuccess) return kvq_cuda_fail(e2);
      if (fa.maxThreadsPerBlock < kvq::kSplitThreads) return kvq_cuda_fail(cudaErrorLaunchOutOfResources);
      done = true;
    }
  }
  if (kvq_launch_pdl(split, p.plan.C, kvq::kSplitThreads, kSplitSmemBytes, stream, &p) != 0)
    return KVQ_ERR_CUDA;
  if (kvq_launch_pdl(reinterpret_cast<const void*>(&kvq::combine_kernel), L->d.B * L->d.H_q,
                     kvq::kCombineWarps * 32, 0, stream, &p) != 0)
    return KVQ_ERR_CUDA;
  return KVQ_OK;
}
