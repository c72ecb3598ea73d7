// kvq_decode.cu -- the decode entry points (kvq_decode_attention and its
// ragged and multi-query forms, kvq_decode_step and its ragged form): argument
// checks, the work plan, and the launches of the split-KV kernel
// (kvq_split.cuh) and, for the two-call forms, the cross-split log-sum-exp
// combine.
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

#include <algorithm>
#include <cmath>
#include <atomic>
#include <mutex>

#include "kvq_device.cuh"
#include "kvq_ptx.cuh"
#include "kvq_mq_umma.cuh"
#include "kvq_split.cuh"

namespace kvq {

const void* split_kernel_k2(int vb, int G, bool step, int halves, bool general);
const void* split_kernel_k4(int vb, int G, bool step, int halves, bool general);
const void* split_kernel_k8(int vb, int G, bool step, int halves, bool general);
const void* split_kernel_k16(int vb, int G, bool step, int halves, bool general);
const void* split_kernel_cl_k2(int vb, int G, bool step, int halves, bool general);
const void* split_kernel_cl_k4(int vb, int G, bool step, int halves, bool general);
const void* split_kernel_cl_k8(int vb, int G, bool step, int halves, bool general);
const void* split_kernel_cl_k16(int vb, int G, bool step, int halves, bool general);
const void* mq_umma_kernel_k2(int vb, int G);
const void* mq_umma_kernel_k4(int vb, int G);
const void* mq_umma_kernel_k8(int vb, int G);
const void* mq_umma_kernel_k16(int vb, int G);

// Combine: one CTA per output row (b, token i, hq), NW warps (combine_row):
// 16 when some unit has many chunks, 2 when every unit has at most 16 (the
// two warps fold them in one pass, and many more rows are resident at once).
template <int NW>
__global__ void __launch_bounds__(NW * 32) combine_kernel(const __grid_constant__ Params p) {
  __shared__ float sm_ml[NW][2];
  __shared__ float4 sm_o[NW][32];
  const int bq = blockIdx.x;  // (b * n_q + i) * Hq + hq
  const int bi = bq / p.Hq;
  const int hq = bq - bi * p.Hq;
  const int b = bi / p.n_q, i = bi - (bi / p.n_q) * p.n_q;
  const int h = hq / p.g;
  const int c = (hq - h * p.g) * p.n_q + i;  // column among the KV head's g * n_q
  const int hc = c / kNH;
  const int u = unit_of(p, b, h, hc);
  int cf, cl;
  plan_unit_chunks(p.plan, p.cuts, u, &cf, &cl);
  pdl_wait();
  combine_row<NW>(p, u, c - hc * kNH, cf, cl, bq, threadIdx.x >> 5, threadIdx.x & 31, sm_ml, sm_o, false,
                  []() { __syncthreads(); });
}

}  // namespace kvq

namespace {

// Positions per packed tile and its sub-buffer offsets inside one stage.
// 64-position packed blocks only when packed chunks are long (>= 1024
// positions: enough blocks for every consumer warp); else 32.
int packed_halves(const kvq::Plan& P, const kvq_layout* L, int n_q) {
  if (L->n_konly > 0 || n_q > 1) return 2;  // the general kernels: 32-position blocks only
  if (kvq::packed_block_halves(L->d.k_bits, L->d.v_bits, L->d.group_size) < 4) return 2;
  const int64_t per_chunk = P.aligned ? P.T / (P.n_q > 0 ? P.n_q : 1) : P.T;
  return per_chunk >= 1024 ? 4 : 2;
}

// K-only tiles: bf16 K rows, then the packed V rows and their scale/zero.
void konly_tile_geometry(kvq::Params* p) {
  const int w = 2 * kvq::kD + p->vrow + p->vszrow;
  const int tt = kvq::packed_tile_rows32(w);
  auto r128 = [](int x) { return (x + 127) / 128 * 128; };
  p->tt_ko = tt;
  p->ko_off_vc = r128(tt * 2 * kvq::kD);
  p->ko_off_vsz = p->ko_off_vc + r128(tt * p->vrow);
}

void packed_tile_geometry(kvq::Params* p) {
  const int w = p->krow + p->kszrow + p->vrow + p->vszrow;
  int tt = kvq::packed_tile_rows32(w);  // whole blocks
  const int bs = 16 * p->pk_halves;
  tt = tt / bs * bs;
  auto r128 = [](int x) { return (x + 127) / 128 * 128; };
  p->tt_pk = tt;
  p->pk_off_vc = r128(tt * p->krow);
  p->pk_off_ksz = p->pk_off_vc + r128(tt * p->vrow);
  p->pk_off_vsz = p->pk_off_ksz + r128(tt * p->kszrow);
}

// Every staged tile holds at least one 32-row block and fits its stage (the
// kernels walk pieces in steps of whole tiles).
bool tile_geometry_ok(const kvq::Params* p) {
  const int bs = 16 * p->pk_halves;
  if (p->tt_pk < bs || p->tt_pk % bs || p->tt_ko < 32 || p->tt_ko % 32) return false;
  if (p->pk_off_vsz + p->tt_pk * p->vszrow > kvq::kStageBytes) return false;
  if (p->ko_off_vsz + p->tt_ko * p->vszrow > kvq::kStageBytes) return false;
  return p->pk_off_vc + p->tt_pk * p->vrow <= kvq::kStageBytes && p->ko_off_vc + p->tt_ko * p->vrow <= kvq::kStageBytes;
}

// general: the variant for layouts with K-only heads and multi-query calls.
const void* split_kernel_for(int kb, int vb, int G, bool step, int halves, bool general, bool cluster) {
  switch (kb) {
    case 2: return (cluster ? kvq::split_kernel_cl_k2 : kvq::split_kernel_k2)(vb, G, step, halves, general);
    case 4: return (cluster ? kvq::split_kernel_cl_k4 : kvq::split_kernel_k4)(vb, G, step, halves, general);
    case 8: return (cluster ? kvq::split_kernel_cl_k8 : kvq::split_kernel_k8)(vb, G, step, halves, general);
    case 16: return (cluster ? kvq::split_kernel_cl_k16 : kvq::split_kernel_k16)(vb, G, step, halves, general);
  }
  return nullptr;
}

// One-time per kernel: >48 KB dynamic shared memory, clusters of 16 CTAs
// allowed, a check that the 12-warp block fits (per-partition register
// budget), and how many 16-CTA clusters of it the GPU holds at once.
constexpr int kClusterCtas = kvq::kMaxClusterCtas;
struct SplitInfo {
  const void* fn;
  int max_clusters;  // 16-CTA clusters resident at once (0: cluster launches unavailable)
};
kvq_status prepare_split(const void* fn, size_t smem, int* max_clusters) {
  static std::mutex mu;
  static SplitInfo done[512];
  static int n_done = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_done; ++i)
    if (done[i].fn == fn) {
      *max_clusters = done[i].max_clusters;
      return KVQ_OK;
    }
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
  if (e != cudaSuccess) return kvq_cuda_fail(e);
  cudaFuncAttributes fa;
  const cudaError_t e2 = cudaFuncGetAttributes(&fa, fn);
  if (e2 != cudaSuccess) return kvq_cuda_fail(e2);
  if (fa.maxThreadsPerBlock < kvq::kSplitThreads) return kvq_cuda_fail(cudaErrorLaunchOutOfResources);
  int ncl = 0;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kClusterCtas);
    cfg.blockDim = dim3(kvq::kSplitThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = kClusterCtas;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&ncl, fn, &cfg) != cudaSuccess) ncl = 0;
  }
  (void)cudaGetLastError();  // a refused cluster query only disables cluster mode
  if (n_done < 512) done[n_done++] = SplitInfo{fn, ncl};
  *max_clusters = ncl;
  return KVQ_OK;
}

// Cluster mode pays when every unit fits one resident 16-CTA cluster and a
// sixteenth of the largest unit is still a small piece of work (at most
// kClusterMaxCtaCost cost units, about that many bytes): then the cluster's
// merge through distributed shared memory replaces the workspace partials,
// the counters and the combine.  Larger units stream faster over every SM
// (global mode).
constexpr int64_t kClusterMaxCtaCost = 512 * 1024;
bool use_cluster_mode(const kvq::Plan& P, int max_clusters) {
  if (P.U > max_clusters || static_cast<int64_t>(P.U) * kClusterCtas > KVQ_MAX_CTAS) return false;
  int64_t biggest = P.U_p ? P.ub_p : 0;
  if (P.U_k) biggest = std::max(biggest, P.ub_k);
  if (P.U - P.U_p - P.U_k) biggest = std::max(biggest, P.ub_u);
  return biggest / kClusterCtas <= kClusterMaxCtaCost;
}

// Wait limits of the calling host thread (kvq_set_wait_limits); 0 = default.
thread_local uint32_t tl_tile_polls = 0;
thread_local uint32_t tl_peer_polls = 0;
// Early cache-tile copies of the calling host thread (kvq_set_cache_preload).
thread_local int32_t tl_preload = 0;

// Units of a decode call with n_q query tokens per sequence.
int64_t decode_units(const kvq_layout* L, int32_t n_q) {
  return static_cast<int64_t>(L->d.B) * L->d.H_kv * ((static_cast<int64_t>(L->g) * n_q + kvq::kNH - 1) / kvq::kNH);
}

// Shared argument checks and parameter set-up of the decode entry points
// (n_q query tokens per sequence).
kvq_status decode_params(const kvq_layout* L, const void* cache, const void* q_bf16, int32_t T,
                         float softmax_scale, void* out_bf16, float* lse, void* workspace,
                         size_t ws_bytes, kvq::Params* p, int32_t n_q = 1) {
  const kvq_status st = kvq_check_layout(L);
  if (st != KVQ_OK) return st;
  if (!cache || !q_bf16 || !out_bf16 || !workspace) return KVQ_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(cache) % 256 || reinterpret_cast<uintptr_t>(workspace) % 256 ||
      reinterpret_cast<uintptr_t>(q_bf16) % 16 || reinterpret_cast<uintptr_t>(out_bf16) % 16 ||
      reinterpret_cast<uintptr_t>(lse) % 4)
    return KVQ_ERR_INVALID_ARG;
  if (T < 1 || T > L->d.T_cap) return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  const int64_t units = decode_units(L, n_q);
  if (ws_bytes < static_cast<size_t>(kvq::ws_total_bytes(units))) return KVQ_ERR_CAPACITY;
  int n_sm = 0;
  if (kvq_device_sm_count(&n_sm) != 0) return KVQ_ERR_CUDA;
  kvq_fill_params(L, p);
  const uint8_t* base = static_cast<const uint8_t*>(cache);
  for (int s = 0; s < KVQ_NSEG; ++s) p->seg[s] = base + L->off[s];
  p->T = T;
  p->q = static_cast<const uint16_t*>(q_bf16);
  p->out = static_cast<uint16_t*>(out_bf16);
  p->lse = lse;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int64_t cnt_bytes = kvq::ws_counter_bytes(units);
  p->status = reinterpret_cast<uint32_t*>(ws);
  p->cnt = reinterpret_cast<uint32_t*>(ws + kvq::kWsHeadBytes);
  p->ws_o = reinterpret_cast<float*>(ws + kvq::kWsHeadBytes + cnt_bytes);
  p->ws_ml = reinterpret_cast<float*>(ws + kvq::kWsHeadBytes + cnt_bytes + kvq::ws_o_bytes(units));
  p->tile_polls = tl_tile_polls ? tl_tile_polls : kvq::kDefaultTilePolls;
  p->peer_polls = tl_peer_polls ? tl_peer_polls : kvq::kDefaultPeerPolls;
  p->preload = tl_preload;
  p->scale_log2 = softmax_scale * 1.4426950408889634f;
  p->seq_len = nullptr;  // uniform call; the ragged entry points set it
  p->n_q = n_q;
  p->plan = kvq_make_plan(L, T, n_sm, n_q);  // one CTA per SM
  p->NHC = p->plan.NHC;
  kvq_plan_cuts(&p->plan, p->cuts);
  p->pk_halves = packed_halves(p->plan, L, n_q);
  packed_tile_geometry(p);
  konly_tile_geometry(p);
  if (!tile_geometry_ok(p)) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

// One CTA per SM: the stage ring, merge buffers and barriers must fit the
// 227 KiB a CTA may use.
constexpr size_t kSplitSmemCl = sizeof(kvq::SplitSmem<true>);   // cluster mode
constexpr size_t kSplitSmemGl = sizeof(kvq::SplitSmem<false>);  // global mode
static_assert(kSplitSmemCl <= 232448 && kSplitSmemGl <= 232448, "split kernel shared memory exceeds one CTA's limit");
size_t split_smem(const kvq::Params* p) { return p->plan.cs > 1 ? kSplitSmemCl : kSplitSmemGl; }


// Launch the split kernel: one CTA per chunk, programmatic serialisation
// allowed (the kernel waits with griddepcontrol.wait before touching
// memory), in clusters of plan.cs CTAs in cluster mode, cooperative when
// requested (the global-mode fused step, whose combining CTAs may wait for
// other CTAs of their unit).  Programmatic serialisation is dropped if the
// runtime refuses it.
kvq_status launch_split(const void* fn, kvq::Params* p, void* stream, bool cooperative, size_t smem,
                        int threads = kvq::kSplitThreads) {
  static std::atomic<int> pdl_ok{1};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p->plan.C);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[3];
  int na = 0;
  if (p->plan.cs > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = p->plan.cs;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  } else if (cooperative) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  void* args[1] = {p};
  cudaError_t e = cudaErrorUnknown;
  if (pdl_ok.load()) {
    cfg.numAttrs = na + 1;
    e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      pdl_ok.store(0);
    }
  }
  if (!pdl_ok.load()) {
    cfg.numAttrs = na;
    e = cudaLaunchKernelExC(&cfg, fn, args);
  }
  if (e != cudaSuccess) return kvq_cuda_fail(e);
  return KVQ_OK;
}

// Pick the split kernel of a call (p prepared in global mode), switching the
// plan to cluster mode where that pays; *fn gets the kernel.
kvq_status choose_split(const kvq_layout* L, kvq::Params* p, bool step, const void** fn) {
  const bool general = L->n_konly > 0 || p->n_q > 1;
  // the cluster-mode kernel of the same shape: how many of its clusters fit
  const void* fn_cl = split_kernel_for(L->d.k_bits, L->d.v_bits, L->d.group_size, step, p->pk_halves, general, true);
  if (!fn_cl) return KVQ_ERR_UNSUPPORTED;
  int max_clusters = 0;
  kvq_status st = prepare_split(fn_cl, kSplitSmemCl, &max_clusters);
  if (st != KVQ_OK) return st;
  if (!use_cluster_mode(p->plan, max_clusters)) {
    p->preload = 0;  // early copies are a cluster-mode feature (a CTA's whole piece fits its ring)
    *fn = split_kernel_for(L->d.k_bits, L->d.v_bits, L->d.group_size, step, p->pk_halves, general, false);
    if (!*fn) return KVQ_ERR_UNSUPPORTED;
    return prepare_split(*fn, kSplitSmemGl, &max_clusters);
  }
  p->plan.cs = kClusterCtas;
  kvq_plan_cuts(&p->plan, p->cuts);
  p->pk_halves = packed_halves(p->plan, L, p->n_q);
  packed_tile_geometry(p);
  if (!tile_geometry_ok(p)) return KVQ_ERR_UNSUPPORTED;
  *fn = split_kernel_for(L->d.k_bits, L->d.v_bits, L->d.group_size, step, p->pk_halves, general, true);
  if (!*fn) return KVQ_ERR_UNSUPPORTED;
  return prepare_split(*fn, kSplitSmemCl, &max_clusters);
}

// The split kernel and, in global mode, the combine of one decode call (p
// prepared).  In cluster mode the split kernel writes the outputs itself.
kvq_status launch_decode(const kvq_layout* L, kvq::Params* p, void* stream) {
  const void* split = nullptr;
  kvq_status st = choose_split(L, p, false, &split);
  if (st != KVQ_OK) return st;
  st = launch_split(split, p, stream, false, split_smem(p));
  if (st != KVQ_OK || p->plan.cs > 1) return st;
  const bool wide = kvq::plan_max_unit_chunks(p->plan, p->cuts) > 16;
  const void* comb = wide ? reinterpret_cast<const void*>(&kvq::combine_kernel<16>)
                          : reinterpret_cast<const void*>(&kvq::combine_kernel<2>);
  if (kvq_launch_pdl(comb, L->d.B * p->n_q * L->d.H_q, (wide ? 16 : 2) * 32, 0, stream, p) != 0)
    return KVQ_ERR_CUDA;
  return KVQ_OK;
}

// Checks of the fused step's new rows.
kvq_status step_rows_ok(const kvq_layout* L, const void* k_new_bf16, const void* v_new_bf16) {
  if (!L || !k_new_bf16 || !v_new_bf16) return KVQ_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(k_new_bf16) % 16 || reinterpret_cast<uintptr_t>(v_new_bf16) % 16)
    return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

// The fused step's single launch (p prepared).  Global mode is cooperative:
// a combining CTA may wait for other CTAs of its unit, so all CTAs must be
// resident together (one per SM, C <= SM count).  Cluster mode merges inside
// each unit's cluster and never waits on another cluster.
kvq_status launch_step(const kvq_layout* L, kvq::Params* p, void* stream) {
  const void* fn = nullptr;
  const kvq_status st = choose_split(L, p, true, &fn);  // the fused step is single-query
  if (st != KVQ_OK) return st;
  return launch_split(fn, p, stream, true, split_smem(p));
}

// The parameter block of a call is built on the calling host thread and
// copied into the launch; it is large (the cut table), so it lives in
// thread-local storage rather than on the stack.  Calls from different host
// threads therefore neither share nor wait for one another.
kvq::Params* call_params() {
  thread_local kvq::Params p;
  return &p;
}

}  // namespace

extern "C" kvq_status kvq_decode_attention(const kvq_layout* L, const void* cache, const void* q_bf16,
                                           int32_t T, float softmax_scale, void* out_bf16, float* lse,
                                           void* workspace, size_t ws_bytes, void* stream) {
  kvq::Params* p = call_params();
  const kvq_status st = decode_params(L, cache, q_bf16, T, softmax_scale, out_bf16, lse, workspace,
                                      ws_bytes, p);
  if (st != KVQ_OK) return st;
  return launch_decode(L, p, stream);
}

extern "C" kvq_status kvq_decode_attention_ragged(const kvq_layout* L, const void* cache,
                                                  const void* q_bf16, const int32_t* seq_len,
                                                  int32_t T_max, float softmax_scale, void* out_bf16,
                                                  float* lse, void* workspace, size_t ws_bytes,
                                                  void* stream) {
  if (!seq_len || reinterpret_cast<uintptr_t>(seq_len) % 4) return KVQ_ERR_INVALID_ARG;
  kvq::Params* p = call_params();
  const kvq_status st = decode_params(L, cache, q_bf16, T_max, softmax_scale, out_bf16, lse, workspace,
                                      ws_bytes, p);
  if (st != KVQ_OK) return st;
  p->seq_len = seq_len;
  return launch_decode(L, p, stream);
}

// ---- multi-query decode on the tensor-core kernel (kvq_mq_umma.cuh) ----------
// Used when a KV head has more than eight (query head, token) columns: one
// pass over a unit's cache serves up to 128 columns.

const void* mq_umma_for(int kb, int vb, int G) {
  switch (kb) {
    case 2: return kvq::mq_umma_kernel_k2(vb, G);
    case 4: return kvq::mq_umma_kernel_k4(vb, G);
    case 8: return kvq::mq_umma_kernel_k8(vb, G);
    case 16: return kvq::mq_umma_kernel_k16(vb, G);
  }
  return nullptr;
}

constexpr size_t kMqSmemBytes = sizeof(kvq::mq::Smem);
static_assert(kMqSmemBytes <= 232448, "multi-query kernel shared memory exceeds one CTA's limit");

// One-time per kernel: shared memory, non-portable clusters, and how many
// clusters of 16 / 8 / 4 / 2 CTAs the GPU holds at once (index log2(cs)).
struct MqInfo {
  const void* fn;
  int max_clusters[5];
};
kvq_status prepare_mq(const void* fn, int* max_clusters) {
  static std::mutex mu;
  static MqInfo done[64];
  static int n_done = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_done; ++i)
    if (done[i].fn == fn) {
      for (int k = 0; k < 5; ++k) max_clusters[k] = done[i].max_clusters[k];
      return KVQ_OK;
    }
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMqSmemBytes));
  if (e != cudaSuccess) return kvq_cuda_fail(e);
  MqInfo info;
  info.fn = fn;
  info.max_clusters[0] = 0;
  const bool nonportable = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  for (int k = 1; k < 5; ++k) {
    const int cs = 1 << k;
    int ncl = 0;
    if (cs <= 8 || nonportable) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(cs);
      cfg.blockDim = dim3(kvq::mq::kThreads);
      cfg.dynamicSmemBytes = kMqSmemBytes;
      cudaLaunchAttribute at;
      at.id = cudaLaunchAttributeClusterDimension;
      at.val.clusterDim.x = cs;
      at.val.clusterDim.y = 1;
      at.val.clusterDim.z = 1;
      cfg.attrs = &at;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&ncl, fn, &cfg) != cudaSuccess) ncl = 0;
    }
    info.max_clusters[k] = ncl;
  }
  (void)cudaGetLastError();
  if (n_done < 64) done[n_done++] = info;
  for (int k = 0; k < 5; ++k) max_clusters[k] = info.max_clusters[k];
  return KVQ_OK;
}

// Units of up to 128 columns; a cluster of cs CTAs per unit at a time, cs
// chosen for the shortest estimated run: rounds of units over the resident
// clusters times a cs-th of the largest unit's cost, plus a merge per round
// for cs > 1.
kvq_status launch_mq_umma(const kvq_layout* L, kvq::Params* p, void* stream) {
  const void* fn = mq_umma_for(L->d.k_bits, L->d.v_bits, L->d.group_size);
  if (!fn) return KVQ_ERR_UNSUPPORTED;
  int maxcl[5];
  kvq_status st = prepare_mq(fn, maxcl);
  if (st != KVQ_OK) return st;
  int n_sm = 0;
  if (kvq_device_sm_count(&n_sm) != 0) return KVQ_ERR_CUDA;
  const int cols = kvq::mq::kCols;
  p->NHC = (L->g * p->n_q + cols - 1) / cols;
  const kvq::Plan& P = p->plan;
  const int64_t U = static_cast<int64_t>(L->d.B) * L->d.H_kv * p->NHC;
  int64_t biggest = P.U_p ? P.ub_p : 0;
  if (P.U_k) biggest = std::max(biggest, P.ub_k);
  if (P.U - P.U_p - P.U_k) biggest = std::max(biggest, P.ub_u);
  constexpr int64_t kMergeCost = 64 * 1024;  // cost units of one cluster merge (measured order)
  int best_cs = 1;
  int64_t best_grid = std::min<int64_t>(U, n_sm);
  double best = 1e300;
  for (int k = 4; k >= 0; --k) {
    const int cs = 1 << k;
    const int64_t ncl = k == 0 ? n_sm : maxcl[k];
    if (ncl <= 0) continue;
    const int64_t rounds = (U + ncl - 1) / ncl;
    const double est = static_cast<double>(rounds) * (static_cast<double>(biggest) / cs + (cs > 1 ? kMergeCost : 0));
    if (est < best) {
      best = est;
      best_cs = cs;
      best_grid = std::min<int64_t>(ncl, U) * cs;
    }
  }
  p->plan.U = static_cast<int32_t>(U);
  p->plan.cs = best_cs;
  p->plan.C = static_cast<int32_t>(best_grid);
  return launch_split(fn, p, stream, false, kMqSmemBytes, kvq::mq::kThreads);
}

// Which multi-query path is faster, from measured crossovers (GB300, both
// paths timed on the same calls; L2 flushed): the split kernel re-reads a KV
// head's cache once per 8 columns but runs at a high rate per CTA; the
// tcgen05 kernel reads it once per 128 columns at a lower rate per CTA.  The
// tcgen05 kernel wins only when the split passes fill the GPU several times
// over: at least 32 (sequence, KV head) pairs and either >= 128 columns per
// KV head, or >= 32 columns with a short history (T <= 2048).
bool use_mq_umma(const kvq_layout* L, int32_t n_q, int32_t T) {
  const int64_t cols = static_cast<int64_t>(L->g) * n_q;
  if (cols <= kvq::kNH || static_cast<int64_t>(L->d.B) * L->d.H_kv < 32) return false;
  return cols >= 128 || (cols >= 32 && T <= 2048);
}

extern "C" size_t kvq_decode_mq_workspace_bytes(const kvq_layout* L, int32_t n_q) {
  if (kvq_check_layout(L) != KVQ_OK || n_q < 1 || n_q > KVQ_MAX_QUERY_TOKENS) return 0;
  return static_cast<size_t>(kvq::ws_total_bytes(decode_units(L, n_q)));
}

extern "C" kvq_status kvq_decode_attention_mq(const kvq_layout* L, const void* cache, const void* q_bf16,
                                              int32_t n_q, int32_t T, float softmax_scale, void* out_bf16,
                                              float* lse, void* workspace, size_t ws_bytes, void* stream) {
  if (!L) return KVQ_ERR_INVALID_ARG;
  if (n_q < 1 || n_q > KVQ_MAX_QUERY_TOKENS || T < n_q) return KVQ_ERR_INVALID_ARG;
  // the positions some tokens do not attend, [T - n_q + 1, T), must be text
  if (n_q > 1 && L->d.vis_start < L->d.vis_end && T - n_q + 1 < L->d.vis_end && T > L->d.vis_start)
    return KVQ_ERR_INVALID_ARG;
  kvq::Params* p = call_params();
  const kvq_status st = decode_params(L, cache, q_bf16, T, softmax_scale, out_bf16, lse, workspace,
                                      ws_bytes, p, n_q);
  if (st != KVQ_OK) return st;
  if (use_mq_umma(L, n_q, T)) return launch_mq_umma(L, p, stream);  // one pass for up to 128 columns
  return launch_decode(L, p, stream);  // one split pass per 8 columns
}

extern "C" kvq_status kvq_decode_step(const kvq_layout* L, void* cache, const void* q_bf16,
                                      const void* k_new_bf16, const void* v_new_bf16, int32_t t_new,
                                      float softmax_scale, void* out_bf16, float* lse, void* workspace,
                                      size_t ws_bytes, void* stream) {
  kvq_status st = step_rows_ok(L, k_new_bf16, v_new_bf16);
  if (st != KVQ_OK) return st;
  if (t_new < 0 || t_new >= L->d.T_cap) return KVQ_ERR_INVALID_ARG;
  if (t_new >= L->d.vis_start && t_new < L->d.vis_end) return KVQ_ERR_INVALID_ARG;
  kvq::Params* p = call_params();
  st = decode_params(L, cache, q_bf16, t_new + 1, softmax_scale, out_bf16, lse, workspace, ws_bytes, p);
  if (st != KVQ_OK) return st;
  p->k_new = static_cast<const uint16_t*>(k_new_bf16);
  p->v_new = static_cast<const uint16_t*>(v_new_bf16);
  p->t_new = t_new;
  return launch_step(L, p, stream);
}

extern "C" kvq_status kvq_decode_step_ragged(const kvq_layout* L, void* cache, const void* q_bf16,
                                             const void* k_new_bf16, const void* v_new_bf16,
                                             const int32_t* t_new, int32_t T_max, float softmax_scale,
                                             void* out_bf16, float* lse, void* workspace, size_t ws_bytes,
                                             void* stream) {
  kvq_status st = step_rows_ok(L, k_new_bf16, v_new_bf16);
  if (st != KVQ_OK) return st;
  if (!t_new || reinterpret_cast<uintptr_t>(t_new) % 4) return KVQ_ERR_INVALID_ARG;
  kvq::Params* p = call_params();
  st = decode_params(L, cache, q_bf16, T_max, softmax_scale, out_bf16, lse, workspace, ws_bytes, p);
  if (st != KVQ_OK) return st;
  p->k_new = static_cast<const uint16_t*>(k_new_bf16);
  p->v_new = static_cast<const uint16_t*>(v_new_bf16);
  p->t_new = T_max - 1;  // the largest step position a sequence may have
  p->seq_len = t_new;
  return launch_step(L, p, stream);
}

extern "C" void kvq_set_wait_limits(uint32_t tile_polls, uint32_t peer_polls) {
  tl_tile_polls = tile_polls;
  tl_peer_polls = peer_polls;
}

extern "C" void kvq_set_cache_preload(int32_t enable) { tl_preload = enable != 0; }

extern "C" kvq_status kvq_workspace_status(const void* workspace, uint32_t* status, void* stream) {
  if (!workspace || !status || reinterpret_cast<uintptr_t>(workspace) % 4) return KVQ_ERR_INVALID_ARG;
  const cudaError_t e = cudaMemcpyAsync(status, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return kvq_cuda_fail(e);
  return KVQ_OK;
}
