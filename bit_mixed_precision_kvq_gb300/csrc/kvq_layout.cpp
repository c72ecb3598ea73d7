// kvq_layout.cpp -- host side of the cache layout, validation and the
// split-KV work plan.
//
// The layout follows the pages' problem statement: a per-layer cache
// [B, H_kv, T, D] ("VLM_KV_Quantization", section 2) whose visual block is
// quantised group-wise with separate K and V bit-widths (sections 1 and 4),
// while text positions and a per-layer set of protected KV heads (HeadGuard
// brief, key ideas) stay bf16.
#include <cuda_runtime.h>

#include <cmath>
#include <algorithm>
#include <cstring>
#include <mutex>

#include "kvq_internal.h"

namespace {

constexpr int64_t kAlign = 256;   // segment alignment in the cache buffer
constexpr int64_t kPad = 256;     // slack after each segment (rounded tile copies)

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bool valid_bits(int b) { return b == 2 || b == 4 || b == 8 || b == 16; }

kvq_status build_layout(const kvq_layout_desc* desc, kvq_layout* out) {
  if (!desc || !out) return KVQ_ERR_INVALID_ARG;
  const kvq_layout_desc& d = *desc;
  if (d.B < 1 || d.H_kv < 1 || d.H_kv > KVQ_MAX_HEADS || d.H_q < 1 || d.H_q % d.H_kv != 0)
    return KVQ_ERR_INVALID_ARG;
  if (d.D < 1 || d.D % 32 != 0) return KVQ_ERR_INVALID_ARG;
  if (d.T_cap < 1) return KVQ_ERR_INVALID_ARG;
  if (d.vis_start < 0 || d.vis_end < d.vis_start || d.vis_end > d.T_cap) return KVQ_ERR_INVALID_ARG;
  if (!valid_bits(d.k_bits) || !valid_bits(d.v_bits)) return KVQ_ERR_INVALID_ARG;
  if (!(d.group_size == 32 || d.group_size == 64 || d.group_size == 128)) return KVQ_ERR_INVALID_ARG;
  if (d.D % d.group_size != 0) return KVQ_ERR_INVALID_ARG;
  for (int h = 0; h < KVQ_MAX_HEADS; ++h)
    if (d.protected_heads[h] > 2 || (h >= d.H_kv && d.protected_heads[h] != 0))
      return KVQ_ERR_INVALID_ARG;
  if (d.D != kvq::kD) return KVQ_ERR_UNSUPPORTED;

  kvq_layout L;
  std::memset(&L, 0, sizeof(L));
  L.d = d;
  L.g = d.H_q / d.H_kv;
  L.Tv = d.vis_end - d.vis_start;
  // Packed segments keep every (b, head) block of visual rows on a 16-row
  // boundary so that a tile of scale/zero rows (4-16 bytes each) starting at
  // a 16-aligned visual row is 16-byte aligned for bulk copies.
  L.Tv_pad = (L.Tv + 15) / 16 * 16;
  L.T_text = d.T_cap - L.Tv;
  for (int h = 0; h < d.H_kv; ++h) {
    if (d.protected_heads[h] == 1) {
      L.slot[h] = L.n_prot;
      L.prot_head[L.n_prot++] = static_cast<uint8_t>(h);
    } else if (d.protected_heads[h] == 2) {
      L.slot[h] = L.n_konly;
      L.konly_head[L.n_konly++] = static_cast<uint8_t>(h);
    } else {
      L.slot[h] = L.n_packed;
      L.packed_head[L.n_packed++] = static_cast<uint8_t>(h);
    }
  }
  const int nhc = (L.g + kvq::kNH - 1) / kvq::kNH;
  L.units = d.B * d.H_kv * nhc;

  const int64_t D = d.D, G = d.group_size;
  L.row_bytes[KVQ_SEG_K_CODES] = D * d.k_bits / 8;
  L.row_bytes[KVQ_SEG_K_SZ] = d.k_bits < 16 ? 4 * D / G : 0;
  L.row_bytes[KVQ_SEG_V_CODES] = D * d.v_bits / 8;
  L.row_bytes[KVQ_SEG_V_SZ] = d.v_bits < 16 ? 4 * D / G : 0;
  L.row_bytes[KVQ_SEG_PROT_K] = 2 * D;
  L.row_bytes[KVQ_SEG_PROT_V] = 2 * D;
  L.row_bytes[KVQ_SEG_TEXT_K] = 2 * D;
  L.row_bytes[KVQ_SEG_TEXT_V] = 2 * D;
  // K-only heads (mode 2) keep their K with the protected heads' K and their
  // V with the packed heads' V (after them).
  const int64_t packed_k_rows = static_cast<int64_t>(d.B) * L.n_packed * L.Tv_pad;
  const int64_t packed_v_rows = static_cast<int64_t>(d.B) * (L.n_packed + L.n_konly) * L.Tv_pad;
  const int64_t prot_k_rows = static_cast<int64_t>(d.B) * (L.n_prot + L.n_konly) * L.Tv;
  const int64_t prot_v_rows = static_cast<int64_t>(d.B) * L.n_prot * L.Tv;
  const int64_t text_rows = static_cast<int64_t>(d.B) * d.H_kv * L.T_text;
  const int64_t rows[KVQ_NSEG] = {packed_k_rows, packed_k_rows, packed_v_rows, packed_v_rows,
                                  prot_k_rows,   prot_v_rows,   text_rows,     text_rows};
  int64_t off = 0;
  for (int s = 0; s < KVQ_NSEG; ++s) {
    L.off[s] = off;
    L.bytes[s] = rows[s] * L.row_bytes[s];
    off = align_up(off + L.bytes[s] + kPad, kAlign);
  }
  L.total_bytes = off;
  L.workspace_bytes = kvq::ws_total_bytes(L.units);
  L.eff_bits_k = d.k_bits < 16 ? d.k_bits + 32.0 / d.group_size : 16.0;
  L.eff_bits_v = d.v_bits < 16 ? d.v_bits + 32.0 / d.group_size : 16.0;
  *out = L;
  return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_cache_layout(const kvq_layout_desc* desc, kvq_layout* out) {
  return build_layout(desc, out);
}

extern "C" const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_INVALID_ARG: return "KVQ_ERR_INVALID_ARG";
    case KVQ_ERR_UNSUPPORTED: return "KVQ_ERR_UNSUPPORTED";
    case KVQ_ERR_CAPACITY: return "KVQ_ERR_CAPACITY";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA";
  }
  return "kvq_status(unknown)";
}

// A layout handed back by the caller must be exactly what kvq_cache_layout
// derives from its own description (guards against corrupted structs).
kvq_status kvq_check_layout(const kvq_layout* L) {
  if (!L) return KVQ_ERR_INVALID_ARG;
  kvq_layout ref;
  const kvq_status st = build_layout(&L->d, &ref);
  if (st != KVQ_OK) return st;
  if (std::memcmp(&ref, L, sizeof(kvq_layout)) != 0) return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

void kvq_fill_params(const kvq_layout* L, kvq::Params* p) {
  std::memset(p, 0, sizeof(*p));
  const kvq_layout_desc& d = L->d;
  p->B = d.B;
  p->Hq = d.H_q;
  p->Hkv = d.H_kv;
  p->g = L->g;
  p->NHC = (L->g + kvq::kNH - 1) / kvq::kNH;
  p->T = d.T_cap;
  p->vs = d.vis_start;
  p->ve = d.vis_end;
  p->Tv = L->Tv;
  p->Tv_pad = L->Tv_pad;
  p->T_text = L->T_text;
  p->kb = d.k_bits;
  p->vb = d.v_bits;
  p->G = d.group_size;
  p->n_prot = L->n_prot;
  p->n_packed = L->n_packed;
  p->n_konly = L->n_konly;
  p->krow = static_cast<int32_t>(L->row_bytes[KVQ_SEG_K_CODES]);
  p->kszrow = static_cast<int32_t>(L->row_bytes[KVQ_SEG_K_SZ]);
  p->vrow = static_cast<int32_t>(L->row_bytes[KVQ_SEG_V_CODES]);
  p->vszrow = static_cast<int32_t>(L->row_bytes[KVQ_SEG_V_SZ]);
  for (int h = 0; h < KVQ_MAX_HEADS; ++h) {
    p->prot[h] = d.protected_heads[h];
    p->slot[h] = L->slot[h];
    p->prot_head[h] = L->prot_head[h];
    p->packed_head[h] = L->packed_head[h];
    p->konly_head[h] = L->konly_head[h];
  }
}

kvq::Plan kvq_make_plan(const kvq_layout* L, int32_t T, int32_t n_chunks_target, int32_t n_q) {
  kvq::Plan P;
  std::memset(&P, 0, sizeof(P));
  const kvq_layout_desc& d = L->d;
  P.T = T;
  P.NHC = (L->g * n_q + kvq::kNH - 1) / kvq::kNH;
  P.vsa = d.vis_start < T ? d.vis_start : T;
  P.vea = d.vis_end < T ? d.vis_end : T;
  const int64_t vrow = L->row_bytes[KVQ_SEG_V_CODES] + L->row_bytes[KVQ_SEG_V_SZ];
  P.w_vis = static_cast<int32_t>(L->row_bytes[KVQ_SEG_K_CODES] + L->row_bytes[KVQ_SEG_K_SZ] + vrow) +
            kvq::kPosCost;
  P.w_kvis = static_cast<int32_t>(2 * kvq::kD + vrow) + kvq::kPosCost;
  P.U_p = d.B * L->n_prot * P.NHC;
  P.U_k = d.B * L->n_konly * P.NHC;
  P.U = d.B * d.H_kv * P.NHC;
  P.ub_p = static_cast<int64_t>(T) * kvq::kBf16PosCost;
  const int64_t n_vis = P.vea - P.vsa;
  P.ub_k = (static_cast<int64_t>(T) - n_vis) * kvq::kBf16PosCost + n_vis * P.w_kvis;
  P.ub_u = (static_cast<int64_t>(T) - n_vis) * kvq::kBf16PosCost + n_vis * P.w_vis;
  P.P_bytes = static_cast<int64_t>(P.U_p) * P.ub_p;
  P.K_bytes = static_cast<int64_t>(P.U_k) * P.ub_k;
  P.total = P.P_bytes + P.K_bytes + static_cast<int64_t>(P.U - P.U_p - P.U_k) * P.ub_u;
  // Chunks: the target (a whole number of CTAs per SM), but no chunk below
  // 8 Ki cost units and never more than KVQ_MAX_CTAS.
  int64_t C = n_chunks_target;
  const int64_t by_size = (P.total + 8191) / 8192;
  if (C > by_size) C = by_size;
  if (C > KVQ_MAX_CTAS) C = KVQ_MAX_CTAS;
  if (C < 1) C = 1;
  P.C = static_cast<int32_t>(C);
  P.cs = 1;
  return P;
}

void kvq_plan_cuts(kvq::Plan* Pp, kvq::Cut* cuts) {
  using kvq::Cut;
  kvq::Plan& P = *Pp;
  if (P.cs > 1) {
    // Cluster mode: unit u is cut into exactly cs chunks of equal cost,
    // chunks u * cs .. u * cs + cs - 1 (the CTAs of cluster u).
    P.C = P.U * P.cs;
    P.aligned = 1;
    P.n_p = P.n_k = P.n_q = P.cs;
    P.R = 0;
    int32_t c = 0;
    for (int32_t u = 0; u < P.U; ++u) {
      const int cls = kvq::unit_class(P, u);
      const int64_t ucost = cls == kvq::kClsProt ? P.ub_p : (cls == kvq::kClsKonly ? P.ub_k : P.ub_u);
      for (int32_t k = 0; k < P.cs; ++k) cuts[c++] = Cut{u, kvq::unit_cut_pos(P, cls, ucost * k / P.cs)};
    }
    cuts[P.C] = Cut{P.U, 0};
    return;
  }
  cuts[P.C] = Cut{P.U, 0};
  P.aligned = P.C >= P.U ? 1 : 0;
  P.n_p = P.n_k = P.n_q = P.R = 0;
  const int64_t U_q = P.U - P.U_p - P.U_k;
  if (!P.aligned) {
    // Equal-cost cuts of the concatenated stream of units.
    for (int32_t c = 0; c < P.C; ++c) {
      const int64_t X = (P.total * static_cast<int64_t>(c)) / P.C;
      if (X < P.P_bytes) {
        const int64_t u = X / P.ub_p;
        cuts[c] = Cut{static_cast<int32_t>(u), kvq::unit_cut_pos(P, kvq::kClsProt, X - u * P.ub_p)};
      } else if (X < P.P_bytes + P.K_bytes) {
        const int64_t u = (X - P.P_bytes) / P.ub_k;
        cuts[c] = Cut{P.U_p + static_cast<int32_t>(u),
                      kvq::unit_cut_pos(P, kvq::kClsKonly, X - P.P_bytes - u * P.ub_k)};
      } else {
        const int64_t Xu = X - P.P_bytes - P.K_bytes;
        const int64_t u = Xu / P.ub_u;
        cuts[c] = Cut{P.U_p + P.U_k + static_cast<int32_t>(u),
                      kvq::unit_cut_pos(P, kvq::kClsPacked, Xu - u * P.ub_u)};
      }
    }
    return;
  }
  // Per-unit chunks: n per unit of each class in proportion to its cost (at
  // least one each); the R chunks left over go one each to the first R
  // units.
  const int64_t Uc[3] = {P.U_p, P.U_k, U_q};
  const int64_t uc[3] = {P.ub_p, P.ub_k, P.ub_u};
  int64_t n[3];
  for (int k = 0; k < 3; ++k) n[k] = Uc[k] ? std::max<int64_t>(1, P.C * uc[k] / P.total) : 0;
  while (n[0] * Uc[0] + n[1] * Uc[1] + n[2] * Uc[2] > P.C) {  // only when a share was raised to 1
    int pick = -1;  // the class with the most chunks per unit of cost
    for (int k = 0; k < 3; ++k)
      if (Uc[k] && n[k] > 1 && (pick < 0 || n[k] * uc[pick] > n[pick] * uc[k])) pick = k;
    --n[pick];  // exists: with every n at 1 the sum is U <= C
  }
  const int64_t R = P.C - n[0] * Uc[0] - n[1] * Uc[1] - n[2] * Uc[2];
  P.n_p = static_cast<int32_t>(n[0]);
  P.n_k = static_cast<int32_t>(n[1]);
  P.n_q = static_cast<int32_t>(n[2]);
  P.R = static_cast<int32_t>(R);
  int32_t c = 0;
  for (int32_t u = 0; u < P.U; ++u) {
    const int cls = kvq::unit_class(P, u);
    const int64_t nu = n[cls] + (u < R ? 1 : 0);
    for (int64_t k = 0; k < nu; ++k) cuts[c++] = Cut{u, kvq::unit_cut_pos(P, cls, uc[cls] * k / nu)};
  }
}

namespace {
thread_local int last_cuda_error = 0;
}

kvq_status kvq_cuda_fail(int err) {
  last_cuda_error = err;
  return KVQ_ERR_CUDA;
}

extern "C" int kvq_last_cuda_error(void) { return last_cuda_error; }

int kvq_device_sm_count(int* n_sm) {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return kvq_cuda_fail(e), -1;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && cache[dev] > 0) {
    *n_sm = cache[dev];
    return 0;
  }
  int v = 0;
  e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return kvq_cuda_fail(e), -1;
  if (dev >= 0 && dev < 64) cache[dev] = v;
  *n_sm = v;
  return 0;
}

int kvq_launch_pdl(const void* fn, unsigned grid, unsigned block, size_t smem, void* stream,
                   kvq::Params* p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[1] = {p};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) {
    kvq_cuda_fail(e);
    return -1;
  }
  return 0;
}
