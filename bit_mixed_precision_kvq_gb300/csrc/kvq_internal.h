// kvq_internal.h -- shared by the library's host code and CUDA kernels.
//
// Work decomposition for split-KV decoding (flash-decoding pipeline of the
// WSVD summary, section 2.라, restated for a mixed-precision cache):
//   * a "unit" is one (sequence b, KV head h, chunk hc of up to 8 of the
//     query columns that read h: its g query heads, or for a multi-query
//     call its g * n_q (head, token) pairs).  Protected-head units come
//     first, then the K-only ones, then the packed-head units; inside each
//     class the order is (b, slot, hc).
//   * every unit is a stream of positions 0..T-1; a position costs its cache
//     bytes -- 512 (bf16 K + V rows), or for a visual position of a packed
//     head the packed K and V rows plus their fp16 scale/zero -- plus a
//     fixed compute cost (kPosCost).
//   * chunks: when there are at least as many chunks C as units, every unit
//     gets its own chunks, in number proportional to its cost (at least
//     one), cut at equal cost inside the unit -- no chunk spans two units.
//     Otherwise the concatenated cost stream of all units is cut into C
//     chunks of equal cost.  CTA c processes [cut(c), cut(c+1)).  Cuts
//     inside a packed visual range are rounded down to a multiple of 16
//     rows so every staged tile starts on a 16-byte boundary in every
//     segment.
//   * CTA c writes one partial result (o, m, l) per unit it touches into
//     workspace slot u + c.  The (u, c) pairs form a monotone staircase, so
//     u + c is unique; there are at most units + C - 1 slots.
//   * the fused decode step combines a unit's partials in the CTAs that
//     finish the unit's last chunks (per-unit arrival counters in the
//     workspace).
//   * cluster mode (plan.cs > 1, when every unit fits one thread-block
//     cluster of the GPU at once): unit u is cut into exactly cs chunks,
//     processed by the cs CTAs of cluster u, which merge their partials
//     through distributed shared memory -- no workspace partials, no
//     counters, no inter-CTA waiting -- and write the outputs directly.
#pragma once

#include <stdint.h>

#include "../../include/kvq.h"

#if defined(__CUDACC__)
#define KVQ_HD __host__ __device__ __forceinline__
#else
#define KVQ_HD inline
#endif

namespace kvq {

constexpr int kD = 128;          // head dimension supported by the kernels
constexpr int kNH = KVQ_HEADS_PER_UNIT;  // query heads per unit (MMA N = 8)
constexpr int kBf16PosBytes = 4 * kD;    // K + V bf16 rows of one position
constexpr int kVisAlign = 16;            // visual-row alignment of chunk cuts
// Stage size of the split kernel's shared-memory ring, and the staging of
// packed tiles: positions per tile (a multiple of the block size, <= 512)
// and the largest block size of the kernel for (k_bits, v_bits, G) -- 64
// positions (4 MMA row-tiles per softmax update) when a tile holds >= 256
// positions, else 32; a call uses 64 only when its chunks are long enough to
// keep the consumer warps busy with it.
constexpr int kStageBytes = 40 * 1024;
KVQ_HD constexpr int packed_row_bytes(int kb, int vb, int G) {
  return 16 * kb + 16 * vb + (kb < 16 ? 4 * (kD / G) : 0) + (vb < 16 ? 4 * (kD / G) : 0);
}
// Tiles are whole multiples of 32 rows and every row size is a multiple of
// 4 bytes, so each of a stage's sub-buffers (K codes, V codes, K and V
// scale/zero rows) ends on a 128-byte boundary by itself: w bytes per row
// fill a stage with (kStageBytes / w) rows, rounded down to 32.  A row is at
// most 512 bytes (bf16 K and V), so every tile holds at least 32 rows.
KVQ_HD constexpr int packed_tile_rows32(int w) {
  return (kStageBytes / w) / 32 * 32 > 512 ? 512 : (kStageBytes / w) / 32 * 32;
}
static_assert(packed_tile_rows32(4 * kD) >= 32, "a stage must hold 32 bf16 K + V rows");
KVQ_HD constexpr int packed_block_halves(int kb, int vb, int G) {
  return packed_tile_rows32(packed_row_bytes(kb, vb, G)) >= 256 ? 4 : 2;
}

// Work balance: a position costs its cache bytes plus this many byte
// equivalents of unpack / tensor-core / softmax work, so that chunks of
// cheap packed rows do not get several times more positions to compute.
constexpr int kPosCost = 256;
constexpr int kBf16PosCost = kBf16PosBytes + kPosCost;

// Unit classes, in unit order: protected heads (K and V bf16), K-only
// protected heads (K bf16, V packed), packed heads.
enum UnitClass { kClsProt = 0, kClsKonly = 1, kClsPacked = 2 };

struct Plan {
  int32_t U_p;        // protected units
  int32_t U;          // all units
  int32_t C;          // chunks (= CTAs of the split kernel)
  int32_t NHC;        // query-head chunks per KV head
  int32_t vsa, vea;   // attended visual positions [vsa, vea)
  int32_t T;          // attended positions
  int32_t w_vis;      // cost of one packed visual position (bytes + kPosCost)
  int64_t ub_p, ub_u; // cost of a protected / packed unit
  int64_t P_bytes;    // U_p * ub_p
  int64_t total;      // cost of all units
  // per-unit chunks (aligned != 0, when C >= U): n_p per protected, n_k per
  // K-only and n_q per packed unit, plus one for each of the first R units
  int32_t aligned, n_p, n_q, R;
  // K-only protected units (after the protected ones)
  int32_t U_k, n_k;
  int32_t w_kvis;     // cost of one K-only visual position
  int64_t ub_k;       // cost of a K-only unit
  int64_t K_bytes;    // U_k * ub_k
  int32_t cs;         // cluster mode: CTAs per cluster (= chunks per unit); 1 otherwise
};

struct Cut {
  int32_t u;  // unit
  int32_t p;  // position inside the unit
};

// Position inside a unit of class cls at cost offset `rem` (0 <= rem < unit
// cost).  Visual cuts of units with packed rows are 16-row aligned.
KVQ_HD int32_t unit_cut_pos(const Plan& P, int cls, int64_t rem) {
  if (cls == kClsProt) return static_cast<int32_t>(rem / kBf16PosCost);
  const int64_t w = cls == kClsKonly ? P.w_kvis : P.w_vis;
  const int64_t pre = static_cast<int64_t>(P.vsa) * kBf16PosCost;
  const int64_t vis = static_cast<int64_t>(P.vea - P.vsa) * w;
  if (rem < pre) return static_cast<int32_t>(rem / kBf16PosCost);
  if (rem < pre + vis) {
    int64_t row = (rem - pre) / w;
    row -= row % kVisAlign;
    return P.vsa + static_cast<int32_t>(row);
  }
  return P.vea + static_cast<int32_t>((rem - pre - vis) / kBf16PosCost);
}

// Class of unit u.
KVQ_HD int unit_class(const Plan& P, int32_t u) {
  return u < P.U_p ? kClsProt : (u < P.U_p + P.U_k ? kClsKonly : kClsPacked);
}

// Last unit of chunk c: a chunk that ends exactly at the start of a unit
// (cut (u, 0)) does not touch that unit.
KVQ_HD int32_t chunk_last_unit(const Cut* cuts, int32_t c, int32_t U) {
  const Cut a = cuts[c], e = cuts[c + 1];
  if (e.p == 0 && e.u > a.u) return e.u - 1;
  return e.u < U ? e.u : U - 1;
}

// Chunks that hold a piece of unit u: [c_first, c_last]; closed form for
// per-unit chunks, else a binary search over the cut table (cuts[0..C]).
//   c_last  = max c with cuts[c].u <= u
//   c_first = min c with chunk_last_unit(c) >= u
KVQ_HD void plan_unit_chunks(const Plan& P, const Cut* cuts, int32_t u, int32_t* c_first,
                             int32_t* c_last) {
  if (P.aligned) {  // closed form of the per-unit allocation
    const int32_t Uk_end = P.U_p + P.U_k;
    const int32_t base = u <= P.U_p ? u * P.n_p
                         : u <= Uk_end ? P.U_p * P.n_p + (u - P.U_p) * P.n_k
                                       : P.U_p * P.n_p + P.U_k * P.n_k + (u - Uk_end) * P.n_q;
    const int32_t c0 = base + (u < P.R ? u : P.R);
    const int32_t n = (u < P.U_p ? P.n_p : (u < Uk_end ? P.n_k : P.n_q)) + (u < P.R ? 1 : 0);
    *c_first = c0;
    *c_last = c0 + n - 1;
    return;
  }
  int32_t lo = 0, hi = P.C - 1;  // invariant: cuts[lo].u <= u
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) / 2;
    if (cuts[mid].u <= u) lo = mid; else hi = mid - 1;
  }
  *c_last = lo;
  lo = 0;
  hi = P.C - 1;  // the last chunk ends with unit U-1 >= u
  while (lo < hi) {
    const int32_t mid = (lo + hi) / 2;
    if (chunk_last_unit(cuts, mid, P.U) >= u) hi = mid; else lo = mid + 1;
  }
  *c_first = lo;
}

// Most chunks any unit of the plan is split over (host; sizes the combine).
inline int32_t plan_max_unit_chunks(const Plan& P, const Cut* cuts) {
  if (P.aligned) {
    const int32_t n = P.n_p > P.n_k ? P.n_p : P.n_k;
    return (n > P.n_q ? n : P.n_q) + (P.R > 0 ? 1 : 0);
  }
  int32_t best = 1, run_u = -1, run = 0;  // chunks touching unit run_u so far (cuts are monotone)
  for (int32_t c = 0; c < P.C; ++c) {
    const int32_t u0 = cuts[c].u, u1 = chunk_last_unit(cuts, c, P.U);
    run = u0 == run_u ? run + 1 : 1;
    if (run > best) best = run;
    run_u = u1;
    if (u1 != u0) run = 1;  // the chunk ends in a later unit, which it starts
  }
  return best;
}

// Decode workspace: a 256-byte head whose first word is the status word
// (KVQ_STATUS_* bits, OR-ed by the kernels, never cleared by them), the
// per-unit arrival counters of the fused step, then one partial
// (o[kNH][kD] fp32, then (m, l)[kNH] fp32 in a second array) per slot,
// slots <= units + C - 1 <= units + KVQ_MAX_CTAS - 1; each part 256-byte
// aligned.
constexpr int64_t kWsHeadBytes = 256;
KVQ_HD int64_t ws_counter_bytes(int64_t units) { return (4 * units + 255) / 256 * 256; }
KVQ_HD int64_t ws_o_bytes(int64_t units) {
  return ((units + KVQ_MAX_CTAS - 1) * kNH * kD * 4 + 255) / 256 * 256;
}
KVQ_HD int64_t ws_ml_bytes(int64_t units) { return ((units + KVQ_MAX_CTAS - 1) * kNH * 8 + 255) / 256 * 256; }
KVQ_HD int64_t ws_total_bytes(int64_t units) {
  return kWsHeadBytes + ws_counter_bytes(units) + ws_o_bytes(units) + ws_ml_bytes(units);
}

// Bounded waits: polls of an mbarrier try_wait (each suspends the thread for
// a hardware-chosen interval) and of the fused step's inter-CTA counter
// (each followed by a short sleep) before a wait gives up.
constexpr uint32_t kDefaultTilePolls = 1u << 24;
constexpr uint32_t kDefaultPeerPolls = 1u << 21;

// Everything a kernel needs about one layer and one call (passed by value).
struct Params {
  // geometry
  int32_t B, Hq, Hkv, g, NHC;
  int32_t T;           // attended positions (decode) / T_cap (append)
  int32_t vs, ve;      // visual range of the layout
  int32_t Tv, Tv_pad, T_text;
  int32_t kb, vb, G;
  int32_t n_prot, n_packed;
  int32_t krow, kszrow, vrow, vszrow;  // bytes per row of the packed segments
  int32_t tt_pk;                       // positions per packed tile (multiple of the block)
  int32_t pk_halves;                   // 16-row MMA halves per packed block: 2 or 4
  int32_t pk_off_vc, pk_off_ksz, pk_off_vsz;  // packed-tile offsets in a stage
  // cache segments
  const uint8_t* seg[KVQ_NSEG];
  // decode call
  const uint16_t* q;   // bf16 [B][Hq][D]
  uint16_t* out;       // bf16 [B][Hq][D]
  float* lse;          // [B][Hq] or null
  float* ws_o;         // [slots][kNH][kD]
  float* ws_ml;        // [slots][kNH][2]
  // fused decode step only
  const uint16_t* k_new;  // bf16 [B][Hkv][D]
  const uint16_t* v_new;
  int32_t t_new;          // uniform fused step: its position (= T - 1); the kernels use each unit's end
  uint32_t* cnt;          // per-unit arrival counters (zero between calls)
  uint32_t* status;       // workspace status word (KVQ_STATUS_* bits)
  uint32_t tile_polls;    // bounded mbarrier waits on staged tiles
  uint32_t peer_polls;    // bounded wait of the fused step's combining CTAs
  int32_t preload;        // uniform calls: copy the leading cache tiles before the dependency wait
  float scale_log2;    // softmax_scale * log2(e)
  Plan plan;
  Cut cuts[KVQ_MAX_CTAS + 1];         // cut(c) for c = 0..C, computed on the host
  uint8_t prot[KVQ_MAX_HEADS];        // head -> protection mode (0, 1 both, 2 K only)
  int32_t slot[KVQ_MAX_HEADS];        // head -> slot
  uint8_t prot_head[KVQ_MAX_HEADS];   // protected slot -> head
  uint8_t packed_head[KVQ_MAX_HEADS]; // packed slot -> head
  // K-only protected heads (layouts that have them)
  uint8_t konly_head[KVQ_MAX_HEADS];  // K-only slot -> head
  int32_t n_konly;
  int32_t tt_ko;                       // positions per K-only tile (bf16 K + packed V rows)
  int32_t ko_off_vc, ko_off_vsz;       // K-only-tile offsets in a stage
  // ragged calls: device int32 [B] of attended positions (decode) or step
  // positions (fused step) per sequence; null for uniform calls
  const int32_t* seq_len;
  // multi-query decode: query tokens per sequence (1 otherwise).  A unit's
  // columns are (head j, token i) pairs, column c = j * n_q + i; token i
  // attends the unit's positions except the last n_q - 1 - i.
  int32_t n_q;
};

// unit -> (b, head, hc, slot, class).  kGen: the general kernels (layouts
// with K-only protected heads -- three unit classes -- and multi-query
// calls); else only protected and packed units.
struct UnitInfo {
  int32_t b, h, hc, slot;
  int32_t cls;
  bool prot;  // cls == kClsProt
};

template <bool kGen>
KVQ_HD UnitInfo unit_info(const Params& p, int32_t u) {
  UnitInfo r;
  int cls;
  int32_t v, nslots;
  if constexpr (kGen) {
    cls = unit_class(p.plan, u);
    v = cls == kClsProt ? u : (cls == kClsKonly ? u - p.plan.U_p : u - p.plan.U_p - p.plan.U_k);
    nslots = cls == kClsProt ? p.n_prot : (cls == kClsKonly ? p.n_konly : p.n_packed);
  } else {
    cls = u < p.plan.U_p ? kClsProt : kClsPacked;
    v = cls == kClsProt ? u : u - p.plan.U_p;
    nslots = cls == kClsProt ? p.n_prot : p.n_packed;
  }
  r.b = v / (nslots * p.NHC);
  const int32_t rem = v - r.b * nslots * p.NHC;
  r.slot = rem / p.NHC;
  r.hc = rem - r.slot * p.NHC;
  if constexpr (kGen) {
    r.h = cls == kClsProt ? p.prot_head[r.slot] : (cls == kClsKonly ? p.konly_head[r.slot] : p.packed_head[r.slot]);
  } else {
    r.h = cls == kClsProt ? p.prot_head[r.slot] : p.packed_head[r.slot];
  }
  r.cls = cls;
  r.prot = cls == kClsProt;
  return r;
}

// Row of q / out / lse (in units of D elements, or of one lse value) of
// column c of KV head h of sequence b: [B][n_q][H_q] row-major.
KVQ_HD int64_t col_row(const Params& p, int32_t b, int32_t h, int32_t c) {
  if (p.n_q == 1) return static_cast<int64_t>(b) * p.Hq + h * p.g + c;
  const int32_t j = c / p.n_q, i = c - (c / p.n_q) * p.n_q;
  return (static_cast<int64_t>(b) * p.n_q + i) * p.Hq + h * p.g + j;
}

// (b, head, hc) -> unit
KVQ_HD int32_t unit_of(const Params& p, int32_t b, int32_t h, int32_t hc) {
  const int32_t s = p.slot[h];
  if (p.prot[h] == 1) return (b * p.n_prot + s) * p.NHC + hc;
  if (p.prot[h] == 2) return p.plan.U_p + (b * p.n_konly + s) * p.NHC + hc;
  return p.plan.U_p + p.plan.U_k + (b * p.n_packed + s) * p.NHC + hc;
}

// Rows of the visual segments.  Protected K rows hold the protected heads
// then the K-only heads; packed V rows hold the packed heads then the
// K-only heads.
KVQ_HD int64_t prot_k_row(const Params& p, int32_t b, int cls, int32_t slot) {
  return static_cast<int64_t>(b) * (p.n_prot + p.n_konly) + (cls == kClsKonly ? p.n_prot : 0) + slot;
}
KVQ_HD int64_t packed_v_row(const Params& p, int32_t b, int cls, int32_t slot) {
  return static_cast<int64_t>(b) * (p.n_packed + p.n_konly) + (cls == kClsKonly ? p.n_packed : 0) + slot;
}

}  // namespace kvq

// Host helpers implemented in kvq_layout.cpp.
kvq_status kvq_check_layout(const kvq_layout* L);
void kvq_fill_params(const kvq_layout* L, kvq::Params* p);
// n_q: query tokens per sequence (multi-query decode; 1 otherwise).
kvq::Plan kvq_make_plan(const kvq_layout* L, int32_t T, int32_t n_chunks_target, int32_t n_q = 1);
// The cut table cuts[0..P->C] of a plan (see the decomposition above); sets
// the plan's per-unit chunk fields.
void kvq_plan_cuts(kvq::Plan* P, kvq::Cut* cuts);
int kvq_device_sm_count(int* n_sm);
// Record a failed CUDA call for kvq_last_cuda_error(); returns KVQ_ERR_CUDA.
kvq_status kvq_cuda_fail(int err);
// Launch `fn(*p)` with programmatic stream serialisation allowed, so that its
// CTAs may be scheduled while the previous kernel in the stream drains (the
// kernel itself waits with griddepcontrol.wait before touching memory).
int kvq_launch_pdl(const void* fn, unsigned grid, unsigned block, size_t smem, void* stream,
                   kvq::Params* p);
