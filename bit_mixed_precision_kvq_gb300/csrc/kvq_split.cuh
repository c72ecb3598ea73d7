// kvq_split.cuh -- split-KV partial attention over the mixed-precision cache.
//
// Flash-decoding with on-chip reconstruction (WSVD summary, section 2.라):
// cache tiles are streamed into shared memory, unpacked and dequantised in
// registers, and consumed at once by QK, an online softmax and PV; nothing
// dequantised is ever written to device memory.
//
// CTA = 1 producer warp + 11 consumer warps, one CTA per SM.
//   producer : one lane walks the CTA's tiles and issues 1-D bulk async
//              copies (TMA) of the tile's K/V rows (+ scale/zero rows) into a
//              5-stage ring of 32 KB stages, signalled by mbarriers.
//   consumers: the CTA's blocks (32 positions, or 64 for long packed
//              chunks) are dealt round-robin to the 11 warps across tile
//              boundaries (every warp still waits for and releases every
//              tile, which keeps the mbarrier phases exact).  QK and PV run on
//              the tensor cores (mma.sync m16n8k16, fp16 in, fp32 accumulate)
//              with the unit's <= 8 query columns as N = 8; a block is two (or
//              four) 16-row MMA halves sharing one softmax update:
//                QK: S^T[t][j] = K[t][:] . q[j][:]    (M = 16 positions)
//                PV: O^T[d][j] += V^T[d][t] P^T[t][j] (M = 16 of the D rows)
//              Packed codes enter the MMAs as exact fp16 subnormals (a code
//              masked in place at mantissa bits [p, p + b) is c * 2^(p - 24));
//              the storage order of the rows (kvq.h) makes every operand
//              register one AND of a word.  Per quantisation group
//                q.k_hat = s_g * sum_g q c + z_g * sum_g q
//              (the z-term on the tensor cores as well); for V the scales
//              fold into the B operand (s * P^T per group) and the zeros
//              accumulate in a separate MMA fragment.  Details at the
//              fragment builders below.
// Per unit piece the 11 warps' (m, l, o) are merged in shared memory and
// either finish the unit (fused step, unit held by one CTA) or go to the
// workspace slot (unit + chunk) for the cross-split combine.
#pragma once

#include "kvq_device.cuh"
#include "kvq_ptx.cuh"

namespace kvq {

// 11 consumers + 1 producer = 12 warps, 3 per SM sub-partition (latency
// hiding for the unpack chains); each sub-partition's 16K registers then
// allow 168 registers per thread.
constexpr int kConsumerWarps = 11;
constexpr int kSplitThreads = (kConsumerWarps + 1) * 32;
constexpr int kStagesCl = 5;                   // cluster mode: 5 x 40 KB = 200 KB in flight per CTA
constexpr int kStagesGl = 4;                   // global mode: 4 x 40 KB (its warp merge needs 46 KB)
constexpr int kTileBf16 = 80;                  // positions per bf16 tile: 80 * 512 B = 40 KB
constexpr int kBf16VOff = kTileBf16 * 2 * kD;  // V rows start 20 KB into a bf16 stage
// Cluster mode: text tiles of at most 16 rows (a text prefix, the step's
// row) go to a small stage of their own, so that a CTA's whole piece can be
// resident at once (16 CTAs of a bf16 head's unit hold ~200 KB each).
constexpr int kTextStageRows = 16;
constexpr int kTextVOff = kTextStageRows * 2 * kD;     // V rows start 4 KB into the text stage
constexpr int kTextStageBytes = 2 * kTextVOff;
constexpr uint32_t kPrefetchBytes = 32 * 1024;  // L2 prefetch before the dependency wait
constexpr int kNoLimit = 1 << 30;              // kblock: no multi-query column limit
constexpr int kMaxClusterCtas = 16;            // cluster mode: CTAs per cluster (at most)

// Cluster mode: one rank's partial of a column (o row, then M and L).
constexpr uint32_t kRecvBytes = (kD + 2) * 4;

// Shared memory of the split kernel, per combine mode.
template <bool kCl>
struct SplitSmem;

template <>
struct SplitSmem<true> {  // cluster mode
  static constexpr int kRing = kStagesCl;
  alignas(128) uint8_t stage[kRing][kStageBytes];
  alignas(128) uint8_t tstage[kTextStageBytes];  // short text tiles
  // CTA rank j receives column j's partial of every rank r here (o row,
  // then M and L), stored by rank r.
  alignas(16) float recv[kMaxClusterCtas][kD + 4];
  float merge_ml[kConsumerWarps][kNH][2];
  float qsum[kConsumerWarps][kNH][4];
  uint64_t full[kRing];
  uint64_t empty[kRing];
  uint64_t full_t, empty_t;  // the text stage
  uint64_t recv_bar;         // the other ranks' partials landed (transaction bytes)
  int abort;
  int role, ncomb;           // (global mode only)
};

template <>
struct SplitSmem<false> {  // global mode
  static constexpr int kRing = kStagesGl;
  alignas(128) uint8_t stage[kRing][kStageBytes];
  alignas(128) uint8_t tstage[16];  // (no text stage in global mode)
  // the consumer warps' o rows at a unit's end, merged after one barrier
  alignas(16) float merge_o[kConsumerWarps][kNH][kD + 4];  // padded rows: fewer bank conflicts
  float merge_ml[kConsumerWarps][kNH][2];
  float qsum[kConsumerWarps][kNH][4];
  uint64_t full[kRing];
  uint64_t empty[kRing];
  uint64_t full_t, empty_t;  // (unused)
  uint64_t recv_bar;         // (unused)
  int abort;
  int role;   // fused step: combine role of this CTA for the current unit
  int ncomb;  // fused step: CTAs combining the current unit
};

// A bounded wait gave up (or a counter was found corrupt): mark the call's
// status word and this CTA's outputs.
template <typename Sm>
__device__ __forceinline__ void report_failure(const Params& p, Sm& sm, uint32_t bit) {
  sm.abort = 1;
  if (p.status) atomicOr(p.status, bit);
}

// Tile kinds: bf16 text rows, bf16 protected visual rows, packed visual
// rows, K-only visual rows (bf16 K + packed V).
enum TileKind { kTileText = 0, kTileProt = 1, kTilePacked = 2, kTileKonly = 3 };

// Walk the tiles of one piece [ps, pe) of a unit of class cls: text prefix,
// visual block, text suffix, each cut into tiles.  f(kind, t0, n).
template <bool kGen, typename F>
__device__ __forceinline__ void walk_piece(const Params& p, int cls, int ps, int pe, F&& f) {
  const int b1 = max(ps, min(pe, p.vs)), b2 = max(ps, min(pe, p.ve));
#pragma unroll 1
  for (int seg = 0; seg < 3; ++seg) {  // selects, not an array: no local memory
    const int s0 = seg == 0 ? ps : (seg == 1 ? b1 : b2);
    const int s1 = seg == 0 ? b1 : (seg == 1 ? b2 : pe);
    int kind, tt;
    if constexpr (kGen) {
      kind = seg == 1 ? (cls == kClsProt ? kTileProt : (cls == kClsKonly ? kTileKonly : kTilePacked)) : kTileText;
      tt = kind == kTilePacked ? p.tt_pk : (kind == kTileKonly ? p.tt_ko : kTileBf16);
    } else {
      kind = seg == 1 ? (cls == kClsProt ? kTileProt : kTilePacked) : kTileText;
      tt = kind == kTilePacked ? p.tt_pk : kTileBf16;
    }
    for (int t0 = s0; t0 < s1; t0 += tt) f(kind, t0, min(tt, s1 - t0));
  }
}

__device__ __forceinline__ uint32_t round16(uint32_t x) { return (x + 15u) & ~15u; }

// ---------------------------------------------------------------------------
// Producer
// ---------------------------------------------------------------------------
// The bulk copies of one tile, as f(stage offset, source, bytes) calls (2 to
// 4 of them).  In the fused step the step's own row (position Tu - 1 of a
// unit whose sequence attends [0, Tu): the last row of its last text tile)
// comes from the k_new / v_new inputs rather than from the cache row that
// the launch itself writes.
template <bool kStep, bool kGen, typename F>
__device__ __forceinline__ void tile_sources(const Params& p, const UnitInfo& ui, int Tu, int kind,
                                             int t0, int n, F&& f, uint32_t voff = kBf16VOff) {
  if (kGen && kind == kTileKonly) {
    // bf16 K rows (protected K segment) + packed V rows and their scale/zero
    const int64_t krow = prot_k_row(p, ui.b, kClsKonly, ui.slot) * p.Tv + (t0 - p.vs);
    const int64_t vrow = packed_v_row(p, ui.b, kClsKonly, ui.slot) * p.Tv_pad + (t0 - p.vs);
    const uint32_t bv = round16(n * p.vrow), bvs = round16(n * p.vszrow);
    f(0u, p.seg[KVQ_SEG_PROT_K] + krow * (2 * kD), static_cast<uint32_t>(n) * (2 * kD));
    f(static_cast<uint32_t>(p.ko_off_vc), p.seg[KVQ_SEG_V_CODES] + vrow * p.vrow, bv);
    if (bvs) f(static_cast<uint32_t>(p.ko_off_vsz), p.seg[KVQ_SEG_V_SZ] + vrow * p.vszrow, bvs);
  } else if (kind != kTilePacked) {
    int64_t row;
    const uint8_t *ks, *vs;
    int64_t vrow_p = 0;
    if (kind == kTileText) {
      const int tr = t0 < p.vs ? t0 : t0 - p.Tv;
      row = (static_cast<int64_t>(ui.b) * p.Hkv + ui.h) * p.T_text + tr;
      vrow_p = row;
      ks = p.seg[KVQ_SEG_TEXT_K];
      vs = p.seg[KVQ_SEG_TEXT_V];
    } else {
      vrow_p = (static_cast<int64_t>(ui.b) * p.n_prot + ui.slot) * p.Tv + (t0 - p.vs);
      row = kGen ? prot_k_row(p, ui.b, kClsProt, ui.slot) * p.Tv + (t0 - p.vs) : vrow_p;
      ks = p.seg[KVQ_SEG_PROT_K];
      vs = p.seg[KVQ_SEG_PROT_V];
    }
    const uint32_t bytes = static_cast<uint32_t>(n) * (2 * kD);
    if (kStep && kind == kTileText && t0 + n == Tu) {
      const uint32_t head = bytes - 2 * kD;
      const int64_t nrow = (static_cast<int64_t>(ui.b) * p.Hkv + ui.h) * kD;
      if (head) {
        f(0u, ks + row * (2 * kD), head);
        f(voff, vs + vrow_p * (2 * kD), head);
      }
      f(head, reinterpret_cast<const uint8_t*>(p.k_new + nrow), static_cast<uint32_t>(2 * kD));
      f(voff + head, reinterpret_cast<const uint8_t*>(p.v_new + nrow), static_cast<uint32_t>(2 * kD));
    } else {
      f(0u, ks + row * (2 * kD), bytes);
      f(voff, vs + vrow_p * (2 * kD), bytes);
    }
  } else {
    const int64_t row = (static_cast<int64_t>(ui.b) * p.n_packed + ui.slot) * p.Tv_pad + (t0 - p.vs);
    const int64_t vrow = kGen ? packed_v_row(p, ui.b, kClsPacked, ui.slot) * p.Tv_pad + (t0 - p.vs) : row;
    const uint32_t bk = round16(n * p.krow), bv = round16(n * p.vrow);
    const uint32_t bks = round16(n * p.kszrow), bvs = round16(n * p.vszrow);
    f(0u, p.seg[KVQ_SEG_K_CODES] + row * p.krow, bk);
    f(static_cast<uint32_t>(p.pk_off_vc), p.seg[KVQ_SEG_V_CODES] + vrow * p.vrow, bv);
    if (bks) f(static_cast<uint32_t>(p.pk_off_ksz), p.seg[KVQ_SEG_K_SZ] + row * p.kszrow, bks);
    if (bvs) f(static_cast<uint32_t>(p.pk_off_vsz), p.seg[KVQ_SEG_V_SZ] + vrow * p.vszrow, bvs);
  }
}

// Positions attended by sequence b: the plan's T for uniform calls; for
// ragged calls seq_len[b] (decode) or t_new[b] + 1 (fused step, where the
// step position must be a text position), and 0 -- an inactive sequence --
// for an entry outside that range.  Read only after the dependency wait.
template <bool kStep>
__device__ __forceinline__ int seq_end(const Params& p, int b) {
  if (p.seq_len == nullptr) return p.plan.T;
  const int t = p.seq_len[b];
  if constexpr (kStep) {
    const bool ok = t >= 0 && t < p.plan.T && (t < p.vs || t >= p.ve);
    return ok ? t + 1 : 0;
  } else {
    return (t >= 1 && t <= p.plan.T) ? t : 0;
  }
}

// Walk the CTA's tiles: f(unit info, unit end Tu, kind, t0, n).  kEnds:
// clip every unit at its sequence's end (seq_end); the L2 prefetch, issued
// before the dependency wait, walks the unclipped pieces instead.
template <bool kGen, bool kStep, bool kEnds, typename F>
__device__ __forceinline__ void walk_chunk(const Params& p, int c, F&& f) {
  const Cut a = p.cuts[c];
  const Cut e = p.cuts[c + 1];
  const int u_last = chunk_last_unit(p.cuts, c, p.plan.U);
  for (int u = a.u; u <= u_last; ++u) {
    const UnitInfo ui = unit_info<kGen>(p, u);
    const int Tu = kEnds ? seq_end<kStep>(p, ui.b) : p.plan.T;
    const int pe = min((u == e.u) ? e.p : p.plan.T, Tu);
    const int ps = min((u == a.u) ? a.p : 0, pe);
    walk_piece<kGen>(p, ui.cls, ps, pe, [&](int kind, int t0, int n) { f(ui, Tu, kind, t0, n); });
  }
}

// Where a tile is staged: the text stage (cluster mode, text tiles of at
// most kTextStageRows rows) or the ring.  Producer and consumers count the
// tiles of each in walk order: TileSeq::r ring tiles, TileSeq::t text-stage
// tiles so far.
template <bool kCl>
__device__ __forceinline__ bool in_text_stage(int kind, int n) {
  return kCl && kind == kTileText && n <= kTextStageRows;
}
struct TileSeq {
  uint32_t r = 0, t = 0;
};

// Issue the bulk copies of one tile into its stage (waiting, bounded, for the
// stage's previous tile to be released) and advance the sequence.
template <bool kStep, bool kGen, bool kCl>
__device__ __forceinline__ void issue_tile(const Params& p, SplitSmem<kCl>& sm, const UnitInfo& ui, int Tu, int kind,
                                           int t0, int n, TileSeq& seq) {
  uint8_t* dst;
  uint64_t* full;
  uint32_t voff = kBf16VOff;
  if (in_text_stage<kCl>(kind, n)) {
    if (seq.t > 0 && !mbar_wait(&sm.empty_t, (seq.t - 1) & 1, p.tile_polls))
      report_failure(p, sm, KVQ_STATUS_TILE_WAIT);
    dst = sm.tstage;
    full = &sm.full_t;
    voff = kTextVOff;
    ++seq.t;
  } else {
    constexpr int kRing = SplitSmem<kCl>::kRing;
    const int st = seq.r % kRing;
    const uint32_t round = seq.r / kRing;
    if (round > 0 && !mbar_wait(&sm.empty[st], (round - 1) & 1, p.tile_polls))
      report_failure(p, sm, KVQ_STATUS_TILE_WAIT);
    dst = sm.stage[st];
    full = &sm.full[st];
    ++seq.r;
  }
  uint32_t total = 0;
  tile_sources<kStep, kGen>(p, ui, Tu, kind, t0, n, [&](uint32_t, const uint8_t*, uint32_t bytes) { total += bytes; },
                            voff);
  mbar_arrive_expect_tx(full, total);
  tile_sources<kStep, kGen>(p, ui, Tu, kind, t0, n, [&](uint32_t off, const uint8_t* src, uint32_t bytes) {
    bulk_g2s(dst + off, src, bytes, full);
  }, voff);
}

// Before griddepcontrol.wait, with preload set in a uniform call: copy the
// CTA's leading tiles (one ring at most) into shared memory, stopping at the
// first tile that holds the fused step's own row (it comes from the previous
// kernel).  Only cache rows are read.  Sound because every kernel of this
// library lets the next kernel in the stream launch only after its own
// dependency wait and after its cache writes are fenced (so when this CTA
// runs, every earlier cache write of the stream's library kernels is in L2);
// the caller enables it only where no other kernel writes the cache just
// before.  Returns the number of tiles issued.
template <bool kStep, bool kGen, bool kCl>
__device__ __forceinline__ uint32_t producer_preload(const Params& p, SplitSmem<kCl>& sm, int c) {
  if (!kCl || !p.preload || p.seq_len != nullptr) return 0;
  uint32_t it = 0;
  TileSeq seq;
  bool stop = false;
  walk_chunk<kGen, kStep, true>(p, c, [&](const UnitInfo& ui, int Tu, int kind, int t0, int n) {
    const bool full = in_text_stage<kCl>(kind, n) ? seq.t >= 1 : seq.r >= static_cast<uint32_t>(SplitSmem<kCl>::kRing);
    if (stop || full || (kStep && kind == kTileText && t0 + n == Tu)) {
      stop = true;
      return;
    }
    issue_tile<kStep, kGen, kCl>(p, sm, ui, Tu, kind, t0, n, seq);
    ++it;
  });
  return it;
}

// Before griddepcontrol.wait (after the early tile copies are issued): the
// query rows of the chunk's units into L2 -- the consumers need them before
// any tile (single-query units read nh consecutive rows of D bf16).
template <bool kGen>
__device__ __forceinline__ void prefetch_q(const Params& p, int c) {
  const Cut a = p.cuts[c];
  const int u_last = chunk_last_unit(p.cuts, c, p.plan.U);
  for (int u = a.u; u <= u_last; ++u) {
    const UnitInfo ui = unit_info<kGen>(p, u);
    const int c0 = ui.hc * kNH;
    if (kGen && p.n_q > 1) {
      const int nh = min(kNH, p.g * p.n_q - c0);
      for (int j = 0; j < nh; ++j) prefetch_l2(p.q + col_row(p, ui.b, ui.h, c0 + j) * kD, 2 * kD);
    } else {
      const int nh = min(kNH, p.g - c0);
      prefetch_l2(p.q + (static_cast<int64_t>(ui.b) * p.Hq + ui.h * p.g + c0) * kD,
                  static_cast<uint32_t>(nh) * 2 * kD);
    }
  }
}

// Pull the CTA's next cache rows (after the `skip` tiles already copied)
// into L2 -- a stage's worth, or in cluster mode the rest of the chunk --
// so that the copies issued later hit L2: before griddepcontrol.wait when
// nothing was copied early (L2 is coherent with every SM's stores, so a line
// that the previous kernel writes later is simply updated there), else right
// after it, off the path of the early copies.  More only delays the first
// tile and q behind the other SMs' prefetches.
template <bool kGen, bool kCl>
__device__ __forceinline__ void producer_prefetch(const Params& p, int c, uint32_t skip) {
  uint32_t budget = kCl ? 0xffffffffu : kPrefetchBytes;
  uint32_t k = 0;
  walk_chunk<kGen, false, false>(p, c, [&](const UnitInfo& ui, int Tu, int kind, int t0, int n) {
    if (k++ < skip || budget == 0) return;
    tile_sources<false, kGen>(p, ui, Tu, kind, t0, n, [&](uint32_t, const uint8_t* src, uint32_t bytes) {
      const uint32_t b = min(bytes, budget);
      if (b) prefetch_l2(src, b);
      budget -= b;
    });
  });
}

// The fused step's own K/V row (position Tu - 1, from k_new / v_new) into
// the cache's text segment, for the units (column chunk 0) whose last
// position this CTA holds.  The whole producer warp, after the dependency wait:
// lanes 0-15 the K row, 16-31 the V row, 16 bytes each; then a fence, so the
// row is visible before this CTA lets the next kernel launch.
template <bool kGen>
__device__ __forceinline__ void write_step_rows(const Params& p, int c, int lane) {
  const Cut a = p.cuts[c];
  const Cut e = p.cuts[c + 1];
  const int u_last = chunk_last_unit(p.cuts, c, p.plan.U);
  bool wrote = false;
  for (int u = a.u; u <= u_last; ++u) {
    const UnitInfo ui = unit_info<kGen>(p, u);
    if (ui.hc != 0) continue;
    const int Tu = seq_end<true>(p, ui.b);
    const int pe = min((u == e.u) ? e.p : p.plan.T, Tu);
    const int ps = min((u == a.u) ? a.p : 0, pe);
    if (ps >= pe || pe != Tu) continue;
    const int tr = Tu - 1 < p.vs ? Tu - 1 : Tu - 1 - p.Tv;
    const int64_t bh = static_cast<int64_t>(ui.b) * p.Hkv + ui.h;
    const int half = lane >> 4, q = lane & 15;
    const uint4 w = __ldcg(reinterpret_cast<const uint4*>((half ? p.v_new : p.k_new) + bh * kD) + q);
    uint8_t* dst = const_cast<uint8_t*>(p.seg[half ? KVQ_SEG_TEXT_V : KVQ_SEG_TEXT_K]) +
                   (bh * p.T_text + tr) * (2 * kD) + 16 * q;
    *reinterpret_cast<uint4*>(dst) = w;
    wrote = true;
  }
  if (wrote) __threadfence();
}

// After the dependency wait: the CTA's tiles from ring position `skip` on
// (the first `skip` were issued by producer_preload).
template <bool kStep, bool kGen, bool kCl>
__device__ __forceinline__ void producer_loop(const Params& p, SplitSmem<kCl>& sm, int c, uint32_t skip) {
  uint32_t it = 0;
  TileSeq seq;
  walk_chunk<kGen, kStep, true>(p, c, [&](const UnitInfo& ui, int Tu, int kind, int t0, int n) {
    if (it >= skip) {
      issue_tile<kStep, kGen, kCl>(p, sm, ui, Tu, kind, t0, n, seq);
    } else if (in_text_stage<kCl>(kind, n)) {
      ++seq.t;
    } else {
      ++seq.r;
    }
    ++it;
  });
}

// ---------------------------------------------------------------------------
// Fragment builders.  Lane = 4*gid + tig.
//
// QK A operand (rows = positions gid and gid+8 of a 16-position block,
// K index = d).  The K index is permuted so that each lane reads 8
// consecutive d of a row: k-step pair P (k-steps 2P, 2P+1) covers
// d in [32P, 32P+32), lane tig owns d0 = 32P + 8*tig .. d0+7 and places
//   k-step 2P  : slots (2tig, 2tig+1) <- (d0, d0+4), slots (2tig+8, 2tig+9) <- (d0+1, d0+5)
//   k-step 2P+1: slots (2tig, 2tig+1) <- (d0+2, d0+6), slots (2tig+8, 2tig+9) <- (d0+3, d0+7)
// i.e. register i of pair P holds (d0 + i, d0 + i + 4).  The q operand (B)
// is loaded with the same permutation.  Each k-step pair stays inside one
// quantisation group (G >= 32).
//
// Packed codes enter the tensor cores as exact fp16 subnormals: a b-bit
// code masked in place at mantissa bits [p, p + b) of a half is the value
// c * 2^(p - 24), so one AND (after at most one shift of the word) yields
// a whole operand register.  The storage order of the rows (kvq.h) puts
// the codes of each register at one bit offset p, and makes p the same for
// the four registers of a K k-step pair; V registers may differ in p from
// row to row of the output (their factor is applied per row).
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint2 lds64(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

// bf16 elements -> fp16 pair.
__device__ __forceinline__ uint32_t bf16pair_f16(uint32_t lo_word, bool lo_hi, uint32_t hi_word, bool hi_hi) {
  const float a = lo_hi ? bf16_hi(lo_word) : bf16_lo(lo_word);
  const float b = hi_hi ? bf16_hi(hi_word) : bf16_lo(hi_word);
  return pack_f16x2(a, b);
}

// bf16x2 -> f16x2 (lo stays lo).
__device__ __forceinline__ uint32_t bf16x2_f16x2(uint32_t x) { return pack_f16x2(bf16_lo(x), bf16_hi(x)); }

// Four fp16 pairs (d0,d0+4), (d0+1,d0+5), (d0+2,d0+6), (d0+3,d0+7) of one
// bf16 row's 8 elements starting at d0 = 32P + 8 tig.
__device__ __forceinline__ void k_bf16_pairs(const uint8_t* row, int P, int tig, uint32_t (&f)[4]) {
  const uint4 r = lds128(row + 2 * (32 * P + 8 * tig));
  f[0] = bf16pair_f16(r.x, false, r.z, false);
  f[1] = bf16pair_f16(r.x, true, r.z, true);
  f[2] = bf16pair_f16(r.y, false, r.w, false);
  f[3] = bf16pair_f16(r.y, true, r.w, true);
}

// Packed K: all 16 operand registers f[P][i] (pair P, register i) of one
// row from the lane's slice (slots 32 tig .. 32 tig + 31).  Bit offsets:
//   b = 2: word floor(i/2); P = 0..3 at p = 8, 6, 4, 2 -- member i mod 2 = 0
//          from the word (P = 3: the word << 2), member 1 from the word >> 6
//          (P = 3: the word itself)
//   b = 4: word i; nibble P, P = 0, 1 from the word, 2, 3 from the word >> 8;
//          p = 0, 4, 0, 4
//   b = 8: word 2P + floor(i/2); byte i mod 2 (the word, the word >> 8); p = 0
template <int KB>
__device__ __forceinline__ void k_packed_regs(const uint8_t* row, int tig, uint32_t (&f)[4][4]) {
  if constexpr (KB == 2) {
    const uint2 w = lds64(row + 8 * tig);
    const uint32_t x[2] = {w.x, w.y};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t y = x[h] >> 6, z = x[h] << 2;
      f[0][2 * h] = x[h] & 0x03000300u;
      f[0][2 * h + 1] = y & 0x03000300u;
      f[1][2 * h] = x[h] & 0x00C000C0u;
      f[1][2 * h + 1] = y & 0x00C000C0u;
      f[2][2 * h] = x[h] & 0x00300030u;
      f[2][2 * h + 1] = y & 0x00300030u;
      f[3][2 * h] = z & 0x000C000Cu;
      f[3][2 * h + 1] = x[h] & 0x000C000Cu;
    }
  } else if constexpr (KB == 4) {
    const uint4 w = lds128(row + 16 * tig);
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t y = x[i] >> 8;
      f[0][i] = x[i] & 0x000F000Fu;
      f[1][i] = x[i] & 0x00F000F0u;
      f[2][i] = y & 0x000F000Fu;
      f[3][i] = y & 0x00F000F0u;
    }
  } else {
    const uint4 a = lds128(row + 32 * tig), b = lds128(row + 32 * tig + 16);
    const uint32_t x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int P = 0; P < 4; ++P)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t v = x[2 * P + (i >> 1)];
        f[P][i] = ((i & 1) ? (v >> 8) : v) & 0x00FF00FFu;
      }
  }
}

// 2^e as a compile-time float.
__host__ __device__ constexpr float pow2i(int e) {
  float r = 1.f;
  for (int i = 0; i < (e < 0 ? -e : e); ++i) r = e < 0 ? r * 0.5f : r * 2.f;
  return r;
}

// Bit offset p of K pair P, and 2^(24 - p) (undoes the subnormal placement).
template <int KB>
__host__ __device__ constexpr int kKShift(int P) {
  return KB == 2 ? 8 - 2 * P : (KB == 4 ? 4 * (P & 1) : 0);
}
template <int KB>
__host__ __device__ constexpr float kKFactor(int P) { return pow2i(24 - kKShift<KB>(P)); }

// V operand registers.  Packed V rows: lane gid reads its slice (slots
// 16 gid .. 16 gid + 15 = elements d = 16m + 8r + gid, code index k = 2m + r)
// of the positions of a register pair, merges the two rows' half-words with
// one PRMT and masks every code in place:
//   b = 2: half-word floor(k/8), crumb c = k mod 8 at p = 2c (c <= 4) or
//          from the merged word >> 6 at p = 2c - 6 (c >= 5)
//   b = 4: half-word floor(k/4), nibble c = k mod 4; c = 0, 1 from the
//          merged word, 2, 3 from it >> 8; p = 0, 4, 0, 4
//   b = 8: half-word m, byte r; p = 0
// Output row (m-tile m, row gid + 8r) <-> element d = 16m + 8r + gid.
template <int VB>
__host__ __device__ constexpr int kVShift(int m, int r) {
  return VB == 2 ? ((2 * m + r) % 8 <= 4 ? 2 * ((2 * m + r) % 8) : 2 * ((2 * m + r) % 8) - 6)
                 : VB == 4 ? 4 * (r & 1) : 0;
}

// Online-softmax state of one warp for its unit: m, l for the lane's two
// query-head columns (2tig, 2tig+1); o^T fragments for 8 m-tiles of d.
// Packed units with packed V keep, while in "packed" accumulation, o rows
// in units of 2^(p - 24) of the row's V codes times scales, and zo (an MMA
// fragment: row = group, columns = heads) the sum of p * z per group.
struct Acc {
  float m[2], l[2];
  float o[8][4];
  float zo[4];
};

// Both halves of a half2 register as floats (the split is a register view).
__device__ __forceinline__ void h2_to_f2(uint32_t w, float& lo, float& hi) {
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(w));
}

// QK for one 16-row half [r0, r0 + 16) of a block of bf16 K rows: S[i] for
// rows (gid, gid, gid+8, gid+8) x heads (2tig, 2tig+1, 2tig, 2tig+1), log2
// units.
__device__ __forceinline__ void qk_bf16(const uint8_t* kc, int r0, float sl2, const uint32_t (&qb)[8][2],
                                        int gid, int tig, float (&S)[4]) {
  const uint8_t* krow0 = kc + (r0 + gid) * (2 * kD);
  const uint8_t* krow1 = krow0 + 8 * (2 * kD);
  float C[4][4];
#pragma unroll
  for (int P = 0; P < 4; ++P) {
    C[P][0] = C[P][1] = C[P][2] = C[P][3] = 0.f;
    uint32_t f0[4], f1[4];
    k_bf16_pairs(krow0, P, tig, f0);
    k_bf16_pairs(krow1, P, tig, f1);
    const uint32_t A0[4] = {f0[0], f1[0], f0[1], f1[1]};
    const uint32_t A1[4] = {f0[2], f1[2], f0[3], f1[3]};
    mma_f16(C[P], A0, qb[2 * P][0], qb[2 * P][1]);
    mma_f16(C[P], A1, qb[2 * P + 1][0], qb[2 * P + 1][1]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) S[i] = ((C[0][i] + C[1][i]) + (C[2][i] + C[3][i])) * sl2;
}

// QK for one 16-row half of packed K rows.  Per quantisation group g:
//   q . k_hat = s_g * sum_g q c + z_g * sum_g q,  sum_g q c = 2^(24-p) * (MMA)
// The z-term runs on the tensor cores too: A = the rows' z (fp16, rows =
// positions, K index = group), B = zb = sl2 * 2^-6 * (sum of q over each
// group) as an fp16 hi + lo pair (two MMAs, ~22 bits), scaled back by 2^6.
// The scale/zero row is fp16 [z_0 .., s_0 ..].
constexpr float kZbScale = 64.f;  // zb holds the q sums / 64 (fp16 range)
template <int KB, int G>
__device__ __forceinline__ void qk_packed(const uint8_t* kc, const uint8_t* ksz, int r0, float sl2,
                                          const uint32_t (&qb)[8][2], const uint32_t (&zb)[2], int gid,
                                          int tig, float (&S)[4]) {
  constexpr int KROW = KB * kD / 8;
  constexpr int NG = kD / G;
  constexpr int SZROW = 4 * NG;
  constexpr int PPG = G / 32;
  uint32_t f0[4][4], f1[4][4];
  k_packed_regs<KB>(kc + (r0 + gid) * KROW, tig, f0);
  k_packed_regs<KB>(kc + (r0 + gid + 8) * KROW, tig, f1);
  float C[4][4];
#pragma unroll
  for (int P = 0; P < 4; ++P) {
    C[P][0] = C[P][1] = C[P][2] = C[P][3] = 0.f;
    const uint32_t A0[4] = {f0[P][0], f1[P][0], f0[P][1], f1[P][1]};
    const uint32_t A1[4] = {f0[P][2], f1[P][2], f0[P][3], f1[P][3]};
    mma_f16(C[P], A0, qb[2 * P][0], qb[2 * P][1]);
    mma_f16(C[P], A1, qb[2 * P + 1][0], qb[2 * P + 1][1]);
  }
  const uint8_t* p0 = ksz + (r0 + gid) * SZROW;
  const uint8_t* p1 = p0 + 8 * SZROW;
  // z-term
  float Z[4] = {0.f, 0.f, 0.f, 0.f};
  {
    uint32_t za = 0u, zc = 0u;
    if (tig < (NG + 1) / 2) {  // z halves 2 tig, 2 tig + 1
      za = lds32(p0 + 4 * tig);
      zc = lds32(p1 + 4 * tig);
      if constexpr (NG == 1) {  // the word's high half is s_0
        za &= 0x0000ffffu;
        zc &= 0x0000ffffu;
      }
    }
    const uint32_t A[4] = {za, zc, 0u, 0u};
    mma_f16(Z, A, zb[0], 0u);
    mma_f16(Z, A, zb[1], 0u);
  }
  // scales of rows gid and gid + 8
  float s0f[NG], s1f[NG];
  if constexpr (NG == 4) {
    const uint2 a = lds64(p0 + 8), b = lds64(p1 + 8);
    h2_to_f2(a.x, s0f[0], s0f[1]);
    h2_to_f2(a.y, s0f[2], s0f[3]);
    h2_to_f2(b.x, s1f[0], s1f[1]);
    h2_to_f2(b.y, s1f[2], s1f[3]);
  } else if constexpr (NG == 2) {
    h2_to_f2(lds32(p0 + 4), s0f[0], s0f[1]);
    h2_to_f2(lds32(p1 + 4), s1f[0], s1f[1]);
  } else {
    float zz;
    h2_to_f2(lds32(p0), zz, s0f[0]);
    h2_to_f2(lds32(p1), zz, s1f[0]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) S[i] = Z[i] * kZbScale;
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const int P0 = g * PPG;
    float Cg[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      Cg[i] = C[P0][i];
#pragma unroll
      for (int k = 1; k < PPG; ++k) Cg[i] = fmaf(C[P0 + k][i], kKFactor<KB>(P0 + k) / kKFactor<KB>(P0), Cg[i]);
    }
    const float kf = sl2 * kKFactor<KB>(P0);
    const float a0 = s0f[g] * kf, a1 = s1f[g] * kf;
    S[0] = fmaf(a0, Cg[0], S[0]);
    S[1] = fmaf(a0, Cg[1], S[1]);
    S[2] = fmaf(a1, Cg[2], S[2]);
    S[3] = fmaf(a1, Cg[3], S[3]);
  }
}

// Masks of the halves of a position pair (t, t+1) that lie below n.
__device__ __forceinline__ uint32_t pair_mask(int t, int n) {
  return (t < n ? 0x0000ffffu : 0u) | (t + 1 < n ? 0xffff0000u : 0u);
}

// PV for one 16-row half, bf16 V rows, output rows d = 16 gid + mt (row gid)
// and 16 gid + 8 + mt (row gid + 8) -- the protected-unit mapping.
__device__ __forceinline__ void pv_bf16_lanecols(const uint8_t* vc, int r0, int n, uint32_t pb0,
                                                 uint32_t pb1, int gid, int tig, Acc& acc) {
  const int t[4] = {r0 + 2 * tig, r0 + 2 * tig + 1, r0 + 2 * tig + 8, r0 + 2 * tig + 9};
  uint32_t w[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint8_t* r = vc + t[i] * (2 * kD) + 32 * gid;
    const uint4 x = lds128(r), y = lds128(r + 16);
    w[i][0] = x.x; w[i][1] = x.y; w[i][2] = x.z; w[i][3] = x.w;
    w[i][4] = y.x; w[i][5] = y.y; w[i][6] = y.z; w[i][7] = y.w;
  }
  // Rows past n hold stale shared memory (possibly NaN/Inf patterns): zero
  // their V operands so that 0 * garbage cannot reach the accumulators.
  const bool ragged = r0 + 16 > n;
  const uint32_t ma = ragged ? pair_mask(t[0], n) : 0xffffffffu;
  const uint32_t mc = ragged ? pair_mask(t[2], n) : 0xffffffffu;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int e0 = mt, e1 = 8 + mt;  // local elements of rows gid, gid + 8
    uint32_t A[4] = {bf16pair_f16(w[0][e0 >> 1], e0 & 1, w[1][e0 >> 1], e0 & 1),
                     bf16pair_f16(w[0][e1 >> 1], e1 & 1, w[1][e1 >> 1], e1 & 1),
                     bf16pair_f16(w[2][e0 >> 1], e0 & 1, w[3][e0 >> 1], e0 & 1),
                     bf16pair_f16(w[2][e1 >> 1], e1 & 1, w[3][e1 >> 1], e1 & 1)};
    if (ragged) {
      A[0] &= ma;
      A[1] &= ma;
      A[2] &= mc;
      A[3] &= mc;
    }
    mma_f16(acc.o[mt], A, pb0, pb1);
  }
}

// ldmatrix .x4 .trans: four transposed 8x8 b16 tiles; lane L supplies the
// row address of tile L / 8.
__device__ __forceinline__ void ldsm_x4_trans(const uint8_t* addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(addr)));
}

// PV for one 16-row half, bf16 V rows, packed-unit mapping (output row
// gid + 8r of m-tile m <-> d = 16m + 8r + gid): the V^T operand of m-tile m
// is the transpose of V[t0 .. t0+15][16m .. 16m+15], loaded with ldmatrix.
__device__ __forceinline__ void pv_bf16_dcols(const uint8_t* vc, int r0, int n, uint32_t pb0, uint32_t pb1,
                                              int tig, int lane, Acc& acc) {
  const uint8_t* base = vc + (r0 + (lane & 7) + ((lane >> 4) & 1) * 8) * (2 * kD) + ((lane >> 3) & 1) * 16;
  const bool ragged = r0 + 16 > n;
  const uint32_t ma = ragged ? pair_mask(r0 + 2 * tig, n) : 0xffffffffu;
  const uint32_t mc = ragged ? pair_mask(r0 + 2 * tig + 8, n) : 0xffffffffu;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    uint32_t r[4];
    ldsm_x4_trans(base + 32 * m, r);
    uint32_t A[4] = {bf16x2_f16x2(r[0]) & ma, bf16x2_f16x2(r[1]) & ma, bf16x2_f16x2(r[2]) & mc,
                     bf16x2_f16x2(r[3]) & mc};
    mma_f16(acc.o[m], A, pb0, pb1);
  }
}

// PV for one 16-row half of packed V rows (packed accumulation):
//   sum_t p_t v_hat_td = 2^(24-p_d) * sum_t (c_td 2^(p_d-24)) (s_tg p_t) + sum_t z_tg p_t
// The first sum runs on the tensor cores with B = s * P^T per group; the
// second accumulates into zo by one more MMA (rows = groups, A = z).
template <int VB, int G>
__device__ __forceinline__ void pv_packed(const uint8_t* vc, const uint8_t* vsz, int r0, int n,
                                          uint32_t pb0, uint32_t pb1, int gid, int tig, Acc& acc) {
  constexpr int VROW = VB * kD / 8;
  constexpr int SLICE = 2 * VB;  // bytes of a lane slice
  constexpr int NG = kD / G;
  constexpr int SZROW = 4 * NG;
  const int t[4] = {r0 + 2 * tig, r0 + 2 * tig + 1, r0 + 2 * tig + 8, r0 + 2 * tig + 9};
  const bool ragged = r0 + 16 > n;
  const uint32_t ma = ragged ? pair_mask(t[0], n) : 0xffffffffu;
  const uint32_t mc = ragged ? pair_mask(t[2], n) : 0xffffffffu;
  // scale/zero rows of the four positions
  uint32_t sz[4][(2 * NG + 1) / 2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint8_t* p = vsz + t[i] * SZROW;
    if constexpr (NG == 4) {
      const uint4 a = lds128(p);
      sz[i][0] = a.x; sz[i][1] = a.y; sz[i][2] = a.z; sz[i][3] = a.w;
    } else if constexpr (NG == 2) {
      const uint2 a = lds64(p);
      sz[i][0] = a.x; sz[i][1] = a.y;
    } else {
      sz[i][0] = lds32(p);
    }
  }
  // fp16 halves: z_g at half g, s_g at half NG + g
  auto half_sel = [](int h) { return (h & 1) ? 0x7632u : 0x5410u; };
  uint32_t b0[NG], b1[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const int hs = NG + g;
    uint32_t sa = prmt(sz[0][hs >> 1], sz[1][hs >> 1], half_sel(hs));
    uint32_t sc = prmt(sz[2][hs >> 1], sz[3][hs >> 1], half_sel(hs));
    if (ragged) {
      sa &= ma;
      sc &= mc;
    }
    b0[g] = hmul2_u(pb0, sa);
    b1[g] = hmul2_u(pb1, sc);
  }
  // zo += Z (rows = groups) x P^T
  {
    uint32_t za = 0u, zc = 0u;
    if (gid < NG) {
      const int wsel = gid >> 1;
      const uint32_t w0 = (NG == 4 && wsel) ? sz[0][1] : sz[0][0];
      const uint32_t w1 = (NG == 4 && wsel) ? sz[1][1] : sz[1][0];
      const uint32_t w2 = (NG == 4 && wsel) ? sz[2][1] : sz[2][0];
      const uint32_t w3 = (NG == 4 && wsel) ? sz[3][1] : sz[3][0];
      za = prmt(w0, w1, half_sel(gid));
      zc = prmt(w2, w3, half_sel(gid));
      if (ragged) {
        za &= ma;
        zc &= mc;
      }
    }
    const uint32_t Z[4] = {za, 0u, zc, 0u};
    mma_f16(acc.zo, Z, pb0, pb1);
  }
  // code words of the lane's slice for the four positions
  constexpr int NW = VB / 2;  // words per slice
  uint32_t cw[4][NW];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint8_t* p = vc + t[i] * VROW + SLICE * gid;
    if constexpr (VB == 2) {
      cw[i][0] = lds32(p);
    } else if constexpr (VB == 4) {
      const uint2 a = lds64(p);
      cw[i][0] = a.x; cw[i][1] = a.y;
    } else {
      const uint4 a = lds128(p);
      cw[i][0] = a.x; cw[i][1] = a.y; cw[i][2] = a.z; cw[i][3] = a.w;
    }
  }
  constexpr int NH = 16 / VB;   // codes per half-word
  constexpr int MPH = NH / 2;   // m-tiles per half-word (>= 1)
#pragma unroll
  for (int h = 0; h < VB; ++h) {  // half-words of the slice
    const uint32_t xa = prmt(cw[0][h >> 1], cw[1][h >> 1], half_sel(h));
    const uint32_t xc = prmt(cw[2][h >> 1], cw[3][h >> 1], half_sel(h));
    const uint32_t ya = VB == 2 ? (xa >> 6) : (xa >> 8);
    const uint32_t yc = VB == 2 ? (xc >> 6) : (xc >> 8);
#pragma unroll
    for (int mm = 0; mm < MPH; ++mm) {
      const int m = h * MPH + mm;
      uint32_t A[4];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int c = 2 * mm + r;  // code index inside the half-word
        const bool hi = VB == 2 ? (c >= 5) : (VB == 4 ? (c >= 2) : (c >= 1));
        const uint32_t mask = (VB == 2 ? 0x00030003u : (VB == 4 ? 0x000F000Fu : 0x00FF00FFu))
                              << kVShift<VB>(m, r);
        A[r] = (hi ? ya : xa) & mask;
        A[2 + r] = (hi ? yc : xc) & mask;
      }
      const int g = (16 * m) / G;
      mma_f16(acc.o[m], A, b0[g], b1[g]);
    }
  }
}

// Switch a packed unit's accumulator between bf16 ("true") rows and packed
// accumulation.  to_packed: o <- o * 2^(p-24), zo <- 0.  to_true: o <- o *
// 2^(24-p) + zo[group of the row], zo <- 0 (zo of group g for heads 2tig,
// 2tig+1 lives in lane 4g + tig).
template <int VB>
__device__ __forceinline__ void acc_to_packed(Acc& acc) {
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const float f0 = pow2i(kVShift<VB>(m, 0) - 24);
    const float f1 = pow2i(kVShift<VB>(m, 1) - 24);
    acc.o[m][0] *= f0;
    acc.o[m][1] *= f0;
    acc.o[m][2] *= f1;
    acc.o[m][3] *= f1;
  }
  acc.zo[0] = acc.zo[1] = acc.zo[2] = acc.zo[3] = 0.f;
}

template <int VB, int G>
__device__ __forceinline__ void acc_to_true(Acc& acc, int tig) {
  constexpr int NG = kD / G;
  float z0[NG], z1[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    z0[g] = __shfl_sync(0xffffffffu, acc.zo[0], 4 * g + tig);
    z1[g] = __shfl_sync(0xffffffffu, acc.zo[1], 4 * g + tig);
  }
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const float f0 = pow2i(24 - kVShift<VB>(m, 0));
    const float f1 = pow2i(24 - kVShift<VB>(m, 1));
    const int g = (16 * m) / G;
    acc.o[m][0] = fmaf(acc.o[m][0], f0, z0[g]);
    acc.o[m][1] = fmaf(acc.o[m][1], f0, z1[g]);
    acc.o[m][2] = fmaf(acc.o[m][2], f1, z0[g]);
    acc.o[m][3] = fmaf(acc.o[m][3], f1, z1[g]);
  }
  acc.zo[0] = acc.zo[1] = acc.zo[2] = acc.zo[3] = 0.f;
}

// K / V paths of a block.
enum KPath { kKBf16 = 0, kKPacked = 1 };
enum VPath { kVBf16Lane = 0, kVBf16D = 1, kVPacked = 2 };

// One block [r0, r0 + 16 NH) of a staged tile (n valid positions): NH
// 16-row MMA halves sharing one online-softmax update.
template <int NH, int KP, int VP, int KB, int VB, int G>
__device__ __forceinline__ void kblock(const uint8_t* kc, const uint8_t* ksz, const uint8_t* vc,
                                       const uint8_t* vsz, int r0, int n, int lim0, int lim1, float sl2,
                                       const uint32_t (&qb)[8][2], const uint32_t (&zb)[2], int gid,
                                       int tig, int lane, Acc& acc) {
  float S[NH][4];
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    if (h == 0 || r0 + 16 * h < n) {
      if constexpr (KP == kKPacked) qk_packed<KB, G>(kc, ksz, r0 + 16 * h, sl2, qb, zb, gid, tig, S[h]);
      else qk_bf16(kc, r0 + 16 * h, sl2, qb, gid, tig, S[h]);
    } else {
      S[h][0] = S[h][1] = S[h][2] = S[h][3] = -INFINITY;
    }
  }
  if (r0 + 16 * NH > n) {  // ragged block: mask rows past n
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      if (r0 + 16 * h + gid >= n) S[h][0] = S[h][1] = -INFINITY;
      if (r0 + 16 * h + gid + 8 >= n) S[h][2] = S[h][3] = -INFINITY;
    }
  }
  // Multi-query (general kernels): column 2tig (2tig + 1) sees the rows
  // below lim0 (lim1); the other callers pass the constant kNoLimit, which
  // removes this code from their instantiations.
  if ((lim0 != kNoLimit || lim1 != kNoLimit) && min(lim0, lim1) < r0 + 16 * NH) {
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const int ra = r0 + 16 * h + gid;
      if (ra >= lim0) S[h][0] = -INFINITY;
      if (ra >= lim1) S[h][1] = -INFINITY;
      if (ra + 8 >= lim0) S[h][2] = -INFINITY;
      if (ra + 8 >= lim1) S[h][3] = -INFINITY;
    }
  }

  // ---- online softmax over the block (columns = heads 2tig, 2tig+1) ----
  float mx0 = fmaxf(S[0][0], S[0][2]), mx1 = fmaxf(S[0][1], S[0][3]);
#pragma unroll
  for (int h = 1; h < NH; ++h) {
    mx0 = fmaxf(mx0, fmaxf(S[h][0], S[h][2]));
    mx1 = fmaxf(mx1, fmaxf(S[h][1], S[h][3]));
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
  }
  const float mn0 = fmaxf(acc.m[0], mx0), mn1 = fmaxf(acc.m[1], mx1);
  const float b0s = mn0 == -INFINITY ? 0.f : mn0, b1s = mn1 == -INFINITY ? 0.f : mn1;
  const float c0 = ex2(acc.m[0] - b0s), c1 = ex2(acc.m[1] - b1s);
  float P[NH][4];
  float l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    P[h][0] = ex2(S[h][0] - b0s);
    P[h][1] = ex2(S[h][1] - b1s);
    P[h][2] = ex2(S[h][2] - b0s);
    P[h][3] = ex2(S[h][3] - b1s);
    l0 += P[h][0] + P[h][2];
    l1 += P[h][1] + P[h][3];
  }
  acc.m[0] = mn0;
  acc.m[1] = mn1;
  acc.l[0] = fmaf(acc.l[0], c0, l0);
  acc.l[1] = fmaf(acc.l[1], c1, l1);
  if (!__all_sync(0xffffffffu, c0 == 1.f && c1 == 1.f)) {  // some running max moved
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      acc.o[mt][0] *= c0;
      acc.o[mt][1] *= c1;
      acc.o[mt][2] *= c0;
      acc.o[mt][3] *= c1;
    }
    if constexpr (VP == kVPacked) {  // zo is non-zero only during packed accumulation
      acc.zo[0] *= c0;
      acc.zo[1] *= c1;
      acc.zo[2] *= c0;
      acc.zo[3] *= c1;
    }
  }
  // P^T as the B operand of PV: transpose the 8x8 quarters.
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    if (h > 0 && r0 + 16 * h >= n) break;
    const uint32_t pa0 = movmatrix_trans(pack_f16x2(P[h][0], P[h][1]));
    const uint32_t pa1 = movmatrix_trans(pack_f16x2(P[h][2], P[h][3]));
    if constexpr (VP == kVPacked) pv_packed<VB, G>(vc, vsz, r0 + 16 * h, n, pa0, pa1, gid, tig, acc);
    else if constexpr (VP == kVBf16D) pv_bf16_dcols(vc, r0 + 16 * h, n, pa0, pa1, tig, lane, acc);
    else pv_bf16_lanecols(vc, r0 + 16 * h, n, pa0, pa1, gid, tig, acc);
  }
}

// ---------------------------------------------------------------------------
// Cross-split combine of one output row: column j of unit u, whose partials
// sit in slots u + cf .. u + cl.  NW warps fold the slots with online
// rescaling (warp w takes slots cf + 8w .. cf + 8w + 7, then the next 8 NW;
// the eight loads of a batch are issued before any is used; lane l owns
// d = 4l .. 4l+3), the warp states are merged through shared memory and
// warp 0 writes out[orow] and lse[orow].  Partials are read from L2 (other
// SMs wrote them).  A NaN partial max (a failed wait) or force_nan makes the
// row NaN.  `bar` synchronises the NW warps.
// ---------------------------------------------------------------------------
template <int NW, typename Bar>
__device__ __forceinline__ void combine_row(const Params& p, int u, int j, int cf, int cl,
                                            int64_t orow, int warp, int lane, float (*sm_ml)[2],
                                            float4 (*sm_o)[32], bool force_nan, Bar&& bar) {
  float M = -INFINITY, L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  bool bad = force_nan;
  for (int c0 = cf + 8 * warp; c0 <= cl; c0 += 8 * NW) {
    float mb[8], lb[8];
    float4 ob[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      mb[k] = -INFINITY;
      lb[k] = 0.f;
      ob[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c0 + k <= cl) {
        const int64_t s = (static_cast<int64_t>(u) + c0 + k) * kNH + j;
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + s);
        mb[k] = ml.x;
        lb[k] = ml.y;
        ob[k] = __ldcg(reinterpret_cast<const float4*>(p.ws_o + s * kD) + lane);
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
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    sm_ml[warp][0] = bad ? __int_as_float(0x7fffffff) : M;
    sm_ml[warp][1] = L;
  }
  sm_o[warp][lane] = O;
  bar();
  if (warp == 0) {
    float Mt = -INFINITY;
    bool nan = false;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float m = sm_ml[w][0];
      if (m != m) nan = true; else Mt = fmaxf(Mt, m);
    }
    float Lt = 0.f;
    float4 Ot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float m = sm_ml[w][0];
      if (m == -INFINITY || m != m) continue;
      const float sc = exp2f(m - Mt);
      Lt = fmaf(sm_ml[w][1], sc, Lt);
      const float4 o = sm_o[w][lane];
      Ot.x = fmaf(o.x, sc, Ot.x);
      Ot.y = fmaf(o.y, sc, Ot.y);
      Ot.z = fmaf(o.z, sc, Ot.z);
      Ot.w = fmaf(o.w, sc, Ot.w);
    }
    float inv = Lt > 0.f ? 1.0f / Lt : 0.f;  // Lt = 0: an inactive sequence (out 0, lse -inf)
    if (nan) inv = __int_as_float(0x7fffffff);
    uint2 packed;
    packed.x = static_cast<uint32_t>(f32_to_bf16_bits(Ot.x * inv)) |
               (static_cast<uint32_t>(f32_to_bf16_bits(Ot.y * inv)) << 16);
    packed.y = static_cast<uint32_t>(f32_to_bf16_bits(Ot.z * inv)) |
               (static_cast<uint32_t>(f32_to_bf16_bits(Ot.w * inv)) << 16);
    reinterpret_cast<uint2*>(p.out + orow * kD)[lane] = packed;
    if (lane == 0 && p.lse) p.lse[orow] = nan ? inv : 0.69314718055994531f * (Mt + log2f(Lt));
  }
  bar();  // the shared scratch is reused next
}

// Fused step: wait (bounded) until the unit's last arrival has reset its
// counter to zero.
__device__ __forceinline__ bool wait_unit_released(const uint32_t* cnt, uint32_t polls) {
  for (uint32_t i = 0; i < polls; ++i) {
    if (ld_acquire_gpu(cnt) == 0u) return true;
    __nanosleep(32);
  }
  return false;
}

// Cluster mode, after the consumer warps' barrier (every tile consumed,
// merge_ml published; consumer threads only).  The CTA's partial of column
// j < nh -- its warps' o rows scaled to the CTA's running max M and summed
// in warp order, and (M, L) -- goes to slot [this rank] of CTA rank j's
// receive rows: asynchronous stores that complete on rank j's receive
// barrier (a plain store for j = this rank).  The warps' scaled rows meet in
// the staged-tile ring, idle now (one unit per CTA).  CTA rank j < nh then
// waits (bounded) for the other ranks' slots and writes column j's output
// row, orow; a CTA that receives nothing is done once its stores are issued.
__device__ __forceinline__ void cluster_push_combine(const Params& p, SplitSmem<true>& sm, const Acc& acc, bool prot,
                                                     int nh, int64_t orow, int warp, int lane) {
  constexpr int kPitch = kD + 4;  // padded rows: the fragment stores spread over the banks
  const int gid = lane >> 2, tig = lane & 3;
  const int ctid = threadIdx.x;
  float* scr = reinterpret_cast<float*>(sm.stage[0]);  // [warp][kNH][kPitch]
  {
    float sc[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int j = 2 * tig + e;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm.merge_ml[w][j][0]);
      sc[e] = (M == -INFINITY) ? 0.f : exp2f(sm.merge_ml[warp][j][0] - M);
    }
    // Output rows: packed units d = 16 mt + gid (+ 8), stored at slot d;
    // protected units d = 16 gid + mt (+ 8), stored at slot
    // (d mod 16) * 8 + d / 16 = 8 mt + gid (+ 64) -- both spread a warp's
    // stores over all banks.  The receiver reads slot_of(d).
    float* r0 = scr + (warp * kNH + 2 * tig) * kPitch;
    float* r1 = r0 + kPitch;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int q0 = prot ? 8 * mt + gid : 16 * mt + gid, q1 = q0 + (prot ? 64 : 8);
      r0[q0] = acc.o[mt][0] * sc[0];
      r1[q0] = acc.o[mt][1] * sc[1];
      r0[q1] = acc.o[mt][2] * sc[0];
      r1[q1] = acc.o[mt][3] * sc[1];
    }
  }
  named_bar(1, kConsumerWarps * 32);
  cluster_wait();  // every rank's receive barrier is initialised (arrived at kernel start)
  const int rank = static_cast<int>(cluster_ctarank()), cs = p.plan.cs;
  if (ctid < nh * 32) {  // column j, slots d .. d + 3
    const int j = ctid >> 5, d = (ctid & 31) * 4;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float4 x = *reinterpret_cast<const float4*>(scr + (w * kNH + j) * kPitch + d);
      o.x += x.x;
      o.y += x.y;
      o.z += x.z;
      o.w += x.w;
    }
    float* dst = &sm.recv[rank][d];
    if (j == rank) *reinterpret_cast<float4*>(dst) = o;
    else st_async_v4(dsmem_addr(dst, j), o, dsmem_addr(&sm.recv_bar, j));
  } else if (ctid >= 256 && ctid < 256 + nh) {  // column j's (M, L)
    const int j = ctid - 256;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm.merge_ml[w][j][0]);
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float sc = (M == -INFINITY) ? 0.f : exp2f(sm.merge_ml[w][j][0] - M);
      L = fmaf(sm.merge_ml[w][j][1], sc, L);
    }
    if (sm.abort) M = __int_as_float(0x7fffffff);  // NaN marks a failed wait
    float* dst = &sm.recv[rank][kD];
    const float2 ml = make_float2(M, L);
    if (j == rank) *reinterpret_cast<float2*>(dst) = ml;
    else st_async_v2(dsmem_addr(dst, j), ml, dsmem_addr(&sm.recv_bar, j));
  }
  if (rank >= nh) return;
  named_bar(1, kConsumerWarps * 32);  // this CTA's own slot is written
  if (ctid >= kD) return;
  const bool ok = mbar_wait_cluster(&sm.recv_bar, 0, p.tile_polls);
  if (!ok) report_failure(p, sm, KVQ_STATUS_PEER_WAIT);
  // Every receiving warp forms the cs weights itself, lane r for rank r.
  float mr = -INFINITY, lr = 0.f;
  if (lane < cs) {
    mr = sm.recv[lane][kD];
    lr = sm.recv[lane][kD + 1];
  }
  const bool bad = __any_sync(0xffffffffu, !ok || mr != mr);
  float M = mr != mr ? -INFINITY : mr;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float w = (mr == -INFINITY || mr != mr || M == -INFINITY) ? 0.f : exp2f(mr - M);
  float L = lr * w;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  const int d = ctid, slot = prot ? (d & 15) * 8 + (d >> 4) : d;
  float O = 0.f;
#pragma unroll
  for (int r = 0; r < kMaxClusterCtas; ++r) {
    const float wr = __shfl_sync(0xffffffffu, w, r);
    if (r < cs) O = fmaf(sm.recv[r][slot], wr, O);
  }
  if (bad) M = __int_as_float(0x7fffffff);
  const float inv = (M != M) ? M : (L > 0.f ? 1.0f / L : 0.f);  // L = 0: inactive sequence
  p.out[orow * kD + d] = f32_to_bf16_bits(O * inv);
  if (d == 0 && p.lse) p.lse[orow] = (M != M) ? M : 0.69314718055994531f * (M + log2f(L));
}

template <int KB, int VB, int G, bool kStep, int NHP, bool kGen, bool kCl>
__device__ __forceinline__ void consumer_loop(const Params& p, SplitSmem<kCl>& sm, int c, int warp, int lane) {
  constexpr int kRing = SplitSmem<kCl>::kRing;
  const int gid = lane >> 2, tig = lane & 3;
  const int ctid = warp * 32 + lane;  // 0 .. 32*kConsumerWarps-1
  const Cut a = p.cuts[c];
  const Cut e = p.cuts[c + 1];
  const int u_last = chunk_last_unit(p.cuts, c, p.plan.U);
  constexpr int ppg = G / 32;
  const float sl2 = p.scale_log2;
  uint32_t it = 0;    // tiles seen
  TileSeq seq;        // ... of them in the ring and in the text stage
  uint32_t gblk = 0;  // 32-position blocks dealt so far (round-robin over warps)
  // q of unit uu for lane (gid, tig): elements 32P + 8 tig .. + 7 of head
  // column gid, P = 0..3 (zero past the unit's columns), through L2 (the
  // previous kernel may have written q).  In global mode with 32-position
  // blocks (short units, several per CTA) the next unit's loads are issued
  // before this unit's warp merge, so they land during it; the other
  // kernels load q at the unit's start.
  constexpr bool kPrefQ = !kCl && NHP == 2;
  uint4 qraw[4];
  auto load_q = [&](int uu, uint4 (&r)[4]) {
    const UnitInfo un = unit_info<kGen>(p, uu);
    const int c0n = un.hc * kNH;
    const int nhn = kGen ? min(kNH, p.g * p.n_q - c0n) : min(kNH, p.g - c0n);
    int64_t row;
    if constexpr (kGen) row = col_row(p, un.b, un.h, c0n + (gid < nhn ? gid : 0));
    else row = static_cast<int64_t>(un.b) * p.Hq + un.h * p.g + c0n + gid;
#pragma unroll
    for (int P = 0; P < 4; ++P)
      r[P] = gid < nhn ? __ldcg(reinterpret_cast<const uint4*>(p.q + row * kD + 32 * P + 8 * tig))
                       : make_uint4(0u, 0u, 0u, 0u);
  };
  for (int u = a.u; u <= u_last; ++u) {
    const UnitInfo ui = unit_info<kGen>(p, u);
    // The unit's columns: query heads h*g + hc*kNH + j; in the general
    // kernels (head, token) pairs of a multi-query call, rows via col_row.
    const int c0 = ui.hc * kNH;
    const int hq0 = ui.h * p.g + c0;
    const int nh = kGen ? min(kNH, p.g * p.n_q - c0) : min(kNH, p.g - c0);
    auto out_row = [&](int j) -> int64_t {
      if constexpr (kGen) return col_row(p, ui.b, ui.h, c0 + j);
      else return static_cast<int64_t>(ui.b) * p.Hq + hq0 + j;
    };
    if (u == a.u) {
      pdl_wait();  // q (and the cache) may come from the previous kernel
      if constexpr (kPrefQ) load_q(u, qraw);
    }
    const int Tu = seq_end<kStep>(p, ui.b);
    const int pe = min((u == e.u) ? e.p : p.plan.T, Tu);
    const int ps = min((u == a.u) ? a.p : 0, pe);
    // Multi-query (general kernels): the ends of the lane's two columns
    // (token i does not see the unit's last n_q - 1 - i positions, all text).
    const int endA = kGen ? Tu - (p.n_q - 1 - (c0 + 2 * tig) % p.n_q) : Tu;
    const int endB = kGen ? Tu - (p.n_q - 1 - (c0 + 2 * tig + 1) % p.n_q) : Tu;

    // q of head column gid as the B operand, in the permuted d order; group sums.
    uint32_t qb[8][2];
    float qpart[4];
#pragma unroll
    for (int P = 0; P < 4; ++P) {
      uint4 raw = make_uint4(0u, 0u, 0u, 0u);
      if constexpr (kPrefQ) {
        raw = qraw[P];
      } else if (gid < nh) {
        raw = __ldcg(reinterpret_cast<const uint4*>(p.q + out_row(gid) * kD + 32 * P + 8 * tig));
      }
      const float x[8] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y),
                          bf16_lo(raw.z), bf16_hi(raw.z), bf16_lo(raw.w), bf16_hi(raw.w)};
      qb[2 * P][0] = pack_f16x2(x[0], x[4]);
      qb[2 * P][1] = pack_f16x2(x[1], x[5]);
      qb[2 * P + 1][0] = pack_f16x2(x[2], x[6]);
      qb[2 * P + 1][1] = pack_f16x2(x[3], x[7]);
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) sum += __half2float(__float2half_rn(x[i]));
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      qpart[P] = sum;
    }
    if (tig == 0) {
#pragma unroll
      for (int P = 0; P < 4; ++P) sm.qsum[warp][gid][P] = qpart[P];
    }
    __syncwarp();
    // zb: B operand of the K z-term MMA -- (k = groups 2 tig, 2 tig + 1, n =
    // head gid) of sl2 / 64 * (sum of q over the group), as hi + lo fp16.
    uint32_t zb[2];
    {
      constexpr int NG = kD / G;
      float x[2] = {0.f, 0.f};
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int g = 2 * tig + cc;
        if (g < NG) {
          float s = 0.f;
#pragma unroll
          for (int i = 0; i < ppg; ++i) s += sm.qsum[warp][gid][g * ppg + i];
          x[cc] = s * (sl2 / kZbScale);
        }
      }
      zb[0] = pack_f16x2(x[0], x[1]);
      float h0, h1;
      h2_to_f2(zb[0], h0, h1);
      zb[1] = pack_f16x2(x[0] - h0, x[1] - h1);
    }

    Acc acc;
    acc.m[0] = acc.m[1] = -INFINITY;
    acc.l[0] = acc.l[1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) acc.o[mt][0] = acc.o[mt][1] = acc.o[mt][2] = acc.o[mt][3] = 0.f;
    acc.zo[0] = acc.zo[1] = acc.zo[2] = acc.zo[3] = 0.f;
    bool packed_acc = false;  // packed accumulation (see Acc); packed units only

    // Wait for a tile; voff: where its bf16 V rows start in the stage.
    uint32_t voff = kBf16VOff;
    bool in_text = false;
    auto begin_tile = [&](int kind, int, int n) -> const uint8_t* {
      in_text = in_text_stage<kCl>(kind, n);
      uint64_t* full = in_text ? &sm.full_t : &sm.full[seq.r % kRing];
      const uint32_t parity = in_text ? (seq.t & 1) : ((seq.r / kRing) & 1);
      if (!mbar_wait(full, parity, p.tile_polls)) report_failure(p, sm, KVQ_STATUS_TILE_WAIT);
      voff = in_text ? kTextVOff : kBf16VOff;
      return in_text ? sm.tstage : sm.stage[seq.r % kRing];
    };
    // Release the tile's stage once this warp is done with it.
    auto end_tile = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(in_text ? &sm.empty_t : &sm.empty[seq.r % kRing]);
      if (in_text) ++seq.t;
      else ++seq.r;
      ++it;
    };
    // This warp's blocks (bs rows each) of a tile of n rows: first, first + 11, ...
    auto deal = [&](int n, int bs, int& first) {
      const int nb = (n + bs - 1) / bs;
      first = (warp + kConsumerWarps - static_cast<int>(gblk % kConsumerWarps)) % kConsumerWarps;
      gblk += nb;
      return nb;
    };
    if (ui.prot) {  // protected unit: bf16 rows only
      walk_piece<kGen>(p, kClsProt, ps, pe, [&](int kind, int t0, int n) {
        const uint8_t* base = begin_tile(kind, t0, n);
        int first;
        const int nb = deal(n, 32, first);
        for (int kb = first; kb < nb; kb += kConsumerWarps)
          kblock<2, kKBf16, kVBf16Lane, 16, 16, G>(base, nullptr, base + voff, nullptr, kb * 32, n,
                                                  kGen && kind == kTileText ? endA - t0 : kNoLimit,
                                                  kGen && kind == kTileText ? endB - t0 : kNoLimit, sl2, qb,
                                                  zb, gid, tig, lane, acc);
        end_tile();
      });
    } else {
      walk_piece<kGen>(p, ui.cls, ps, pe, [&](int kind, int t0, int n) {
        const uint8_t* base = begin_tile(kind, t0, n);
        int first;
        if (kind == kTilePacked) {
          const int nb = deal(n, 16 * NHP, first);
          if constexpr (VB < 16) {
            if (first < nb && !packed_acc) {
              acc_to_packed<VB>(acc);
              packed_acc = true;
            }
          }
          for (int kb = first; kb < nb; kb += kConsumerWarps)
            kblock<NHP, (KB < 16 ? kKPacked : kKBf16), (VB < 16 ? kVPacked : kVBf16D), KB, VB, G>(
                base, base + p.pk_off_ksz, base + p.pk_off_vc, base + p.pk_off_vsz, kb * 16 * NHP, n,
                kNoLimit, kNoLimit, sl2, qb, zb, gid, tig, lane, acc);
        } else if (kGen && kind == kTileKonly) {  // bf16 K + packed V
          const int nb = deal(n, 32, first);
          if constexpr (VB < 16) {
            if (first < nb && !packed_acc) {
              acc_to_packed<VB>(acc);
              packed_acc = true;
            }
          }
          for (int kb = first; kb < nb; kb += kConsumerWarps)
            kblock<2, kKBf16, (VB < 16 ? kVPacked : kVBf16D), 16, VB, G>(
                base, nullptr, base + p.ko_off_vc, base + p.ko_off_vsz, kb * 32, n, kNoLimit, kNoLimit, sl2,
                qb, zb, gid, tig, lane, acc);
        } else {  // text rows of a packed or K-only unit
          const int nb = deal(n, 32, first);
          if constexpr (VB < 16) {
            if (first < nb && packed_acc) {
              acc_to_true<VB, G>(acc, tig);
              packed_acc = false;
            }
          }
          for (int kb = first; kb < nb; kb += kConsumerWarps)
            kblock<2, kKBf16, kVBf16D, 16, 16, G>(base, nullptr, base + voff, nullptr, kb * 32, n,
                                                 kGen ? endA - t0 : kNoLimit, kGen ? endB - t0 : kNoLimit, sl2,
                                                 qb, zb, gid, tig, lane, acc);
        }
        end_tile();
      });
    }

    if constexpr (VB < 16) {
      if (packed_acc) acc_to_true<VB, G>(acc, tig);
    }
    if constexpr (kPrefQ) {
      if (u < u_last) load_q(u + 1, qraw);
    }
    // ---- merge the warps' states and write the partial of (u, c) ----
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      acc.l[0] += __shfl_xor_sync(0xffffffffu, acc.l[0], off);
      acc.l[1] += __shfl_xor_sync(0xffffffffu, acc.l[1], off);
    }
    if (gid == 0) {
      sm.merge_ml[warp][2 * tig][0] = acc.m[0];
      sm.merge_ml[warp][2 * tig][1] = acc.l[0];
      sm.merge_ml[warp][2 * tig + 1][0] = acc.m[1];
      sm.merge_ml[warp][2 * tig + 1][1] = acc.l[1];
    }
    // The fused step finishes a unit held by this CTA alone right here;
    // otherwise the partial goes to slot u + c (global mode) or, in cluster
    // mode, to this CTA's shared memory for the cluster's combine.
    constexpr bool cluster = kCl;
    int cf = c, cl = c;
    if constexpr (kStep) plan_unit_chunks(p.plan, p.cuts, u, &cf, &cl);
    const bool sole = kStep && !cluster && cf == cl;
    if constexpr (kCl) {
      named_bar(1, kConsumerWarps * 32);  // every tile consumed, merge_ml published
      cluster_push_combine(p, sm, acc, ui.prot, nh, out_row(static_cast<int>(cluster_ctarank()) < nh
                                                                    ? static_cast<int>(cluster_ctarank()) : 0),
                           warp, lane);
    } else {
      // Every warp's o rows as they are (output rows: protected units
      // d = 16 gid + mt (+ 8), packed units d = 16 mt + gid (+ 8)); after one
      // barrier each thread forms (column j, element d) from all warps in
      // warp order (reproducible bit for bit).
      auto store_rows = [&](int dbase, int dstep) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int d0 = dbase + dstep * mt, d1 = d0 + 8;
          sm.merge_o[warp][2 * tig][d0] = acc.o[mt][0];
          sm.merge_o[warp][2 * tig + 1][d0] = acc.o[mt][1];
          sm.merge_o[warp][2 * tig][d1] = acc.o[mt][2];
          sm.merge_o[warp][2 * tig + 1][d1] = acc.o[mt][3];
        }
      };
      if (ui.prot) store_rows(16 * gid, 1);
      else store_rows(gid, 16);
      named_bar(1, kConsumerWarps * 32);
      const int64_t slot = static_cast<int64_t>(u) + c;
      for (int idx = ctid; idx < nh * kD; idx += kConsumerWarps * 32) {
        const int j = idx / kD, d = idx - j * kD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm.merge_ml[w][j][0]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float sc = exp2f(sm.merge_ml[w][j][0] - M);
            L = fmaf(sm.merge_ml[w][j][1], sc, L);
            O = fmaf(sm.merge_o[w][j][d], sc, O);
          }
        }
        if (sm.abort) M = __int_as_float(0x7fffffff);  // NaN marks a failed wait
        if (sole) {
          const float inv = (M != M) ? M : (L > 0.f ? 1.0f / L : 0.f);  // L = 0: inactive sequence
          const int64_t orow = out_row(j);
          p.out[orow * kD + d] = f32_to_bf16_bits(O * inv);
          if (d == 0 && p.lse) p.lse[orow] = (M != M) ? M : 0.69314718055994531f * (M + log2f(L));
        } else {
          p.ws_o[(slot * kNH + j) * kD + d] = O;
          if (d == 0) {
            p.ws_ml[(slot * kNH + j) * 2] = M;
            p.ws_ml[(slot * kNH + j) * 2 + 1] = L;
          }
        }
      }
      named_bar(1, kConsumerWarps * 32);
      if constexpr (kStep) {
        if (!sole) {
          // Publish the partial.  The last min(n, nh) arrivals at the unit's
          // counter (n = its chunks) combine its rows, arrival n - nh + r
          // taking rows r, r + min(n, nh), ...; the very last one resets the
          // counter to zero (for the next call), which also releases the
          // others, who wait (bounded) for that.  An arrival that finds the
          // counter at n or more (it was not zero when the call started)
          // reports it and writes NaN rows.
          if (ctid == 0) {
            __threadfence();
            const uint32_t n = static_cast<uint32_t>(cl - cf + 1);
            const uint32_t nc = min(n, static_cast<uint32_t>(nh));
            const uint32_t k = atomicAdd(&p.cnt[u], 1u);
            int role = -1;
            if (k >= n) {
              report_failure(p, sm, KVQ_STATUS_COUNTER);
              role = -2;
            } else if (k == n - 1) {
              __threadfence();
              atomicExch(&p.cnt[u], 0u);
              role = static_cast<int>(nc) - 1;
            } else if (k >= n - nc) {
              role = static_cast<int>(k - (n - nc));
              if (!wait_unit_released(&p.cnt[u], p.peer_polls)) report_failure(p, sm, KVQ_STATUS_PEER_WAIT);
            }
            __threadfence();
            sm.role = role;
            sm.ncomb = static_cast<int>(nc);
          }
          named_bar(1, kConsumerWarps * 32);
          const int role = sm.role, nc = sm.ncomb;
          if (role == -2) {  // corrupt counter: every row of the unit becomes NaN
            for (int idx = ctid; idx < nh * kD; idx += kConsumerWarps * 32) {
              const int j = idx / kD, d = idx - j * kD;
              const int64_t orow = out_row(j);
              p.out[orow * kD + d] = 0x7fffu;  // bf16 NaN
              if (d == 0 && p.lse) p.lse[orow] = __int_as_float(0x7fffffff);
            }
          } else if (role >= 0) {
            const bool bad = sm.abort != 0;
            float (*sm_ml)[2] = reinterpret_cast<float (*)[2]>(&sm.merge_ml[0][0][0]);
            float4 (*sm_o)[32] = reinterpret_cast<float4 (*)[32]>(&sm.merge_o[0][0][0]);
            for (int j = role; j < nh; j += nc)
              combine_row<kConsumerWarps>(p, u, j, cf, cl, out_row(j), warp, lane, sm_ml, sm_o, bad,
                                          []() { named_bar(1, kConsumerWarps * 32); });
          }
        }
      }
    }
  }
}

// NHP: 16-row MMA halves per packed block (2 or 4; the launch's pk_halves).
// kGen: the general variant -- K-only protected heads (a third unit class)
// and multi-query columns; the other variants run neither.
template <int KB, int VB, int G, bool kStep, int NHP, bool kGen, bool kCl>
__global__ void __maxnreg__(168) split_mma_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SplitSmem<kCl>& sm = *reinterpret_cast<SplitSmem<kCl>*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < SplitSmem<kCl>::kRing; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsumerWarps);
    }
    mbar_init(&sm.full_t, 1);
    mbar_init(&sm.empty_t, kConsumerWarps);
    mbar_init(&sm.recv_bar, 1);
    sm.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if constexpr (kCl) {
    // Cluster mode: each CTA expects the other ranks' partials of its column
    // as transaction bytes.  The cluster barrier, arrived at here and waited
    // for before the first store into another CTA (consumers) or before the
    // dependency wait (producer), makes every CTA's receive barrier
    // initialised before any rank stores into it.
    if (threadIdx.x == 0) mbar_arrive_expect_tx(&sm.recv_bar, (p.plan.cs - 1) * kRecvBytes);
    cluster_arrive();
  }
  if (warp == kConsumerWarps) {
    uint32_t pre = 0;
    if (lane == 0) {
      pre = producer_preload<kStep, kGen, kCl>(p, sm, blockIdx.x);
      prefetch_q<kGen>(p, blockIdx.x);
      if (pre == 0) producer_prefetch<kGen, kCl>(p, blockIdx.x, 0);
    }
    __syncwarp();
    if constexpr (kCl) cluster_wait();
    pdl_wait();  // the previous kernel in the stream may have written the cache, k_new, v_new
    if constexpr (kStep) write_step_rows<kGen>(p, blockIdx.x, lane);
    __syncwarp();
    if (lane == 0) {
      // The next kernel in the stream may launch (and read cache rows) from
      // here on: this CTA is past its dependency wait and its cache writes
      // are fenced.
      pdl_launch_dependents();
      if (pre > 0) producer_prefetch<kGen, kCl>(p, blockIdx.x, pre);
      producer_loop<kStep, kGen, kCl>(p, sm, blockIdx.x, pre);
    }
    return;
  }
  consumer_loop<KB, VB, G, kStep, NHP, kGen, kCl>(p, sm, blockIdx.x, warp, lane);
}

}  // namespace kvq
