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
//   consumers: the CTA's 32-position blocks are dealt round-robin to the 11
//              warps across tile boundaries (every warp still waits for and
//              releases every tile, which keeps the mbarrier phases exact).  QK and PV
//              run on the tensor cores (mma.sync m16n8k16, fp16 in, fp32
//              accumulate) with the unit's <= 8 query heads as N = 8; a block
//              is two 16-row MMA halves sharing one softmax update:
//                QK: S^T[t][j] = K[t][:] . q[j][:]    (M = 16 positions)
//                PV: O^T[d][j] += V^T[d][t] P^T[t][j] (M = 16 of the D rows)
//              K codes enter QK as the fp16 values v = 1 + c * 2^-m (code in
//              the mantissa below the 1.0 exponent; m = b for 2/4 bits, 10 for
//              8 bits), so per quantisation group
//                sum_d q_d c_d = 2^m (sum_d q_d v_d - sum_d q_d)
//                q.k_hat = sum_g ( 2^m s_g * sum_g q v + (z_g - 2^m s_g) * sum_g q ).
//              V codes become exact fp16 integers (1024 + c, minus 1024) and are
//              dequantised per element in f16x2 (c*s + z, one rounding)
//              because the PV reduction runs over positions.
// Per unit piece the 4 warps' (m, l, o) are merged in shared memory and
// written to the workspace slot (unit + chunk).
#pragma once

#include "kvq_device.cuh"
#include "kvq_ptx.cuh"

namespace kvq {

// 11 consumers + 1 producer = 12 warps, 3 per SM sub-partition (latency
// hiding for the unpack chains); each sub-partition's 16K registers then
// allow 168 registers per thread.
constexpr int kConsumerWarps = 11;
constexpr int kSplitThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 5;
constexpr int kStageBytes = 32 * 1024;
constexpr int kTileBf16 = 64;                  // positions per bf16 tile: 64 * 512 B = 32 KB
constexpr int kBf16VOff = kTileBf16 * 2 * kD;  // V rows start 16 KB into a bf16 stage
constexpr uint32_t kWaitPolls = 1u << 24;      // bounded mbarrier waits
constexpr uint32_t kSpinPolls = 1u << 21;      // bounded inter-CTA wait (fused step)
constexpr uint32_t kF16Magic = 0x64006400u;    // two fp16 1024.0
constexpr uint32_t kF16One = 0x3C003C00u;      // two fp16 1.0

struct SplitSmem {
  alignas(128) uint8_t stage[kStages][kStageBytes];
  float merge_o[kConsumerWarps][kNH][kD];
  float merge_ml[kConsumerWarps][kNH][2];
  float qsum[kConsumerWarps][kNH][4];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort;
  int role;   // fused step: combine role of this CTA for the current unit
  int ncomb;  // fused step: CTAs combining the current unit
};

enum TileKind { kTileText = 0, kTileProt = 1, kTilePacked = 2 };

// Walk the tiles of one piece [ps, pe) of a unit: text prefix, visual block,
// text suffix, each cut into tiles.  f(kind, t0, n).
template <typename F>
__device__ __forceinline__ void walk_piece(const Params& p, bool prot, int ps, int pe, F&& f) {
  const int b1 = max(ps, min(pe, p.vs)), b2 = max(ps, min(pe, p.ve));
#pragma unroll 1
  for (int seg = 0; seg < 3; ++seg) {  // selects, not an array: no local memory
    const int s0 = seg == 0 ? ps : (seg == 1 ? b1 : b2);
    const int s1 = seg == 0 ? b1 : (seg == 1 ? b2 : pe);
    const int kind = seg == 1 ? (prot ? kTileProt : kTilePacked) : kTileText;
    const int tt = kind == kTilePacked ? p.tt_pk : kTileBf16;
    for (int t0 = s0; t0 < s1; t0 += tt) f(kind, t0, min(tt, s1 - t0));
  }
}

__device__ __forceinline__ uint32_t round16(uint32_t x) { return (x + 15u) & ~15u; }

// ---------------------------------------------------------------------------
// Producer
// ---------------------------------------------------------------------------
// The bulk copies of one tile, as f(stage offset, source, bytes) calls (2 to
// 4 of them).  In the fused step the step's own row (position T - 1, the
// last row of the last text tile) comes from the k_new / v_new inputs rather
// than from the cache row that the launch itself writes.
template <bool kStep, typename F>
__device__ __forceinline__ void tile_sources(const Params& p, const UnitInfo& ui, int kind, int t0,
                                             int n, F&& f) {
  if (kind != kTilePacked) {
    int64_t row;
    const uint8_t *ks, *vs;
    if (kind == kTileText) {
      const int tr = t0 < p.vs ? t0 : t0 - p.Tv;
      row = (static_cast<int64_t>(ui.b) * p.Hkv + ui.h) * p.T_text + tr;
      ks = p.seg[KVQ_SEG_TEXT_K];
      vs = p.seg[KVQ_SEG_TEXT_V];
    } else {
      row = (static_cast<int64_t>(ui.b) * p.n_prot + ui.slot) * p.Tv + (t0 - p.vs);
      ks = p.seg[KVQ_SEG_PROT_K];
      vs = p.seg[KVQ_SEG_PROT_V];
    }
    const uint32_t bytes = static_cast<uint32_t>(n) * (2 * kD);
    if (kStep && kind == kTileText && t0 + n == p.plan.T) {
      const uint32_t head = bytes - 2 * kD;
      const int64_t nrow = (static_cast<int64_t>(ui.b) * p.Hkv + ui.h) * kD;
      if (head) {
        f(0u, ks + row * (2 * kD), head);
        f(static_cast<uint32_t>(kBf16VOff), vs + row * (2 * kD), head);
      }
      f(head, reinterpret_cast<const uint8_t*>(p.k_new + nrow), static_cast<uint32_t>(2 * kD));
      f(kBf16VOff + head, reinterpret_cast<const uint8_t*>(p.v_new + nrow), static_cast<uint32_t>(2 * kD));
    } else {
      f(0u, ks + row * (2 * kD), bytes);
      f(static_cast<uint32_t>(kBf16VOff), vs + row * (2 * kD), bytes);
    }
  } else {
    const int64_t row = (static_cast<int64_t>(ui.b) * p.n_packed + ui.slot) * p.Tv_pad + (t0 - p.vs);
    const uint32_t bk = round16(n * p.krow), bv = round16(n * p.vrow);
    const uint32_t bks = round16(n * p.kszrow), bvs = round16(n * p.vszrow);
    f(0u, p.seg[KVQ_SEG_K_CODES] + row * p.krow, bk);
    f(static_cast<uint32_t>(p.pk_off_vc), p.seg[KVQ_SEG_V_CODES] + row * p.vrow, bv);
    if (bks) f(static_cast<uint32_t>(p.pk_off_ksz), p.seg[KVQ_SEG_K_SZ] + row * p.kszrow, bks);
    if (bvs) f(static_cast<uint32_t>(p.pk_off_vsz), p.seg[KVQ_SEG_V_SZ] + row * p.vszrow, bvs);
  }
}

// Walk the CTA's tiles: f(unit info, kind, t0, n).
template <typename F>
__device__ __forceinline__ void walk_chunk(const Params& p, int c, F&& f) {
  const Cut a = p.cuts[c];
  const Cut e = p.cuts[c + 1];
  const int u_last = chunk_last_unit(p.cuts, c, p.plan.U);
  for (int u = a.u; u <= u_last; ++u) {
    const int ps = (u == a.u) ? a.p : 0;
    const int pe = (u == e.u) ? e.p : p.plan.T;
    const UnitInfo ui = unit_info(p, u);
    walk_piece(p, ui.prot, ps, pe, [&](int kind, int t0, int n) { f(ui, kind, t0, n); });
  }
}

// Before griddepcontrol.wait: pull the first kStages stages' worth of the
// CTA's cache rows into L2.  L2 is coherent with every SM's stores, so a
// line that the previous kernel writes later is simply updated there; the
// copies into shared memory all come after the wait.
__device__ __forceinline__ void producer_prefetch(const Params& p, int c) {
  uint32_t budget = kStages * kStageBytes;
  walk_chunk(p, c, [&](const UnitInfo& ui, int kind, int t0, int n) {
    if (budget == 0) return;
    tile_sources<false>(p, ui, kind, t0, n, [&](uint32_t, const uint8_t* src, uint32_t bytes) {
      const uint32_t b = min(bytes, budget);
      if (b) prefetch_l2(src, b);
      budget -= b;
    });
  });
}

template <bool kStep>
__device__ __forceinline__ void producer_loop(const Params& p, SplitSmem& sm, int c) {
  uint32_t it = 0;
  walk_chunk(p, c, [&](const UnitInfo& ui, int kind, int t0, int n) {
    const int st = it % kStages;
    const uint32_t round = it / kStages;
    if (round > 0 && !mbar_wait(&sm.empty[st], (round - 1) & 1, kWaitPolls)) sm.abort = 1;
    uint8_t* dst = sm.stage[st];
    uint32_t total = 0;
    tile_sources<kStep>(p, ui, kind, t0, n, [&](uint32_t, const uint8_t*, uint32_t bytes) { total += bytes; });
    mbar_arrive_expect_tx(&sm.full[st], total);
    tile_sources<kStep>(p, ui, kind, t0, n, [&](uint32_t off, const uint8_t* src, uint32_t bytes) {
      bulk_g2s(dst + off, src, bytes, &sm.full[st]);
    });
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
// The q operand (B) is loaded with the same permutation.  Each k-step pair
// stays inside one quantisation group (G >= 32).
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint2 lds64(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

// Masked code-field pair -> exact fp16 codes (c_lo, c_hi).
__device__ __forceinline__ uint32_t codes_f16(uint32_t x, uint32_t mask) {
  return hsub2_u(and_or(x, mask, kF16Magic), kF16Magic);
}

// bf16 elements -> fp16 pair.
__device__ __forceinline__ uint32_t bf16pair_f16(uint32_t lo_word, bool lo_hi, uint32_t hi_word, bool hi_hi) {
  const float a = lo_hi ? bf16_hi(lo_word) : bf16_lo(lo_word);
  const float b = hi_hi ? bf16_hi(hi_word) : bf16_lo(hi_word);
  return pack_f16x2(a, b);
}

// Four fp16 pairs (d0,d0+4), (d0+1,d0+5), (d0+2,d0+6), (d0+3,d0+7) of one
// row's 8 elements starting at d0.  KB = bits (16 = bf16 row).
// K code pair -> fp16 (v_lo, v_hi) with v = 1 + c * 2^-m: mask the code
// into the mantissa under the exponent of 1.0.
__device__ __forceinline__ uint32_t kcode_pair(uint32_t x, uint32_t mask) { return and_or(x, mask, kF16One); }

// Four fp16 pairs (d0,d0+4), (d0+1,d0+5), (d0+2,d0+6), (d0+3,d0+7) of one
// row's 8 elements starting at d0.  KB = bits (16 = bf16 row).  For packed
// rows the pairs hold 1 + c * 2^-m (m = kKShift<KB>).
template <int KB>
__device__ __forceinline__ void k_row_pairs(const uint8_t* row, int P, int tig, uint32_t (&f)[4]) {
  if constexpr (KB == 4) {
    // nibble k at bits 4k (and 16 + 4k) -> mantissa bits 6..9
    const uint32_t w = lds32(row + 4 * (4 * P + tig));
    f[0] = kcode_pair(w << 6, 0x03C003C0u);
    f[1] = kcode_pair(w << 2, 0x03C003C0u);
    f[2] = kcode_pair(w >> 2, 0x03C003C0u);
    f[3] = kcode_pair(w >> 6, 0x03C003C0u);
  } else if constexpr (KB == 2) {
    // bytes of the lane's half-word split into the two halves, then
    // crumb k at bits 2k (and 16 + 2k) -> mantissa bits 8..9
    const uint32_t w = lds32(row + 4 * (2 * P + (tig >> 1)));
    const uint32_t h = tig & 1;
    const uint32_t r = prmt(w, 0u, (2 * h) | (4u << 4) | ((2 * h + 1) << 8) | (4u << 12));
    f[0] = kcode_pair(r << 8, 0x03000300u);
    f[1] = kcode_pair(r << 6, 0x03000300u);
    f[2] = kcode_pair(r << 4, 0x03000300u);
    f[3] = kcode_pair(r << 2, 0x03000300u);
  } else if constexpr (KB == 8) {
    // byte k of the two words -> mantissa bits 0..7
    const uint2 w = lds64(row + 4 * (8 * P + 2 * tig));
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t x = prmt(w.x, w.y, k | (k << 4) | ((4 + k) << 8) | ((4 + k) << 12));
      f[k] = kcode_pair(x, 0x00FF00FFu);
    }
  } else {  // bf16 row
    const uint4 r = lds128(row + 2 * (32 * P + 8 * tig));
    f[0] = bf16pair_f16(r.x, false, r.z, false);
    f[1] = bf16pair_f16(r.x, true, r.z, true);
    f[2] = bf16pair_f16(r.y, false, r.w, false);
    f[3] = bf16pair_f16(r.y, true, r.w, true);
  }
}

// 2^m of the K code placement above.
template <int KB>
__host__ __device__ constexpr float kKScale() { return KB == 4 ? 16.f : (KB == 2 ? 4.f : 1024.f); }

// PV A operand (rows = d, K index = positions).  Lane gid owns
// d in [16 gid, 16 gid + 16): m-tile mt row gid <-> d = 16 gid + mt,
// row gid+8 <-> d = 16 gid + 8 + mt.  Positions: a0/a1 use (2tig, 2tig+1),
// a2/a3 use (2tig+8, 2tig+9).
//
// VData holds one lane's 16 d of 4 positions in the storage format.
template <int VB>
struct VData {
  static constexpr int kWords = VB == 16 ? 8 : VB / 2;  // 32-bit words per position
  uint32_t w[4][kWords];
};

template <int VB>
__device__ __forceinline__ void v_load(const uint8_t* vrows, int row_bytes, int gid, const int (&t)[4],
                                       VData<VB>& v) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint8_t* r = vrows + t[i] * row_bytes;
    if constexpr (VB == 2) {
      v.w[i][0] = lds32(r + 4 * gid);
    } else if constexpr (VB == 4) {
      const uint2 x = lds64(r + 8 * gid);
      v.w[i][0] = x.x;
      v.w[i][1] = x.y;
    } else if constexpr (VB == 8) {
      const uint4 x = lds128(r + 16 * gid);
      v.w[i][0] = x.x; v.w[i][1] = x.y; v.w[i][2] = x.z; v.w[i][3] = x.w;
    } else {
      const uint4 x = lds128(r + 32 * gid);
      const uint4 y = lds128(r + 32 * gid + 16);
      v.w[i][0] = x.x; v.w[i][1] = x.y; v.w[i][2] = x.z; v.w[i][3] = x.w;
      v.w[i][4] = y.x; v.w[i][5] = y.y; v.w[i][6] = y.z; v.w[i][7] = y.w;
    }
  }
}

// Code pair (position i0, position i1) for local element e in [0, 16) of the
// lane's d range, as exact fp16 (bf16 rows: the value itself).
template <int VB>
__device__ __forceinline__ uint32_t v_pair(const VData<VB>& v, int i0, int i1, int e) {
  if constexpr (VB == 2) {
    const uint32_t x = prmt(v.w[i0][0], v.w[i1][0], e < 8 ? 0x5410u : 0x7632u);
    return codes_f16(x >> (2 * (e & 7)), 0x00030003u);
  } else if constexpr (VB == 4) {
    const int wi = e >> 3, ee = e & 7;
    const uint32_t x = prmt(v.w[i0][wi], v.w[i1][wi], ee < 4 ? 0x5410u : 0x7632u);
    return codes_f16(x >> (4 * (ee & 3)), 0x000F000Fu);
  } else if constexpr (VB == 8) {
    const int wi = e >> 2, b = e & 3;
    const uint32_t x = prmt(v.w[i0][wi], v.w[i1][wi], b | (b << 4) | ((4 + b) << 8) | ((4 + b) << 12));
    return codes_f16(x, 0x00FF00FFu);
  } else {
    const int wi = e >> 1;
    const bool hi = e & 1;
    return bf16pair_f16(v.w[i0][wi], hi, v.w[i1][wi], hi);
  }
}

// ---------------------------------------------------------------------------
// Consumers
// ---------------------------------------------------------------------------

// Online-softmax state of one warp for its unit: m, l for the lane's two
// query-head columns (2tig, 2tig+1); o^T fragments for 8 m-tiles of d.
struct Acc {
  float m[2], l[2];
  float o[8][4];
};

// Both halves of a half2 register as floats (the split is a register view).
__device__ __forceinline__ void h2_to_f2(uint32_t w, float& lo, float& hi) {
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(w));
}

// QK for one 16-row half [r0, r0 + 16) of a block: S[i] for rows
// (gid, gid, gid+8, gid+8) x heads (2tig, 2tig+1, 2tig, 2tig+1), log2 units.
template <int KB, int G>
__device__ __forceinline__ void qk_half(const uint8_t* kc, const uint8_t* ksz, int r0, float sl2,
                                        const uint32_t (&qb)[8][2], const float (&qsP)[4][2], int gid,
                                        int tig, float (&S)[4]) {
  constexpr int KROW = KB * kD / 8;
  constexpr int SZROW = 4 * (kD / G);
  const uint8_t* krow0 = kc + (r0 + gid) * KROW;
  const uint8_t* krow1 = krow0 + 8 * KROW;
  // One accumulator per k-step pair keeps the MMA dependency chains short.
  float C[4][4];
#pragma unroll
  for (int P = 0; P < 4; ++P) {
    C[P][0] = C[P][1] = C[P][2] = C[P][3] = 0.f;
    uint32_t f0[4], f1[4];
    k_row_pairs<KB>(krow0, P, tig, f0);
    k_row_pairs<KB>(krow1, P, tig, f1);
    const uint32_t A0[4] = {f0[0], f1[0], f0[1], f1[1]};
    const uint32_t A1[4] = {f0[2], f1[2], f0[3], f1[3]};
    mma_f16(C[P], A0, qb[2 * P][0], qb[2 * P][1]);
    mma_f16(C[P], A1, qb[2 * P + 1][0], qb[2 * P + 1][1]);
  }
  if constexpr (KB == 16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) S[i] = ((C[0][i] + C[1][i]) + (C[2][i] + C[3][i])) * sl2;
  } else {
    // Sum the pairs of each quantisation group, then apply its scale/zero:
    // sum q c = 2^m (sum q v - sum q), so 2^m s multiplies the group's sum
    // and (z - 2^m s) multiplies the group's q sum (qsP[P] for any pair P of it).
    constexpr int PPG = G / 32;
#pragma unroll
    for (int P = 0; P < 4; ++P) {
      if (P % PPG != 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) C[P - P % PPG][i] += C[P][i];
      }
    }
    const uint8_t* sz0p = ksz + (r0 + gid) * SZROW;
    const uint8_t* sz1p = sz0p + 8 * SZROW;
    const float sc = kKScale<KB>() * sl2;
    S[0] = S[1] = S[2] = S[3] = 0.f;
#pragma unroll
    for (int g = 0; g < 4 / PPG; ++g) {
      const int P = g * PPG;
      float s0, z0, s1, z1;
      h2_to_f2(lds32(sz0p + 4 * g), s0, z0);
      h2_to_f2(lds32(sz1p + 4 * g), s1, z1);
      s0 *= sc;
      s1 *= sc;
      z0 = fmaf(z0, sl2, -s0);
      z1 = fmaf(z1, sl2, -s1);
      S[0] = fmaf(s0, C[P][0], fmaf(z0, qsP[P][0], S[0]));
      S[1] = fmaf(s0, C[P][1], fmaf(z0, qsP[P][1], S[1]));
      S[2] = fmaf(s1, C[P][2], fmaf(z1, qsP[P][0], S[2]));
      S[3] = fmaf(s1, C[P][3], fmaf(z1, qsP[P][1], S[3]));
    }
  }
}

// PV for one 16-row half: O^T += V^T P^T with the half's P^T fragments.
template <int VB, int G>
__device__ __forceinline__ void pv_half(const uint8_t* vc, const uint8_t* vsz, int r0, int n,
                                        uint32_t pb0, uint32_t pb1, int gid, int tig, Acc& acc) {
  constexpr int VROW = VB * kD / 8;
  constexpr int SZROW = 4 * (kD / G);
  const int t[4] = {r0 + 2 * tig, r0 + 2 * tig + 1, r0 + 2 * tig + 8, r0 + 2 * tig + 9};
  VData<VB> v;
  v_load<VB>(vc, VROW, gid, t, v);
  uint32_t s2a = 0, z2a = 0, s2c = 0, z2c = 0;
  if constexpr (VB < 16) {
    const uint8_t* vg = vsz + 4 * ((16 * gid) / G) + r0 * SZROW + 2 * tig * SZROW;
    const uint32_t sa = lds32(vg), sb = lds32(vg + SZROW);
    const uint32_t sc = lds32(vg + 8 * SZROW), sd = lds32(vg + 9 * SZROW);
    s2a = prmt(sa, sb, 0x5410u);
    z2a = prmt(sa, sb, 0x7632u);
    s2c = prmt(sc, sd, 0x5410u);
    z2c = prmt(sc, sd, 0x7632u);
  }
  // Rows past n hold stale shared memory (possibly NaN/Inf patterns): zero
  // their V operands so that 0 * garbage cannot reach the accumulators.
  const bool ragged = r0 + 16 > n;
  uint32_t ma = 0xffffffffu, mc = 0xffffffffu;
  if (ragged) {
    ma = (t[0] < n ? 0x0000ffffu : 0u) | (t[1] < n ? 0xffff0000u : 0u);
    mc = (t[2] < n ? 0x0000ffffu : 0u) | (t[3] < n ? 0xffff0000u : 0u);
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    uint32_t A[4] = {v_pair<VB>(v, 0, 1, mt), v_pair<VB>(v, 0, 1, 8 + mt), v_pair<VB>(v, 2, 3, mt),
                     v_pair<VB>(v, 2, 3, 8 + mt)};
    if constexpr (VB < 16) {
      A[0] = hfma2_u(A[0], s2a, z2a);
      A[1] = hfma2_u(A[1], s2a, z2a);
      A[2] = hfma2_u(A[2], s2c, z2c);
      A[3] = hfma2_u(A[3], s2c, z2c);
    }
    if (ragged) {
      A[0] &= ma;
      A[1] &= ma;
      A[2] &= mc;
      A[3] &= mc;
    }
    mma_f16(acc.o[mt], A, pb0, pb1);
  }
}

// One 32-position block [r0, r0 + 32) of a staged tile (n valid positions):
// two 16-row MMA halves sharing one online-softmax update.
template <int KB, int VB, int G>
__device__ __forceinline__ void kblock32(const uint8_t* kc, const uint8_t* ksz, const uint8_t* vc,
                                         const uint8_t* vsz, int r0, int n, float sl2,
                                         const uint32_t (&qb)[8][2], const float (&qsP)[4][2],
                                         int gid, int tig, Acc& acc) {
  const bool two = r0 + 16 < n;  // the second half holds valid positions
  float S[2][4];
  qk_half<KB, G>(kc, ksz, r0, sl2, qb, qsP, gid, tig, S[0]);
  if (two) {
    qk_half<KB, G>(kc, ksz, r0 + 16, sl2, qb, qsP, gid, tig, S[1]);
  } else {
    S[1][0] = S[1][1] = S[1][2] = S[1][3] = -INFINITY;
  }
  if (r0 + 32 > n) {  // ragged block: mask rows past n
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (r0 + 16 * h + gid >= n) S[h][0] = S[h][1] = -INFINITY;
      if (r0 + 16 * h + gid + 8 >= n) S[h][2] = S[h][3] = -INFINITY;
    }
  }

  // ---- online softmax over the 32 positions (columns = heads 2tig, 2tig+1) ----
  float mx0 = fmaxf(fmaxf(S[0][0], S[0][2]), fmaxf(S[1][0], S[1][2]));
  float mx1 = fmaxf(fmaxf(S[0][1], S[0][3]), fmaxf(S[1][1], S[1][3]));
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
  }
  const float mn0 = fmaxf(acc.m[0], mx0), mn1 = fmaxf(acc.m[1], mx1);
  const float b0s = mn0 == -INFINITY ? 0.f : mn0, b1s = mn1 == -INFINITY ? 0.f : mn1;
  const float c0 = ex2(acc.m[0] - b0s), c1 = ex2(acc.m[1] - b1s);
  float P[2][4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    P[h][0] = ex2(S[h][0] - b0s);
    P[h][1] = ex2(S[h][1] - b1s);
    P[h][2] = ex2(S[h][2] - b0s);
    P[h][3] = ex2(S[h][3] - b1s);
  }
  acc.m[0] = mn0;
  acc.m[1] = mn1;
  acc.l[0] = fmaf(acc.l[0], c0, (P[0][0] + P[0][2]) + (P[1][0] + P[1][2]));
  acc.l[1] = fmaf(acc.l[1], c1, (P[0][1] + P[0][3]) + (P[1][1] + P[1][3]));
  if (!__all_sync(0xffffffffu, c0 == 1.f && c1 == 1.f)) {  // some running max moved
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      acc.o[mt][0] *= c0;
      acc.o[mt][1] *= c1;
      acc.o[mt][2] *= c0;
      acc.o[mt][3] *= c1;
    }
  }
  // P^T as the B operand of PV: transpose the 8x8 quarters.
  const uint32_t pa0 = movmatrix_trans(pack_f16x2(P[0][0], P[0][1]));
  const uint32_t pa1 = movmatrix_trans(pack_f16x2(P[0][2], P[0][3]));
  pv_half<VB, G>(vc, vsz, r0, n, pa0, pa1, gid, tig, acc);
  if (two) {
    const uint32_t pc0 = movmatrix_trans(pack_f16x2(P[1][0], P[1][1]));
    const uint32_t pc1 = movmatrix_trans(pack_f16x2(P[1][2], P[1][3]));
    pv_half<VB, G>(vc, vsz, r0 + 16, n, pc0, pc1, gid, tig, acc);
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
    float inv = 1.0f / Lt;
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
__device__ __forceinline__ bool wait_unit_released(const uint32_t* cnt) {
  for (uint32_t i = 0; i < kSpinPolls; ++i) {
    if (ld_acquire_gpu(cnt) == 0u) return true;
    __nanosleep(32);
  }
  return false;
}

template <int KB, int VB, int G, bool kStep>
__device__ __forceinline__ void consumer_loop(const Params& p, SplitSmem& sm, int c, int warp, int lane) {
  const int gid = lane >> 2, tig = lane & 3;
  const int ctid = warp * 32 + lane;  // 0 .. 32*kConsumerWarps-1
  const Cut a = p.cuts[c];
  const Cut e = p.cuts[c + 1];
  const int u_last = chunk_last_unit(p.cuts, c, p.plan.U);
  constexpr int ppg = G / 32;
  const float sl2 = p.scale_log2;
  uint32_t it = 0;    // tiles seen (stage ring position)
  uint32_t gblk = 0;  // 32-position blocks dealt so far (round-robin over warps)
  for (int u = a.u; u <= u_last; ++u) {
    const int ps = (u == a.u) ? a.p : 0;
    const int pe = (u == e.u) ? e.p : p.plan.T;
    const UnitInfo ui = unit_info(p, u);
    const int hq0 = ui.h * p.g + ui.hc * kNH;
    const int nh = min(kNH, p.g - ui.hc * kNH);
    if (u == a.u) pdl_wait();  // q (and the cache) may come from the previous kernel

    // q of head column gid as the B operand, in the permuted d order; group sums.
    uint32_t qb[8][2];
    float qpart[4];
#pragma unroll
    for (int P = 0; P < 4; ++P) {
      uint4 raw = make_uint4(0u, 0u, 0u, 0u);
      if (gid < nh)
        raw = __ldg(reinterpret_cast<const uint4*>(
            p.q + (static_cast<int64_t>(ui.b) * p.Hq + hq0 + gid) * kD + 32 * P + 8 * tig));
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
    float qsP[4][2];  // sum of q over the quantisation group of k-step pair P
#pragma unroll
    for (int P = 0; P < 4; ++P) {
      const int g0 = (P / ppg) * ppg;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float s = 0.f;
        for (int i = 0; i < ppg; ++i) s += sm.qsum[warp][2 * tig + cc][g0 + i];
        qsP[P][cc] = s;
      }
    }

    Acc acc;
    acc.m[0] = acc.m[1] = -INFINITY;
    acc.l[0] = acc.l[1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) acc.o[mt][0] = acc.o[mt][1] = acc.o[mt][2] = acc.o[mt][3] = 0.f;

    walk_piece(p, ui.prot, ps, pe, [&](int kind, int t0, int n) {
      const int st = it % kStages;
      const uint32_t round = it / kStages;
      if (!mbar_wait(&sm.full[st], round & 1, kWaitPolls)) sm.abort = 1;
      const uint8_t* base = sm.stage[st];
      if (kStep && kind == kTileText && t0 + n == p.plan.T && ui.hc == 0 && warp == 0) {
        // Write the step's row (staged from the input) into the cache's text
        // segment: lanes 0-15 the K row, lanes 16-31 the V row.
        const int tr = p.t_new < p.vs ? p.t_new : p.t_new - p.Tv;
        const int64_t row = (static_cast<int64_t>(ui.b) * p.Hkv + ui.h) * p.T_text + tr;
        const int half = lane >> 4, q = lane & 15;
        const uint4 w = *reinterpret_cast<const uint4*>(base + (half ? kBf16VOff : 0) +
                                                       (n - 1) * (2 * kD) + 16 * q);
        uint8_t* dst = const_cast<uint8_t*>(p.seg[half ? KVQ_SEG_TEXT_V : KVQ_SEG_TEXT_K]) +
                       row * (2 * kD) + 16 * q;
        *reinterpret_cast<uint4*>(dst) = w;
      }
      const int nb = (n + 31) >> 5;
      const int first = (warp + kConsumerWarps - static_cast<int>(gblk % kConsumerWarps)) % kConsumerWarps;
      gblk += nb;
      for (int kb = first; kb < nb; kb += kConsumerWarps) {
        if (kind == kTilePacked)
          kblock32<KB, VB, G>(base, base + p.pk_off_ksz, base + p.pk_off_vc, base + p.pk_off_vsz,
                              kb * 32, n, sl2, qb, qsP, gid, tig, acc);
        else
          kblock32<16, 16, G>(base, nullptr, base + kBf16VOff, nullptr, kb * 32, n, sl2, qb, qsP, gid,
                              tig, acc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[st]);
      ++it;
    });

    // ---- merge the 4 warps' states and write the partial of (u, c) ----
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
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int d0 = 16 * gid + mt, d1 = d0 + 8;
      sm.merge_o[warp][2 * tig][d0] = acc.o[mt][0];
      sm.merge_o[warp][2 * tig + 1][d0] = acc.o[mt][1];
      sm.merge_o[warp][2 * tig][d1] = acc.o[mt][2];
      sm.merge_o[warp][2 * tig + 1][d1] = acc.o[mt][3];
    }
    // The fused step finishes a unit held by this CTA alone right here;
    // otherwise the partial goes to slot u + c.
    int cf = c, cl = c;
    if constexpr (kStep) plan_unit_chunks(p.plan, p.cuts, u, &cf, &cl);
    const bool sole = kStep && cf == cl;
    const int64_t row0 = static_cast<int64_t>(ui.b) * p.Hq + hq0;
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
        const float inv = (M != M) ? M : 1.0f / L;
        p.out[(row0 + j) * kD + d] = f32_to_bf16_bits(O * inv);
        if (d == 0 && p.lse) p.lse[row0 + j] = (M != M) ? M : 0.69314718055994531f * (M + log2f(L));
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
        // others, who wait for that.
        if (ctid == 0) {
          __threadfence();
          const uint32_t n = static_cast<uint32_t>(cl - cf + 1);
          const uint32_t nc = min(n, static_cast<uint32_t>(nh));
          const uint32_t k = atomicAdd(&p.cnt[u], 1u);
          int role = -1;
          if (k == n - 1) {
            __threadfence();
            atomicExch(&p.cnt[u], 0u);
            role = static_cast<int>(nc) - 1;
          } else if (k >= n - nc) {
            role = static_cast<int>(k - (n - nc));
            if (!wait_unit_released(&p.cnt[u])) sm.abort = 1;
          }
          __threadfence();
          sm.role = role;
          sm.ncomb = static_cast<int>(nc);
        }
        named_bar(1, kConsumerWarps * 32);
        const int role = sm.role, nc = sm.ncomb;
        if (role >= 0) {
          const bool bad = sm.abort != 0;
          float (*sm_ml)[2] = reinterpret_cast<float (*)[2]>(&sm.merge_ml[0][0][0]);
          float4 (*sm_o)[32] = reinterpret_cast<float4 (*)[32]>(&sm.merge_o[0][0][0]);
          for (int j = role; j < nh; j += nc)
            combine_row<kConsumerWarps>(p, u, j, cf, cl, row0 + j, warp, lane, sm_ml, sm_o, bad,
                                        []() { named_bar(1, kConsumerWarps * 32); });
        }
      }
    }
  }
}

template <int KB, int VB, int G, bool kStep>
__global__ void __maxnreg__(168) split_mma_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SplitSmem& sm = *reinterpret_cast<SplitSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsumerWarps);
    }
    sm.abort = 0;
    fence_barrier_init();
  }
  pdl_launch_dependents();
  __syncthreads();
  if (warp == kConsumerWarps) {
    if (lane == 0) {
      producer_prefetch(p, blockIdx.x);
      pdl_wait();  // the previous kernel in the stream may have written the cache
      producer_loop<kStep>(p, sm, blockIdx.x);
    }
    return;
  }
  consumer_loop<KB, VB, G, kStep>(p, sm, blockIdx.x, warp, lane);
}

}  // namespace kvq
