// kvq_mq_umma.cuh -- multi-query decode on the fifth-generation tensor cores
// (tcgen05, accumulators in tensor memory).
//
// Same computation as the multi-query form of the split-KV kernel (WSVD
// summary, section 2.라: K/V rebuilt on chip, QK, softmax and PV fused, no
// reconstructed tensor written to device memory; "VLM_KV_Quantization",
// section 2: GQA cache read by its query heads), for calls whose KV heads
// have more than eight (query head, token) columns.  A unit is one
// (sequence b, KV head h, chunk of up to 128 columns); every column of the
// unit is a row of the MMAs (M = 128), so the unit's cache is read once for
// all of them.  Per 32-position sub-tile:
//   S[c][t]  = q_c . k_t      M = 128 columns, N = 32 positions, K = d
//   O[c][d] += P[c][t] v_t    M = 128 columns, N = 128 d, K = 32 positions
// Operands: q (and the per-group q sums) sit in shared memory as the A
// operand of QK; K sub-tiles are written to shared memory as fp16 tiles --
// packed codes moved to bit 0 of their half-word, i.e. the exact subnormals
// c * 2^-24, in the split kernel's permuted d order, one accumulator per
// quantisation group g, plus one for the zero-point term (A = q group sums
// as an fp16 hi + lo pair, B = z) -- or bf16 rows converted to fp16
// (exact); the softmax applies s_g * 2^24 per (position, group).  V sub-tiles are dequantised to fp16
// (code * s + z, one rounding) or converted from bf16, so O accumulates true
// values for every tile kind.  P is written to TMEM (fp16) as the A operand
// of PV.  S has two TMEM buffers, so the QK of the next sub-tile runs while
// the softmax reads this one.  The online softmax keeps a running maximum per column (one TMEM
// lane = one thread) and rescales O only when a column's maximum grows by
// more than 2^8 (P stays <= 256 in fp16).
//
// CTA = 12 warps: warps 0-3 softmax (TMEM lanes 32w .. 32w + 31 = columns),
// warps 4-9 build the operand tiles, warp 10 stages cache tiles by bulk
// copies (TMA) into a 3-stage ring, warp 11 allocates TMEM and one of its
// threads issues the MMAs.  A cluster of cs CTAs takes a unit at a time (unit
// u goes to cluster u mod clusters), splits its positions at equal cost and
// merges the cs partial rows through distributed shared memory; cs = 1 CTAs
// take whole units.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "kvq_device.cuh"
#include "kvq_ptx.cuh"
#include "kvq_split.cuh"
#include "kvq_umma.cuh"

namespace kvq {
namespace mq {

constexpr int kCols = 128;         // columns per unit (MMA M)
constexpr int kSub = 32;           // positions per sub-tile (QK N, PV K)
constexpr int kRing = 3;           // staged-tile ring (3 stages)
constexpr int kOps = 3;            // operand-tile buffers (sub-tiles built ahead of the MMAs)
constexpr int kThreads = 384;
constexpr int kDequantWarps = 6;
constexpr int kProducerWarp = 10;
constexpr int kMmaWarp = 11;
constexpr float kRescaleLog2 = 8.f;  // lazy rescale threshold (log2 units)
// Cluster merge rows in the ring: a column's 128 floats at a pitch of 132
// (consecutive columns start 16 bytes apart in the bank cycle, so a warp's
// 16-byte stores spread over every bank slot).
constexpr int kMergePitch = kD + 4;
static_assert(kCols * kMergePitch * 4 <= kRing * kStageBytes, "merge rows must fit the ring");

// TMEM columns: two S buffers (QK of the next sub-tile runs while the
// softmax reads this one), O, two P buffers.
constexpr uint32_t kTmS = 0;      // S buffer b at kTmS + b * kTmSStride: acc_g, g < D / G <= 4, 32 columns
                                  // each (bf16 tiles use acc_0), then the zero-point term, 32
constexpr uint32_t kTmSStride = 160;
constexpr uint32_t kTmZ = 128;    // zero-point term, inside an S buffer
constexpr uint32_t kTmO = 320;    // O, 128
constexpr uint32_t kTmP = 448;    // P buffers, 2 x 16
constexpr uint32_t kTmCols = 512;

enum SubKind { kSubPackedK = 0, kSubBf16K = 1 };

struct Smem {
  alignas(1024) uint8_t stage[kRing][kStageBytes];  // staged tiles; merge area at unit end
  alignas(1024) uint8_t kt[kOps][kSub * 256];        // K operand: 32 pos x 128 fp16, K-major
  alignas(1024) uint8_t vt[kOps][kSub * 256];        // V operand: 32 pos x 128 fp16, MN-major
  alignas(128) uint8_t zt[kOps][kSub * 32];          // Z operand: 32 pos x 16 fp16, K-major
  alignas(16) float fac[kOps][4][kSub];              // s_g * 2^24 * scale_log2 per (group g, position)
  alignas(1024) uint8_t qt[kCols * kD * 2];         // q: 128 columns x 128 fp16, K-major (A of QK)
  alignas(128) uint8_t qst[kCols * 16 * 2];         // q group sums (hi, lo): 128 x 16 fp16, K-major
  alignas(16) float ml[kCols][2];                    // cluster merge: the CTA's (m, l) per column
  float wm[kCols], wl[kCols];                        // cluster merge: (m, l), then weights, per (column, rank)
  float mML[kCols][2];                               // cluster merge: (M, L) per combined column
  uint64_t full[kRing], empty[kRing];
  uint64_t op_full[kOps], pv_done[kOps], p_full[2];
  uint64_t s_full[2], s_free[2], q_ready;
  uint32_t tmem_base;
  int abort;
};

// Units: (b, h, hc) with hc over ceil(g n_q / 128) column chunks.
struct MqUnit {
  int b, h, hc, cls, ncols;
};
__device__ __forceinline__ MqUnit mq_unit(const Params& p, int u) {
  MqUnit r;
  const int nhc = p.NHC;  // column chunks per KV head (of kCols)
  r.hc = u % nhc;
  const int bh = u / nhc;
  r.b = bh / p.Hkv;
  r.h = bh - r.b * p.Hkv;
  r.cls = p.prot[r.h] == 1 ? kClsProt : (p.prot[r.h] == 2 ? kClsKonly : kClsPacked);
  r.ncols = min(kCols, p.g * p.n_q - r.hc * kCols);
  return r;
}

// Positions [ps, pe) of unit un for cluster rank r of cs: equal-cost cuts.
__device__ __forceinline__ void mq_piece(const Params& p, const MqUnit& un, int r, int cs, int* ps, int* pe) {
  const int64_t uc = un.cls == kClsProt ? p.plan.ub_p : (un.cls == kClsKonly ? p.plan.ub_k : p.plan.ub_u);
  *ps = r == 0 ? 0 : unit_cut_pos(p.plan, un.cls, uc * r / cs);
  *pe = r + 1 == cs ? p.plan.T : unit_cut_pos(p.plan, un.cls, uc * (r + 1) / cs);
  if (*pe < *ps) *pe = *ps;
}

__device__ __forceinline__ void fail(const Params& p, Smem& sm) {
  sm.abort = 1;
  if (p.status) atomicOr(p.status, KVQ_STATUS_TILE_WAIT);
}
__device__ __forceinline__ void wait_bar(const Params& p, Smem& sm, uint64_t* bar, uint32_t parity) {
  if (!mbar_wait(bar, parity, p.tile_polls)) fail(p, sm);
}

// Walk this CTA's pieces unit by unit: start(u, unit, ps, pe) before a
// unit's tiles, tile(u, unit, kind, t0, n) per staged tile, end(u, unit, ps,
// pe) after them.  Unit u goes to cluster u mod clusters; cluster rank r
// takes the r-th of cs equal-cost pieces of it.
template <typename S, typename F, typename E>
__device__ __forceinline__ void mq_walk(const Params& p, S&& start, F&& tile, E&& end) {
  const int cs = p.plan.cs;
  const int clu = blockIdx.x / cs, ncl = gridDim.x / cs, rank = blockIdx.x - clu * cs;
  for (int u = clu; u < p.plan.U; u += ncl) {
    const MqUnit un = mq_unit(p, u);
    int ps, pe;
    mq_piece(p, un, rank, cs, &ps, &pe);
    start(u, un, ps, pe);
    walk_piece<true>(p, un.cls, ps, pe, [&](int kind, int t0, int n) { tile(u, un, kind, t0, n); });
    end(u, un, ps, pe);
  }
}

// The unit's staged-tile sources, as UnitInfo for tile_sources.
__device__ __forceinline__ UnitInfo mq_info(const Params& p, const MqUnit& un) {
  UnitInfo ui;
  ui.b = un.b;
  ui.h = un.h;
  ui.hc = un.hc;
  ui.slot = p.slot[un.h];
  ui.cls = un.cls;
  ui.prot = un.cls == kClsProt;
  return ui;
}

// ---------------------------------------------------------------------------
// Operand builders (dequant warps).  Sub-tile rows pos in [0, 32).
// K operand (K-major, 8 x 16 B core matrices): element kappa of row pos at
// (kappa / 8) * 512 + (pos / 8) * 128 + (pos % 8) * 16 + (kappa % 8) * 2, in
// the split kernel's permuted order kappa = 32P + 8t + 2i + e for
// d = 32P + 8t + 4e + i, so the four registers of block P of lane slice t
// are one 16-byte chunk.
__device__ __forceinline__ uint32_t kt_off(int chunk, int pos) {
  return static_cast<uint32_t>(chunk * 512 + (pos >> 3) * 128 + (pos & 7) * 16);
}
// V operand (MN-major): d of row pos at (pos / 8) * 2048 + (d / 8) * 128 + (pos % 8) * 16 + (d % 8) * 2.
__device__ __forceinline__ uint32_t vt_off(int dchunk, int pos) {
  return static_cast<uint32_t>((pos >> 3) * 2048 + dchunk * 128 + (pos & 7) * 16);
}

// Copy task -> (row pos, 16-byte chunk ch) of a 32-row x 16-chunk bf16 block:
// blocks of 8 rows x 8 chunks, a row's chunk rotated by the row, so that the
// 32 lanes of a warp hit every 16-byte bank slot four times both when they
// read the staged rows (256-byte pitch: slot = ch mod 8) and when they write
// the core-matrix tiles (slot = pos mod 8): no bank conflicts either way.
__device__ __forceinline__ void diag_task(int task, int* pos, int* ch) {
  const int blk = task >> 6, idx = task & 63;
  const int r = idx & 7, c = idx >> 3;
  *pos = 8 * (blk & 3) + r;
  *ch = 8 * (blk >> 2) + ((c + r) & 7);
}

__device__ __forceinline__ void sts128(uint8_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}

// fp16 pair (lo, hi) = (c_lo * s + z, c_hi * s + z) from codes at bits
// [0, b) of each half of x (one rounding each).
__device__ __forceinline__ uint32_t dq_pair(uint32_t x, uint32_t mask, uint32_t s2, uint32_t z2) {
  const uint32_t m = and_or(x, mask, 0x64006400u);  // 1024 + c, exact
  return hfma2_u(hsub2_u(m, 0x64006400u), s2, z2);
}

template <int KB, int VB, int G>
__device__ __forceinline__ void build_sub(const Params& p, Smem& sm, int kind, const uint8_t* base, int r0, int n,
                                          int buf, int tid) {
  constexpr int NG = kD / G;
  constexpr int NT = kDequantWarps * 32;
  uint8_t* kt = sm.kt[buf];
  uint8_t* vt = sm.vt[buf];
  const bool k_codes = KB < 16 && kind == kTilePacked;
  const bool v_codes = VB < 16 && (kind == kTilePacked || kind == kTileKonly);
  // staged sub-buffers: K rows at the stage start (codes, or bf16 rows)
  const uint8_t* kc = base;
  const uint8_t* vc = kind == kTilePacked ? base + p.pk_off_vc : (kind == kTileKonly ? base + p.ko_off_vc : base + kBf16VOff);
  // ---- K ----
  if (k_codes) {
    if constexpr (KB < 16) {
      constexpr int KROW = KB * kD / 8;
      const uint8_t* ksz = base + p.pk_off_ksz;
      for (int task = tid; task < kSub * 4; task += NT) {
        const int pos = task >> 2, t = task & 3;
        uint32_t f[4][4];
        if (pos < n) {
          k_packed_regs<KB>(kc + (r0 + pos) * KROW, t, f);
          // every code to bit 0 of its half-word (c * 2^-24), so that the
          // blocks of one quantisation group share one accumulator
#pragma unroll
          for (int P = 0; P < 4; ++P)
#pragma unroll
            for (int i = 0; i < 4; ++i) f[P][i] >>= kKShift<KB>(P);
        } else {
#pragma unroll
          for (int P = 0; P < 4; ++P) f[P][0] = f[P][1] = f[P][2] = f[P][3] = 0u;
        }
#pragma unroll
        for (int P = 0; P < 4; ++P) sts128(kt + kt_off(4 * P + t, pos), f[P][0], f[P][1], f[P][2], f[P][3]);
      }
      // Z operand (z_g at K index g and NG + g) and the per-(P, position) factors
      for (int pos = tid; pos < kSub; pos += NT) {
        uint32_t zw[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        float s[NG];
        if (pos < n) {
          const uint16_t* row = reinterpret_cast<const uint16_t*>(ksz + (r0 + pos) * (4 * NG));
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            const uint32_t z = row[g];
            zw[g >> 1] |= z << (16 * (g & 1));
            zw[(NG + g) >> 1] |= z << (16 * ((NG + g) & 1));
            s[g] = __half2float(__ushort_as_half(row[NG + g]));
          }
        } else {
#pragma unroll
          for (int g = 0; g < NG; ++g) s[g] = 0.f;
        }
        uint8_t* zt = sm.zt[buf];
        sts128(zt + (pos >> 3) * 128 + (pos & 7) * 16, zw[0], zw[1], zw[2], zw[3]);
        sts128(zt + 512 + (pos >> 3) * 128 + (pos & 7) * 16, zw[4], zw[5], zw[6], zw[7]);
#pragma unroll
        for (int g = 0; g < NG; ++g) sm.fac[buf][g][pos] = s[g] * 16777216.f * p.scale_log2;
      }
    }
  } else {  // bf16 K rows (text, protected, K-only, or 16-bit "packed" K): 16 chunks of 8 d per row
    for (int task = tid; task < kSub * 16; task += NT) {
      int pos, ch;
      diag_task(task, &pos, &ch);
      const int P = ch >> 2, t = ch & 3;
      uint32_t f[4] = {0u, 0u, 0u, 0u};
      if (pos < n) k_bf16_pairs(kc + (r0 + pos) * (2 * kD), P, t, f);
      sts128(kt + kt_off(4 * P + t, pos), f[0], f[1], f[2], f[3]);
    }
  }
  // ---- V ----
  if (v_codes) {
    if constexpr (VB < 16) {
      constexpr int VROW = VB * kD / 8;
      constexpr int CPW = 32 / VB;  // codes per word
      constexpr uint32_t MASK = VB == 2 ? 0x00030003u : (VB == 4 ? 0x000F000Fu : 0x00FF00FFu);
      const uint8_t* vsz = kind == kTilePacked ? base + p.pk_off_vsz : base + p.ko_off_vsz;
      for (int task = tid; task < kSub * 4; task += NT) {
        const int pos = task >> 2, qq = task & 3;  // chunks k = 4 qq .. 4 qq + 3 (d = 8k .. 8k + 7)
        if (pos >= n) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) sts128(vt + vt_off(4 * qq + kk, pos), 0u, 0u, 0u, 0u);
          continue;
        }
        const uint8_t* row = vc + (r0 + pos) * VROW;
        const uint16_t* szr = reinterpret_cast<const uint16_t*>(vsz + (r0 + pos) * (4 * NG));
        // element d = 16m + 8r + n sits in slot 16n + k (k = 2m + r = d / 8):
        // word (16n + k) / CPW = 16n / CPW + k / CPW, the last constant in a quarter
        const int kw = (4 * qq) / CPW;
        uint32_t w[8];
#pragma unroll
        for (int nn = 0; nn < 8; ++nn) w[nn] = lds32(row + 4 * ((16 * nn) / CPW + kw));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int k = 4 * qq + kk;
          const int bit = VB * (k % CPW);
          const uint32_t sel = bit >= 16 ? 0x7632u : 0x5410u;
          const int sh = bit & 15;
          const int g = (8 * k) / G;
          const uint32_t s2 = static_cast<uint32_t>(szr[NG + g]) * 0x10001u;
          const uint32_t z2 = static_cast<uint32_t>(szr[g]) * 0x10001u;
          uint32_t o[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) o[j] = dq_pair(prmt(w[2 * j], w[2 * j + 1], sel) >> sh, MASK, s2, z2);
          sts128(vt + vt_off(k, pos), o[0], o[1], o[2], o[3]);
        }
      }
    }
  } else {  // bf16 V rows
    for (int task = tid; task < kSub * 16; task += NT) {
      int pos, k;
      diag_task(task, &pos, &k);
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (pos < n) {
        const uint4 r = lds128(vc + (r0 + pos) * (2 * kD) + 16 * k);
        x = make_uint4(bf16x2_f16x2(r.x), bf16x2_f16x2(r.y), bf16x2_f16x2(r.z), bf16x2_f16x2(r.w));
      }
      sts128(vt + vt_off(k, pos), x.x, x.y, x.z, x.w);
    }
  }
}

// ---------------------------------------------------------------------------
// Cluster merge of a unit (every thread of the CTA; cs > 1): each CTA's
// softmax threads left their column's O row in the ring area and (m, l) in
// sm.ml; CTA rank r combines the unit's columns r, r + cs, ... from all
// ranks through distributed shared memory and writes the output rows.
__device__ __forceinline__ void cluster_merge(const Params& p, Smem& sm, const MqUnit& un) {
  const int cs = p.plan.cs;
  const int rank = static_cast<int>(cluster_ctarank());
  const int nloc = rank < un.ncols ? (un.ncols - rank + cs - 1) / cs : 0;
  const float* mo = reinterpret_cast<const float*>(sm.stage[0]);  // rows of kMergePitch floats
  cluster_sync();  // every CTA's partial rows are in its shared memory
  for (int i = threadIdx.x; i < nloc * cs; i += kThreads) {
    const int jj = i / cs, rr = i - jj * cs;
    const float2 v = ld_dsmem2(dsmem_addr(&sm.ml[rank + jj * cs][0], rr));
    sm.wm[i] = v.x;
    sm.wl[i] = v.y;
  }
  named_bar(3, kThreads);
  for (int jj = threadIdx.x; jj < nloc; jj += kThreads) {
    float M = -INFINITY;
    bool bad = false;
    for (int rr = 0; rr < cs; ++rr) {
      const float m = sm.wm[jj * cs + rr];
      if (m != m) bad = true; else M = fmaxf(M, m);
    }
    float L = 0.f;
    for (int rr = 0; rr < cs; ++rr) {
      const float m = sm.wm[jj * cs + rr];
      const float w = (m == -INFINITY || m != m || M == -INFINITY) ? 0.f : exp2f(m - M);
      sm.wm[jj * cs + rr] = w;
      L = fmaf(sm.wl[jj * cs + rr], w, L);
    }
    sm.mML[jj][0] = bad ? __int_as_float(0x7fffffff) : M;
    sm.mML[jj][1] = L;
  }
  named_bar(3, kThreads);
  for (int i = threadIdx.x; i < nloc * kD; i += kThreads) {
    const int jj = i / kD, d = i - jj * kD;
    const int c = rank + jj * cs;
    float x[kMaxClusterCtas];
#pragma unroll
    for (int rr = 0; rr < kMaxClusterCtas; ++rr) x[rr] = rr < cs ? ld_dsmem(dsmem_addr(&mo[c * kMergePitch + d], rr)) : 0.f;
    float O = 0.f;
#pragma unroll
    for (int rr = 0; rr < kMaxClusterCtas; ++rr)
      if (rr < cs) O = fmaf(x[rr], sm.wm[jj * cs + rr], O);
    const float M = sm.mML[jj][0], L = sm.mML[jj][1];
    const float inv = (M != M) ? M : (L > 0.f ? 1.0f / L : 0.f);
    const int64_t row = col_row(p, un.b, un.h, un.hc * kCols + c);
    p.out[row * kD + d] = f32_to_bf16_bits(O * inv);
    if (d == 0 && p.lse) p.lse[row] = (M != M) ? M : 0.69314718055994531f * (M + log2f(L));
  }
  cluster_sync();  // the other CTAs' reads of this CTA's rows are done
}

template <int KB, int VB, int G>
__global__ void __launch_bounds__(kThreads, 1) mq_umma_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kDequantWarps);
    }
    for (int b = 0; b < kOps; ++b) {
      mbar_init(&sm.op_full[b], kDequantWarps);
      mbar_init(&sm.pv_done[b], 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(&sm.p_full[b], 4);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.s_free[b], 4);
    }
    mbar_init(&sm.q_ready, 4);
    sm.abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&sm.tmem_base, kTmCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = sm.tmem_base;
  const bool cluster = p.plan.cs > 1;
  auto nothing = [](int, const MqUnit&, int, int) {};
  auto merge_if_cluster = [&](int, const MqUnit& un, int, int) {
    if (cluster) cluster_merge(p, sm, un);
  };

  if (warp == kProducerWarp) {
    // ---------------- staged tiles (bulk copies into the ring) ----------------
    // L2 prefetch (L2 is coherent with the previous kernel's stores): the
    // tiles of the first ring fill before the dependency wait, the rest of
    // the pieces once those tiles' copies are queued behind the wait.
    auto prefetch_tiles = [&](uint32_t from, uint32_t to) {
      uint32_t k = 0;
      mq_walk(p, nothing, [&](int, const MqUnit& un, int kind, int t0, int n) {
        if (k >= from && k < to)
          tile_sources<false, true>(p, mq_info(p, un), p.plan.T, kind, t0, n,
                                    [&](uint32_t, const uint8_t* src, uint32_t bytes) { prefetch_l2(src, bytes); });
        ++k;
      }, nothing);
    };
    if (lane == 0) prefetch_tiles(0, kRing);
    __syncwarp();
    pdl_wait();
    uint32_t it = 0;
    mq_walk(p, nothing, [&](int, const MqUnit& un, int kind, int t0, int n) {
      if (lane == 0 && it == kRing) prefetch_tiles(kRing, 0xffffffffu);
      if (lane == 0) {
        const int st = it % kRing;
        const uint32_t round = it / kRing;
        if (round > 0) wait_bar(p, sm, &sm.empty[st], (round - 1) & 1);
        const UnitInfo ui = mq_info(p, un);
        uint32_t total = 0;
        tile_sources<false, true>(p, ui, p.plan.T, kind, t0, n, [&](uint32_t, const uint8_t*, uint32_t b) { total += b; });
        mbar_arrive_expect_tx(&sm.full[st], total);
        tile_sources<false, true>(p, ui, p.plan.T, kind, t0, n, [&](uint32_t off, const uint8_t* src, uint32_t b) {
          bulk_g2s(sm.stage[st] + off, src, b, &sm.full[st]);
        });
      }
      ++it;
    }, [&](int u, const MqUnit& un, int ps, int pe) {
      __syncwarp();
      merge_if_cluster(u, un, ps, pe);
    });
  } else if (warp >= 4 && warp < 4 + kDequantWarps) {
    // ---------------- operand tiles ----------------
    const int tid = threadIdx.x - 128;
    pdl_wait();
    uint32_t it = 0, q = 0;
    mq_walk(p, nothing, [&](int, const MqUnit&, int kind, int, int n) {
      const int st = it % kRing;
      wait_bar(p, sm, &sm.full[st], (it / kRing) & 1);
      for (int r0 = 0; r0 < n; r0 += kSub) {
        const int buf = q % kOps;
        if (q >= kOps) wait_bar(p, sm, &sm.pv_done[buf], (q / kOps - 1) & 1);
        build_sub<KB, VB, G>(p, sm, kind, sm.stage[st], r0, min(kSub, n - r0), buf, tid);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.op_full[buf]);
        ++q;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[st]);
      ++it;
    }, merge_if_cluster);
  } else if (warp == kMmaWarp) {
    // ---------------- MMAs (one thread issues) ----------------
    pdl_wait();
    if (lane == 0) pdl_launch_dependents();  // past the dependency wait; this kernel writes no cache row
    const uint32_t id_qk = umma_idesc_f16(kCols, kSub, false);
    const uint32_t id_pv = umma_idesc_f16(kCols, kD, true);
    uint32_t q = 0, nu = 0;
    bool pending = false, first_pv = true;
    auto issue_pv = [&](uint32_t qq) {  // O (+)= P(qq) V(qq)
      const int pb = qq & 1, ob = qq % kOps;
      wait_bar(p, sm, &sm.p_full[pb], (qq >> 1) & 1);
      tc_fence_after();
      const uint32_t vb = smem_u32(sm.vt[ob]);
#pragma unroll
      for (int s = 0; s < 2; ++s)
        umma_ts(tm + kTmO, tm + kTmP + 16 * pb + 8 * s, umma_sdesc(vb + s * 2 * 2048, 2048, 128), id_pv,
                !first_pv || s > 0);
      umma_commit(&sm.pv_done[ob]);
      first_pv = false;
    };
    mq_walk(p, [&](int, const MqUnit&, int ps, int pe) {
      if (pe > ps && lane == 0) {
        wait_bar(p, sm, &sm.q_ready, nu & 1);
        tc_fence_after();
      }
      if (pe > ps) ++nu;
      first_pv = true;
    }, [&](int, const MqUnit&, int kind, int, int n) {
      for (int r0 = 0; r0 < n; r0 += kSub) {
        if (lane == 0) {
          const int buf = q % kOps;
          wait_bar(p, sm, &sm.op_full[buf], (q / kOps) & 1);
          if (q >= 2) wait_bar(p, sm, &sm.s_free[q & 1], ((q - 2) >> 1) & 1);
          tc_fence_after();
          const uint32_t kb = smem_u32(sm.kt[buf]);
          const uint32_t qa = smem_u32(sm.qt);  // K step ks of q: chunks 2 ks, 2 ks + 1
          const uint32_t sb = tm + kTmS + (q & 1) * kTmSStride;
          if (KB < 16 && kind == kTilePacked) {
            // one accumulator per quantisation group g: K steps 2P, 2P + 1 of
            // the 32-element blocks P of g
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const int g = (16 * ks) / G;
              umma_ss(sb + 32 * g, umma_sdesc(qa + ks * 4096, 2048, 128), umma_sdesc(kb + ks * 1024, 512, 128),
                      id_qk, (16 * ks) % G != 0);
            }
            umma_ss(sb + kTmZ, umma_sdesc(smem_u32(sm.qst), 2048, 128), umma_sdesc(smem_u32(sm.zt[buf]), 512, 128),
                    id_qk, false);
          } else {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              umma_ss(sb, umma_sdesc(qa + ks * 4096, 2048, 128), umma_sdesc(kb + ks * 1024, 512, 128), id_qk, ks > 0);
          }
          umma_commit(&sm.s_full[q & 1]);
          if (pending) issue_pv(q - 1);
        }
        pending = true;
        ++q;
      }
    }, [&](int u, const MqUnit& un, int ps, int pe) {
      if (pending && lane == 0) issue_pv(q - 1);
      pending = false;
      __syncwarp();
      merge_if_cluster(u, un, ps, pe);
    });
  } else {
    // ---------------- softmax: warps 0-3, thread = column ----------------
    const int c = threadIdx.x;  // column of the unit = TMEM lane
    const uint32_t lb = static_cast<uint32_t>(32 * warp) << 16;
    constexpr int NG = kD / G;
    const float sl2 = p.scale_log2;
    pdl_wait();
    uint32_t q = 0;
    float m_use = -INFINITY, l = 0.f;
    bool have_o = false;
    int end_c = 0;
    mq_walk(p, [&](int, const MqUnit& un, int ps, int pe) {
      m_use = -INFINITY;
      l = 0.f;
      have_o = false;
      const bool active = c < un.ncols;
      const int cg = un.hc * kCols + c;  // column among the KV head's g * n_q
      end_c = active ? p.plan.T - (p.n_q - 1 - cg % p.n_q) : 0;
      if (pe <= ps) return;
      // q of this column as row c of the QK A tile (K-major core matrices:
      // element kappa at (kappa / 8) * 2048 + (c / 8) * 128 + (c % 8) * 16 +
      // (kappa % 8) * 2), fp16 in the permuted order kappa = 32P + 8t + 2i + e
      // for d = 32P + 8t + i + 4e; its group sums as an fp16 hi + lo pair
      // (K index g and NG + g) as row c of the zero-point A tile
      uint32_t qv[32];
      float qs[NG];
#pragma unroll
      for (int g = 0; g < NG; ++g) qs[g] = 0.f;
      const uint4* qrow = reinterpret_cast<const uint4*>(p.q + (active ? col_row(p, un.b, un.h, cg) : 0) * kD);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int P2 = 0; P2 < 2; ++P2) {
          const int P = 2 * half + P2;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint4 r = make_uint4(0u, 0u, 0u, 0u);
            if (active) r = __ldcg(qrow + 4 * P + t);
            const float x[8] = {bf16_lo(r.x), bf16_hi(r.x), bf16_lo(r.y), bf16_hi(r.y),
                                bf16_lo(r.z), bf16_hi(r.z), bf16_lo(r.w), bf16_hi(r.w)};
#pragma unroll
            for (int i = 0; i < 4; ++i) qv[16 * P2 + 4 * t + i] = pack_f16x2(x[i], x[i + 4]);
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) sum += __half2float(__float2half_rn(x[i]));
            qs[(32 * P) / G] += sum;
          }
        }
#pragma unroll
        for (int P2 = 0; P2 < 2; ++P2)
#pragma unroll
          for (int t = 0; t < 4; ++t)
            sts128(sm.qt + (4 * (2 * half + P2) + t) * 2048 + (c >> 3) * 128 + (c & 7) * 16, qv[16 * P2 + 4 * t],
                   qv[16 * P2 + 4 * t + 1], qv[16 * P2 + 4 * t + 2], qv[16 * P2 + 4 * t + 3]);
      }
      uint32_t zq[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) zq[j] = 0u;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const __half hi = __float2half_rn(qs[g]);
        const __half lo = __float2half_rn(qs[g] - __half2float(hi));
        zq[g >> 1] |= static_cast<uint32_t>(__half_as_ushort(hi)) << (16 * (g & 1));
        zq[(NG + g) >> 1] |= static_cast<uint32_t>(__half_as_ushort(lo)) << (16 * ((NG + g) & 1));
      }
#pragma unroll
      for (int k = 0; k < 2; ++k)
        sts128(sm.qst + k * 2048 + (c >> 3) * 128 + (c & 7) * 16, zq[4 * k], zq[4 * k + 1], zq[4 * k + 2],
               zq[4 * k + 3]);
      fence_async_smem();  // the tensor cores read the tiles
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.q_ready);
    }, [&](int, const MqUnit&, int kind, int t0, int n) {
      for (int r0 = 0; r0 < n; r0 += kSub) {
        const int buf = q & 1, ob = q % kOps;
        const int nval = min(kSub, n - r0);
        const int t0s = t0 + r0;
        wait_bar(p, sm, &sm.s_full[q & 1], (q >> 1) & 1);
        tc_fence_after();
        const uint32_t sb = kTmS + (q & 1) * kTmSStride;
        float S[kSub];
        uint32_t a[32];
        if (KB < 16 && kind == kTilePacked) {
          // two halves of 16 positions: the accumulators' loads in flight together
          constexpr int NG = kD / G;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t az[16], ag[NG][16];
            tmem_ld16(tm + lb + sb + kTmZ + 16 * hf, az);
#pragma unroll
            for (int g = 0; g < NG; ++g) tmem_ld16(tm + lb + sb + 32 * g + 16 * hf, ag[g]);
            tmem_ld_wait();
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
              float fa[NG][4];
#pragma unroll
              for (int g = 0; g < NG; ++g) {
                const float4 f = reinterpret_cast<const float4*>(sm.fac[ob][g])[4 * hf + i4];
                fa[g][0] = f.x;
                fa[g][1] = f.y;
                fa[g][2] = f.z;
                fa[g][3] = f.w;
              }
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int i = 4 * i4 + e;
                float x = sl2 * __uint_as_float(az[i]);
#pragma unroll
                for (int g = 0; g < NG; ++g) x = fmaf(fa[g][e], __uint_as_float(ag[g][i]), x);
                S[16 * hf + i] = x;
              }
            }
          }
        } else {
          tmem_ld32(tm + lb + sb, a);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < kSub; ++i) S[i] = sl2 * __uint_as_float(a[i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.s_free[q & 1]);
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < kSub; ++i) {
          if (i >= nval || t0s + i >= end_c) S[i] = -INFINITY;
          mx = fmaxf(mx, S[i]);
        }
        const bool need = mx > m_use + kRescaleLog2 || (m_use == -INFINITY && mx > -INFINITY);
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? mx : m_use;
          const float cr = (need && m_use != -INFINITY) ? ex2(m_use - m_new) : 1.f;
          if (have_o) {  // every earlier PV must have landed before O is rescaled
            wait_bar(p, sm, &sm.pv_done[(q - 1) % kOps], ((q - 1) / kOps) & 1);
            tc_fence_after();
#pragma unroll 1
            for (int k = 0; k < 4; ++k) {
              tmem_ld32(tm + lb + kTmO + 32 * k, a);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) a[i] = __float_as_uint(__uint_as_float(a[i]) * cr);
              tmem_st32(tm + lb + kTmO + 32 * k, a);
            }
            tmem_st_wait();
          }
          l *= cr;
          m_use = m_new;
        }
        uint32_t pp[16];
        float ls = 0.f;
#pragma unroll
        for (int j = 0; j < kSub / 2; ++j) {
          const float p0 = S[2 * j] == -INFINITY ? 0.f : ex2(S[2 * j] - m_use);
          const float p1 = S[2 * j + 1] == -INFINITY ? 0.f : ex2(S[2 * j + 1] - m_use);
          ls += p0 + p1;
          pp[j] = pack_f16x2(p0, p1);
        }
        l += ls;
        tmem_st16(tm + lb + kTmP + 16 * buf, pp);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[buf]);
        have_o = true;
        ++q;
      }
    }, [&](int u, const MqUnit& un, int ps, int pe) {
      const bool active = c < un.ncols;
      if (have_o) {
        wait_bar(p, sm, &sm.pv_done[(q - 1) % kOps], ((q - 1) / kOps) & 1);
        tc_fence_after();
      }
      float M = sm.abort ? __int_as_float(0x7fffffff) : m_use;
      const float inv = (M != M) ? M : (l > 0.f ? 1.0f / l : 0.f);
      const int64_t row = active ? col_row(p, un.b, un.h, un.hc * kCols + c) : 0;
      float* mo = reinterpret_cast<float*>(sm.stage[0]) + c * kMergePitch;
      uint32_t a[32];
#pragma unroll 1
      for (int k = 0; k < 4; ++k) {
        if (have_o) {
          tmem_ld32(tm + lb + kTmO + 32 * k, a);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = 0u;
        }
        if (!active) continue;
        if (cluster) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(mo + 32 * k + i) =
                make_float4(__uint_as_float(a[i]), __uint_as_float(a[i + 1]), __uint_as_float(a[i + 2]),
                            __uint_as_float(a[i + 3]));
        } else {
          uint4* dst = reinterpret_cast<uint4*>(p.out + row * kD + 32 * k);
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
              w[j] = static_cast<uint32_t>(f32_to_bf16_bits(__uint_as_float(a[i + 2 * j]) * inv)) |
                     (static_cast<uint32_t>(f32_to_bf16_bits(__uint_as_float(a[i + 2 * j + 1]) * inv)) << 16);
            dst[i / 8] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (active) {
        if (cluster) {
          sm.ml[c][0] = M;
          sm.ml[c][1] = l;
        } else if (p.lse) {
          p.lse[row] = (M != M) ? M : 0.69314718055994531f * (M + log2f(l));
        }
      }
      tc_fence_before();
      merge_if_cluster(u, un, ps, pe);
    });
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tm, kTmCols);
  }
}

}  // namespace mq
}  // namespace kvq
