// kvq_append.cu -- kvq_quantize_append: write new positions into the cache.
//
// "VLM_KV_Quantization" (nuiw.github.io), sections 1 and 4: the historical
// visual K and V are quantised to INT8/INT4/INT2 with a group size, K and V
// each with their own bit-width; text and current-step positions are never
// quantised (intro checklist).  HeadGuard brief, key ideas: protected KV
// heads keep their visual K and V in bf16.
//
// One warp per (b, h, 8 consecutive positions): 4 lanes per D = 128 row,
// each lane owning 32 consecutive elements (a whole group for G = 32; for
// G = 64 / 128 the 2 / 4 lanes of a group combine min and max with
// shuffles).  The arithmetic is the fp32 spec the
// oracle restates: r = max - min (RN), s = fp16(r / (2^b - 1)) (IEEE div),
// z = fp16(min + 0), code = clamp(rint((x - z) / s), 0, 2^b - 1) using the
// stored s and z, code 0 if s == 0.  Intrinsics pin every rounding so that
// no contraction or fast division can change a code.
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_ptx.cuh"

namespace kvq {
namespace {

struct AppendArgs {
  Params p;
  const uint16_t* kin;
  const uint16_t* vin;
  int64_t sb, sh, st;
  int32_t t0, n_tok;
};

constexpr int kLaneElems = 32;                      // consecutive elements of a row per lane
constexpr int kLanesPerRow = kD / kLaneElems;       // 4
constexpr int kRowsPerWarp = 32 / kLanesPerRow;     // 8

// The correctly rounded quotient, kept out of line: it is needed only for
// near-ties.
__device__ __noinline__ float exact_quotient(float d, float s) { return __fdiv_rn(d, s); }

// Value of blk[sel] for a runtime sel in [0, 4) without local memory.
__device__ __forceinline__ uint32_t pick4(const uint32_t (&blk)[4], int sel) {
  const uint32_t lo = (sel & 1) ? blk[1] : blk[0];
  const uint32_t hi = (sel & 1) ? blk[3] : blk[2];
  return (sel & 2) ? hi : lo;
}

// Quantise the lane's 32 elements (16 bf16 pairs in w[]) of one row and
// store them in the cache's storage order (slot sigma(d) of the row, see
// kvq.h).  The lane (part) owns elements d = 32 part + e, e in [0, 32).  Its
// codes land in every lane's slice of the row, so each lane first builds,
// for each of the row's 4 lanes, the words of that lane's slice with its own
// codes already in place (zeros elsewhere); a 4-lane exchange (3 xor-shuffle
// rounds) then gives every lane the pieces of its own slice, which it ORs
// and stores.
//   K, d = 32P + 8t + 4e' + i (P = part): slice t (slots 32t ..) belongs to
//     lane t.  Code (t, e', i) goes to slice word / bit
//       b = 2: word floor(i/2), bit 16e' + 2c(P, i mod 2)
//       b = 4: word i,          bit 16e' + 4P
//       b = 8: word 2P + floor(i/2), bit 16e' + 8 (i mod 2)
//   V, d = 16m + 8r + n (m = 2 part + m'): slices 2l, 2l+1 (slots 16n ..)
//     belong to lane l = floor(n/2).  Code (m', r, n) goes to bit
//       b = 2: 8 part + 2c'            of the slice's word
//       b = 4: 16 (part mod 2) + 4c'   of the slice's word floor(part/2)
//       b = 8: 8c'                     of the slice's word part
//     with c' = 2m' + r.
// `gmask` = the 4 lanes of this row (shuffle partners).
template <int BITS, bool kV>
__device__ __forceinline__ void quantize_lane(const uint32_t (&w)[16], int G, int part, uint32_t gmask,
                                              uint8_t* codes_row, uint8_t* sz_row) {
  // group min / max over the lane's elements (packed bf16 pairs), then over
  // the lanes of the group
  __nv_bfloat162 mn2 = *reinterpret_cast<const __nv_bfloat162*>(&w[0]);
  __nv_bfloat162 mx2 = mn2;
#pragma unroll
  for (int i = 1; i < 16; ++i) {
    const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
    mn2 = __hmin2(mn2, v);
    mx2 = __hmax2(mx2, v);
  }
  float mn = fminf(__low2float(mn2), __high2float(mn2));
  float mx = fmaxf(__low2float(mx2), __high2float(mx2));
  for (int off = 1; off < G / kLaneElems; off <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(gmask, mn, off, kLanesPerRow));
    mx = fmaxf(mx, __shfl_xor_sync(gmask, mx, off, kLanesPerRow));
  }
  mn = __fadd_rn(mn, 0.0f);  // -0 -> +0: signed zeros compare equal
  constexpr uint32_t cmax = (1u << BITS) - 1u;
  const float s32 = __fdiv_rn(__fsub_rn(mx, mn), static_cast<float>(cmax));
  const __half sh = __float2half_rn(s32);
  const __half zh = __float2half_rn(mn);
  const float sf = __half2float(sh);
  const float zf = __half2float(zh);
  // Store the group's z and s once (first lane of the group): fp16 row
  // [z_0 .. z_{ng-1}, s_0 .. s_{ng-1}].
  if ((part & (G / kLaneElems - 1)) == 0) {
    const int ng = kD / G, g = (part * kLaneElems) / G;
    reinterpret_cast<__half*>(sz_row)[g] = zh;
    reinterpret_cast<__half*>(sz_row)[ng + g] = sh;
  }
  // blk[x][l]: word x of what this lane sends to row lane l
  constexpr int kSend = (!kV && BITS == 4) ? 4 : 2;
  uint32_t blk[kSend][4];
#pragma unroll
  for (int x = 0; x < kSend; ++x)
#pragma unroll
    for (int l = 0; l < 4; ++l) blk[x][l] = 0u;
  // crumb table of 2-bit K registers: c(P, 0), c(P, 1)
  const uint32_t c0 = (0x0234u >> (4 * part)) & 0xFu;  // P = 0..3 -> 4, 3, 2, 0
  const uint32_t c1 = (0x1567u >> (4 * part)) & 0xFu;  // P = 0..3 -> 7, 6, 5, 1
  // code = clamp(rint(fl(fl(x - z) / s))).  The quotient is first formed as
  // fl(d * fl(1/s)), within 3 * 2^-24 |u| of the correctly rounded one; rint
  // is constant between half-integers, so both give the same code unless the
  // product lies within that distance of k + 1/2.  |u| <= 1.5 (2^b - 1) + 1
  // for finite inputs, so a fixed window of 2^-21 (2 (2^b - 1) + 2) covers
  // it; only then is the IEEE division evaluated (out of line, rare).
  // A group whose stored scale is 0 gets code 0 everywhere: with rs = 0 every
  // quotient is 0 (or NaN for an infinite input, which also converts to 0)
  // and no near-tie is flagged.  Every lane runs the same code so that the
  // row's shuffles and votes stay converged.
  {
    const float rs = sf != 0.0f ? __frcp_rn(sf) : 0.0f;
    const float win = 4.76837158203125e-7f * (2.0f * static_cast<float>(cmax) + 2.0f);
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {  // 8 elements at a time: e = 8 c8 + k
      float d[8], u[8];
      uint32_t need = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t pw = w[c8 * 4 + (k >> 1)];
        const float x = (k & 1) ? bf16_hi(pw) : bf16_lo(pw);
        d[k] = __fsub_rn(x, zf);
        u[k] = __fmul_rn(d[k], rs);
        const float fr = __fsub_rn(__fsub_rn(u[k], floorf(u[k])), 0.5f);  // exact for |u| < 2^23
        if (fabsf(fr) <= win) need |= 1u << k;
      }
      if (__any_sync(gmask, need != 0)) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (need & (1u << k)) u[k] = exact_quotient(d[k], sf);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t code = min(__float2uint_rn(u[k]), cmax);  // round half to even; < 0 -> 0
        if constexpr (!kV) {
          // K: destination lane t = c8, e' = k / 4, i = k % 4
          const int ep = k >> 2, i = k & 3;
          if constexpr (BITS == 2) {
            blk[i >> 1][c8] |= code << (16 * ep + 2 * ((i & 1) ? c1 : c0));
          } else if constexpr (BITS == 4) {
            blk[i][c8] |= code << (16 * ep + 4 * part);
          } else {
            blk[i >> 1][c8] |= code << (16 * ep + 8 * (i & 1));
          }
        } else {
          // V: c' = c8 (= 2m' + r), n = k -> destination lane k / 2, slice k % 2
          if constexpr (BITS == 2) {
            blk[k & 1][k >> 1] |= code << (8 * part + 2 * c8);
          } else if constexpr (BITS == 4) {
            blk[k & 1][k >> 1] |= code << (16 * (part & 1) + 4 * c8);
          } else {
            blk[k & 1][k >> 1] |= code << (8 * c8);
          }
        }
      }
    }
  }
  // 4-lane exchange: in round r each lane swaps with lane part ^ r.
  uint32_t piece[kSend][4];  // piece[x][src]: word x received from row lane src
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int peer = part ^ r;
#pragma unroll
    for (int x = 0; x < kSend; ++x) {
      const uint32_t mine = pick4(blk[x], peer);
      const uint32_t got = r ? __shfl_xor_sync(gmask, mine, r, kLanesPerRow) : mine;
#pragma unroll
      for (int src = 0; src < 4; ++src)
        if (peer == src) piece[x][src] = got;  // selects: stays in registers
    }
  }
  // This lane's BITS words: its K slice, or its two V slices (2 part, 2 part + 1).
  uint32_t out[BITS];
#pragma unroll
  for (int q = 0; q < BITS; ++q) out[q] = 0u;
#pragma unroll
  for (int src = 0; src < 4; ++src) {
    if constexpr (!kV) {
      if constexpr (BITS == 8) {
        out[2 * src] = piece[0][src];
        out[2 * src + 1] = piece[1][src];
      } else {
#pragma unroll
        for (int x = 0; x < kSend; ++x) out[x] |= piece[x][src];
      }
    } else {
      constexpr int kSliceWords = BITS / 2;
#pragma unroll
      for (int sl = 0; sl < 2; ++sl) {
        if constexpr (BITS == 2) out[sl] |= piece[sl][src];
        else if constexpr (BITS == 4) out[kSliceWords * sl + src / 2] |= piece[sl][src];
        else out[kSliceWords * sl + src] = piece[sl][src];
      }
    }
  }
  uint8_t* dst = codes_row + part * 4 * BITS;
  if constexpr (BITS == 2) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(out[0], out[1]);
  } else if constexpr (BITS == 4) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
  } else {
    *reinterpret_cast<uint4*>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
    *reinterpret_cast<uint4*>(dst + 16) = make_uint4(out[4], out[5], out[6], out[7]);
  }
}

// One warp per (b, h, 8 consecutive positions); 4 lanes per row, each lane
// 32 consecutive elements (four 16-byte loads of K and of V, all in flight
// before any use).
__global__ void __launch_bounds__(256) append_kernel(const __grid_constant__ AppendArgs a) {
  pdl_wait();  // the previous kernel in the stream may still read the cache
  pdl_launch_dependents();
  const Params& p = a.p;
  const int lane = threadIdx.x & 31;
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int32_t n_chunks = (a.n_tok + kRowsPerWarp - 1) / kRowsPerWarp;
  const int64_t nwarps = static_cast<int64_t>(p.B) * p.Hkv * n_chunks;
  if (wid >= nwarps) return;
  const int rr = lane / kLanesPerRow, part = lane % kLanesPerRow;
  const uint32_t gmask = 0xfu << (kLanesPerRow * rr);
  const int32_t i = static_cast<int32_t>(wid % n_chunks) * kRowsPerWarp + rr;
  if (i >= a.n_tok) return;  // whole 4-lane row groups leave together
  const int64_t bh = wid / n_chunks;
  const int32_t h = static_cast<int32_t>(bh % p.Hkv);
  const int32_t b = static_cast<int32_t>(bh / p.Hkv);
  const int32_t t = a.t0 + i;
  const bool visual = t >= p.vs && t < p.ve;
  const bool prot = p.prot[h] != 0;

  const int64_t src = b * a.sb + h * a.sh + i * a.st + part * kLaneElems;
  uint32_t kw[16], vw[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(a.kin + src) + q);
    const uint4 y = __ldg(reinterpret_cast<const uint4*>(a.vin + src) + q);
    kw[4 * q] = x.x; kw[4 * q + 1] = x.y; kw[4 * q + 2] = x.z; kw[4 * q + 3] = x.w;
    vw[4 * q] = y.x; vw[4 * q + 1] = y.y; vw[4 * q + 2] = y.z; vw[4 * q + 3] = y.w;
  }
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const uint32_t (&w)[16] = which ? vw : kw;
    uint8_t* dst;
    if (!visual) {
      const int64_t tr = t < p.vs ? t : t - p.Tv;
      const int64_t row = (static_cast<int64_t>(b) * p.Hkv + h) * p.T_text + tr;
      dst = const_cast<uint8_t*>(p.seg[which ? KVQ_SEG_TEXT_V : KVQ_SEG_TEXT_K]) + row * (2 * kD);
    } else if (prot) {
      const int64_t row = (static_cast<int64_t>(b) * p.n_prot + p.slot[h]) * p.Tv + (t - p.vs);
      dst = const_cast<uint8_t*>(p.seg[which ? KVQ_SEG_PROT_V : KVQ_SEG_PROT_K]) + row * (2 * kD);
    } else {
      const int bits = which ? p.vb : p.kb;
      const int64_t row = (static_cast<int64_t>(b) * p.n_packed + p.slot[h]) * p.Tv_pad + (t - p.vs);
      uint8_t* codes = const_cast<uint8_t*>(p.seg[which ? KVQ_SEG_V_CODES : KVQ_SEG_K_CODES]) +
                       row * (which ? p.vrow : p.krow);
      if (bits < 16) {
        uint8_t* sz = const_cast<uint8_t*>(p.seg[which ? KVQ_SEG_V_SZ : KVQ_SEG_K_SZ]) +
                      row * (which ? p.vszrow : p.kszrow);
        if (which) {
          if (bits == 2) quantize_lane<2, true>(w, p.G, part, gmask, codes, sz);
          else if (bits == 4) quantize_lane<4, true>(w, p.G, part, gmask, codes, sz);
          else quantize_lane<8, true>(w, p.G, part, gmask, codes, sz);
        } else {
          if (bits == 2) quantize_lane<2, false>(w, p.G, part, gmask, codes, sz);
          else if (bits == 4) quantize_lane<4, false>(w, p.G, part, gmask, codes, sz);
          else quantize_lane<8, false>(w, p.G, part, gmask, codes, sz);
        }
        continue;
      }
      dst = codes;
    }
    uint4* o = reinterpret_cast<uint4*>(dst + part * kLaneElems * 2);
#pragma unroll
    for (int q = 0; q < 4; ++q) o[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  }
}

}  // namespace
}  // namespace kvq

extern "C" kvq_status kvq_quantize_append(const kvq_layout* L, void* cache, const void* k_bf16,
                                          const void* v_bf16, int64_t stride_b, int64_t stride_h,
                                          int64_t stride_t, int32_t t0, int32_t n_tok,
                                          void* stream) {
  const kvq_status st = kvq_check_layout(L);
  if (st != KVQ_OK) return st;
  if (!cache || !k_bf16 || !v_bf16) return KVQ_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(cache) % 256 != 0) return KVQ_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(k_bf16) % 16 != 0 || reinterpret_cast<uintptr_t>(v_bf16) % 16 != 0)
    return KVQ_ERR_INVALID_ARG;
  if (stride_b < 0 || stride_h < 0 || stride_t < 0 || stride_b % 8 || stride_h % 8 || stride_t % 8)
    return KVQ_ERR_INVALID_ARG;
  if (t0 < 0 || n_tok < 0) return KVQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(t0) + n_tok > L->d.T_cap) return KVQ_ERR_CAPACITY;
  if (n_tok == 0) return KVQ_OK;
  kvq::Params p;
  kvq_fill_params(L, &p);
  uint8_t* base = static_cast<uint8_t*>(cache);
  for (int s = 0; s < KVQ_NSEG; ++s) p.seg[s] = base + L->off[s];
  const int64_t warps = static_cast<int64_t>(L->d.B) * L->d.H_kv *
                       ((n_tok + kvq::kRowsPerWarp - 1) / kvq::kRowsPerWarp);
  const int64_t blocks = (warps + 7) / 8;
  if (blocks > 0x7fffffffLL) return KVQ_ERR_UNSUPPORTED;
  kvq::AppendArgs a;
  a.p = p;
  a.kin = static_cast<const uint16_t*>(k_bf16);
  a.vin = static_cast<const uint16_t*>(v_bf16);
  a.sb = stride_b;
  a.sh = stride_h;
  a.st = stride_t;
  a.t0 = t0;
  a.n_tok = n_tok;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* kargs[1] = {&a};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(&kvq::append_kernel), kargs);
  if (e != cudaSuccess) return kvq_cuda_fail(e);
  return KVQ_OK;
}
