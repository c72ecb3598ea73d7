// kvq_append.cu -- kvq_quantize_append: write new positions into the cache.
//
// "VLM_KV_Quantization" (nuiw.github.io), sections 1 and 4: the historical
// visual K and V are quantised to INT8/INT4/INT2 with a group size, K and V
// each with their own bit-width; text and current-step positions are never
// quantised (intro checklist).  HeadGuard brief, key ideas: protected KV
// heads keep their visual K and V in bf16.
//
// One warp per (b, h, 8 consecutive positions): 4 lanes per D = 128 row,
// each lane owning the 32 elements of its slice of the stored row (group
// min and max combine over the row's 4 lanes with shuffles).  The
// arithmetic is the fp32 spec the
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

constexpr int kLanesPerRow = 4;                     // lanes per D = 128 row

constexpr int kRowsPerWarp = 32 / kLanesPerRow;     // 8


// The row's 4 lanes each own one slice of the stored row (kvq.h storage
// order): K slice t = elements d = 32P + 8t + j (P = 0..3, j = 0..7); V
// slices 2l, 2l + 1 = elements d = 16m + 8r + 2l + n' (m = 0..7, r, n' =
// 0, 1).  A lane loads exactly those elements, as 4 chunks of 8 (chunk k =
// 32-element block k of the row for K; m in {2k, 2k+1} for V, so chunk k
// lies in quantisation group k / (G/32) either way), quantises them and
// packs its slice words without any exchange.  w[k][q] holds elements
// j = 2q, 2q + 1 of chunk k (K: d = 32k + 8t + j; V: q = 2m' + r, m = 2k + m',
// n' = j mod 2).
//
// Destination of element j = 4e + i (K) / j = 2q + n' (V) of chunk k:
//   K b = 2: word floor(i/2), bit 16e + 2 c(k, i mod 2), c = {4,7},{3,6},{2,5},{0,1}
//   K b = 4: word i,          bit 16e + 4k
//   K b = 8: word 2k + floor(i/2), bit 16e + 8 (i mod 2)
//   V b = 2: word n',              bit 8k + 2q
//   V b = 4: word 2n' + floor(k/2), bit 16 (k mod 2) + 4q
//   V b = 8: word 4n' + k,          bit 8q
template <int BITS, bool kV>
__device__ __forceinline__ int dst_word(int k, int j) {
  if constexpr (!kV) {
    const int i = j & 3;
    return BITS == 2 ? (i >> 1) : (BITS == 4 ? i : 2 * k + (i >> 1));
  } else {
    const int n = j & 1;
    return BITS == 2 ? n : (BITS == 4 ? 2 * n + (k >> 1) : 4 * n + k);
  }
}
template <int BITS, bool kV>
__device__ __forceinline__ int dst_bit(int k, int j) {
  if constexpr (!kV) {
    const int e = j >> 2, i = j & 3;
    if constexpr (BITS == 2) {
      const int c = k == 0 ? ((i & 1) ? 7 : 4) : k == 1 ? ((i & 1) ? 6 : 3) : k == 2 ? ((i & 1) ? 5 : 2) : (i & 1);
      return 16 * e + 2 * c;
    }
    return BITS == 4 ? 16 * e + 4 * k : 16 * e + 8 * (i & 1);
  } else {
    const int q = j >> 1;
    return BITS == 2 ? 8 * k + 2 * q : (BITS == 4 ? 16 * (k & 1) + 4 * q : 8 * q);
  }
}

// Quantise the lane's 32 elements (4 chunks of 8, see above) and store its
// slice words and, for the groups this lane is responsible for, z and s.
// `gmask` = the 4 lanes of this row (shuffle partners).
template <int BITS, bool kV, int G>
__device__ __forceinline__ void quantize_lane(const uint32_t (&w)[4][4], int part, uint32_t gmask,
                                              uint8_t* codes_row, uint8_t* sz_row) {
  constexpr int NG = kD / G;        // groups per row
  constexpr int CPG = G / 32;       // chunks per group
  constexpr uint32_t cmax = (1u << BITS) - 1u;
  // group min / max: the lane's chunks, then the row's 4 lanes
  float mn[NG], mx[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&w[g * CPG][0]);
    __nv_bfloat162 bb = a;
#pragma unroll
    for (int k = g * CPG; k < (g + 1) * CPG; ++k)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&w[k][q]);
        a = __hmin2(a, v);
        bb = __hmax2(bb, v);
      }
    mn[g] = fminf(__low2float(a), __high2float(a));
    mx[g] = fmaxf(__low2float(bb), __high2float(bb));
  }
#pragma unroll
  for (int off = 1; off < kLanesPerRow; off <<= 1)
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      mn[g] = fminf(mn[g], __shfl_xor_sync(gmask, mn[g], off, kLanesPerRow));
      mx[g] = fmaxf(mx[g], __shfl_xor_sync(gmask, mx[g], off, kLanesPerRow));
    }
  float zf[NG], sf[NG], rs[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const float m0 = __fadd_rn(mn[g], 0.0f);  // -0 -> +0: signed zeros compare equal
    const float s32 = __fdiv_rn(__fsub_rn(mx[g], m0), static_cast<float>(cmax));
    const __half sh = __float2half_rn(s32);
    const __half zh = __float2half_rn(m0);
    sf[g] = __half2float(sh);
    zf[g] = __half2float(zh);
    // A group whose stored scale is 0 gets code 0 everywhere: with rs = 0
    // every quotient is 0 (or NaN for an infinite input, which also converts
    // to 0) and no near-tie is flagged.
    rs[g] = sf[g] != 0.0f ? __frcp_rn(sf[g]) : 0.0f;
    if (g == part) {  // lane g stores group g: fp16 [z_0 .., s_0 ..]
      reinterpret_cast<__half*>(sz_row)[g] = zh;
      reinterpret_cast<__half*>(sz_row)[NG + g] = sh;
    }
  }
  // code = clamp(rint(fl(fl(x - z) / s))).  With d = fl(x - z) and
  // rs = fl(1/s), the exact product p = d * rs is within 2^-24 |q| of the
  // quotient q = d / s, so rint(p) = rint(q) unless p lies that close to
  // k + 1/2.  One FMA, t = fl(p + 1.5 * 2^23), rounds p to an integer once
  // (|p| < 2^22: t = 1.5 * 2^23 + rint(p), half to even) and its low mantissa
  // bits are that integer -- no conversion instruction; a second FMA gives
  // e = fl(p - rint(p)), within 2^-25 of the exact distance.  |q| <= 1.5
  // (2^b - 1) + 1 for finite inputs, so a window of 2^-21 (2 (2^b - 1) + 2)
  // around 1/2 (0.5 - win is exact) holds every near-tie with room to
  // spare; only those are redone with the IEEE division (rare), after one
  // vote for the row slice.  Every lane runs the same instructions so the
  // row's votes stay converged.
  const float win = 4.76837158203125e-7f * (2.0f * static_cast<float>(cmax) + 2.0f);
  constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
  uint32_t out[BITS];
#pragma unroll
  for (int q = 0; q < BITS; ++q) out[q] = 0u;
  uint32_t need = 0;  // near-ties: bit 8k + j
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int g = k / CPG;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t pw = w[k][j >> 1];
      const float x = (j & 1) ? bf16_hi(pw) : bf16_lo(pw);
      const float d = __fsub_rn(x, zf[g]);
      const float t = __fmaf_rn(d, rs[g], kRound);
      const float e = __fmaf_rn(d, rs[g], -__fsub_rn(t, kRound));
      if (fabsf(e) >= 0.5f - win) need |= 1u << (8 * k + j);
      const int ci = static_cast<int>(__float_as_uint(t) - __float_as_uint(kRound));
      const uint32_t code = static_cast<uint32_t>(__vimin_s32_relu(ci, static_cast<int>(cmax)));
      out[dst_word<BITS, kV>(k, j)] += code << dst_bit<BITS, kV>(k, j);  // disjoint bit fields
    }
  }
  if (__any_sync(gmask, need != 0)) {
    // Rare: the flagged elements of each chunk one at a time; registers are
    // picked with selects so that no array goes to local memory.
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t nk = (need >> (8 * k)) & 0xffu;
#pragma unroll 1
      while (nk) {
        const int j = __ffs(nk) - 1;
        nk &= nk - 1u;
        const uint32_t lo = (j & 2) ? w[k][1] : w[k][0], hi = (j & 2) ? w[k][3] : w[k][2];
        const uint32_t pw = (j & 4) ? hi : lo;
        const float x = (j & 1) ? bf16_hi(pw) : bf16_lo(pw);
        const float u = __fdiv_rn(__fsub_rn(x, zf[k / CPG]), sf[k / CPG]);
        const uint32_t code = min(__float2uint_rn(u), cmax);  // round half to even; < 0 -> 0
        const int wd = dst_word<BITS, kV>(k, j), bt = dst_bit<BITS, kV>(k, j);
#pragma unroll
        for (int q = 0; q < BITS; ++q)
          if (q == wd) out[q] = (out[q] & ~(cmax << bt)) | (code << bt);
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

template <int BITS, bool kV>
__device__ __forceinline__ void quantize_lane_g(int G, const uint32_t (&w)[4][4], int part, uint32_t gmask,
                                                uint8_t* codes_row, uint8_t* sz_row) {
  if (G == 32) quantize_lane<BITS, kV, 32>(w, part, gmask, codes_row, sz_row);
  else if (G == 64) quantize_lane<BITS, kV, 64>(w, part, gmask, codes_row, sz_row);
  else quantize_lane<BITS, kV, 128>(w, part, gmask, codes_row, sz_row);
}

// Element offsets (in bf16) of the lane's words: K chunk k word q -> 32k +
// 8 part + 2q; V chunk k word q (= 2m' + r) -> 16 (2k + m') + 8r + 2 part.
__device__ __forceinline__ int k_elem(int k, int q, int part) { return 32 * k + 8 * part + 2 * q; }
__device__ __forceinline__ int v_elem(int k, int q, int part) {
  return 16 * (2 * k + (q >> 1)) + 8 * (q & 1) + 2 * part;
}

// One warp per (b, h, 8 consecutive positions); 4 lanes per row, each lane
// the elements of its slice of the stored row (K: four 16-byte loads; V:
// sixteen 4-byte loads, all in flight before any use).
__device__ __forceinline__ void append_rows(const AppendArgs& a) {
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
  const int mode = p.prot[h];  // 0 quantised, 1 K and V protected, 2 K protected

  const int64_t src = b * a.sb + h * a.sh + i * a.st;
  uint32_t kw[4][4], vw[4][4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(a.kin + src + k_elem(k, 0, part)));
    kw[k][0] = x.x; kw[k][1] = x.y; kw[k][2] = x.z; kw[k][3] = x.w;
#pragma unroll
    for (int q = 0; q < 4; ++q) vw[k][q] = __ldg(reinterpret_cast<const uint32_t*>(a.vin + src + v_elem(k, q, part)));
  }
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const uint32_t (&w)[4][4] = which ? vw : kw;
    uint8_t* dst;
    if (!visual) {
      const int64_t tr = t < p.vs ? t : t - p.Tv;
      const int64_t row = (static_cast<int64_t>(b) * p.Hkv + h) * p.T_text + tr;
      dst = const_cast<uint8_t*>(p.seg[which ? KVQ_SEG_TEXT_V : KVQ_SEG_TEXT_K]) + row * (2 * kD);
    } else if (which == 0 && mode != 0) {  // protected or K-only head: bf16 K
      const int64_t row = prot_k_row(p, b, mode == 1 ? kClsProt : kClsKonly, p.slot[h]) * p.Tv + (t - p.vs);
      dst = const_cast<uint8_t*>(p.seg[KVQ_SEG_PROT_K]) + row * (2 * kD);
    } else if (which == 1 && mode == 1) {  // protected head: bf16 V
      const int64_t row = (static_cast<int64_t>(b) * p.n_prot + p.slot[h]) * p.Tv + (t - p.vs);
      dst = const_cast<uint8_t*>(p.seg[KVQ_SEG_PROT_V]) + row * (2 * kD);
    } else {
      const int bits = which ? p.vb : p.kb;
      const int64_t row =
          (which ? packed_v_row(p, b, mode == 2 ? kClsKonly : kClsPacked, p.slot[h])
                 : static_cast<int64_t>(b) * p.n_packed + p.slot[h]) * p.Tv_pad + (t - p.vs);
      uint8_t* codes = const_cast<uint8_t*>(p.seg[which ? KVQ_SEG_V_CODES : KVQ_SEG_K_CODES]) +
                       row * (which ? p.vrow : p.krow);
      if (bits < 16) {
        uint8_t* sz = const_cast<uint8_t*>(p.seg[which ? KVQ_SEG_V_SZ : KVQ_SEG_K_SZ]) +
                      row * (which ? p.vszrow : p.kszrow);
        if (which) {
          if (bits == 2) quantize_lane_g<2, true>(p.G, w, part, gmask, codes, sz);
          else if (bits == 4) quantize_lane_g<4, true>(p.G, w, part, gmask, codes, sz);
          else quantize_lane_g<8, true>(p.G, w, part, gmask, codes, sz);
        } else {
          if (bits == 2) quantize_lane_g<2, false>(p.G, w, part, gmask, codes, sz);
          else if (bits == 4) quantize_lane_g<4, false>(p.G, w, part, gmask, codes, sz);
          else quantize_lane_g<8, false>(p.G, w, part, gmask, codes, sz);
        }
        continue;
      }
      dst = codes;
    }
    // bf16 row: the lane's elements go back to where they came from
    uint16_t* o = reinterpret_cast<uint16_t*>(dst);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (which) {
#pragma unroll
        for (int q = 0; q < 4; ++q) *reinterpret_cast<uint32_t*>(o + v_elem(k, q, part)) = w[k][q];
      } else {
        *reinterpret_cast<uint4*>(o + k_elem(k, 0, part)) = make_uint4(w[k][0], w[k][1], w[k][2], w[k][3]);
      }
    }
  }
}

// The next kernel in the stream may read cache rows before its own
// dependency wait (decode preload), so a CTA lets it launch only once all of
// the CTA's rows are written and fenced.
__global__ void __launch_bounds__(256, 3) append_kernel(const __grid_constant__ AppendArgs a) {
  pdl_wait();  // the previous kernel in the stream may still read the cache
  append_rows(a);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) pdl_launch_dependents();
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
