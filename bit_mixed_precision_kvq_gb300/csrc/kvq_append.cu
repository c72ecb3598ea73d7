// kvq_append.cu -- kvq_quantize_append: write new positions into the cache.
//
// "VLM_KV_Quantization" (nuiw.github.io), sections 1 and 4: the historical
// visual K and V are quantised to INT8/INT4/INT2 with a group size, K and V
// each with their own bit-width; text and current-step positions are never
// quantised (intro checklist).  HeadGuard brief, key ideas: protected KV
// heads keep their visual K and V in bf16.
//
// One warp per (b, h, position); lane l owns elements 4l..4l+3 of the
// D = 128 row (one 8-byte load).  A quantisation group of G elements spans
// G/4 lanes, reduced with xor-shuffles.  The arithmetic is the fp32 spec the
// oracle restates: r = max - min (RN), s = fp16(r / (2^b - 1)) (IEEE div),
// z = fp16(min + 0), code = clamp(rint((x - z) / s), 0, 2^b - 1) using the
// stored s and z, code 0 if s == 0.  Intrinsics pin every rounding so that
// no contraction or fast division can change a code.
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_ptx.cuh"

namespace kvq {
namespace {

__device__ __forceinline__ void quantize_store(const Params& p, uint8_t* codes_row, uint8_t* sz_row,
                                               int bits, const float x[4], int lane) {
  const int lanes_per_group = p.G >> 2;  // 8, 16 or 32
  float mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
  float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  for (int off = 1; off < lanes_per_group; off <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  mn = __fadd_rn(mn, 0.0f);  // -0 -> +0: signed zeros compare equal
  const float qmax = static_cast<float>((1 << bits) - 1);
  const float s32 = __fdiv_rn(__fsub_rn(mx, mn), qmax);
  const __half sh = __float2half_rn(s32);
  const __half zh = __float2half_rn(mn);
  const float sf = __half2float(sh);
  const float zf = __half2float(zh);
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float r = 0.0f;
    if (sf != 0.0f) {
      r = rintf(__fdiv_rn(__fsub_rn(x[i], zf), sf));
      r = fminf(fmaxf(r, 0.0f), qmax);
    }
    c[i] = static_cast<uint32_t>(r);
  }
  uint32_t* words = reinterpret_cast<uint32_t*>(codes_row);
  if (bits == 8) {
    words[lane] = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
  } else if (bits == 4) {
    const uint32_t mine = c[0] | (c[1] << 4) | (c[2] << 8) | (c[3] << 12);
    const uint32_t next = __shfl_down_sync(0xffffffffu, mine, 1);
    if ((lane & 1) == 0) words[lane >> 1] = mine | (next << 16);
  } else {  // bits == 2
    const uint32_t mine = c[0] | (c[1] << 2) | (c[2] << 4) | (c[3] << 6);
    const uint32_t n1 = __shfl_down_sync(0xffffffffu, mine, 1);
    const uint32_t n2 = __shfl_down_sync(0xffffffffu, mine, 2);
    const uint32_t n3 = __shfl_down_sync(0xffffffffu, mine, 3);
    if ((lane & 3) == 0) words[lane >> 2] = mine | (n1 << 8) | (n2 << 16) | (n3 << 24);
  }
  if ((lane & (lanes_per_group - 1)) == 0) {
    __half2 sz;
    sz.x = sh;
    sz.y = zh;
    reinterpret_cast<__half2*>(sz_row)[(4 * lane) / p.G] = sz;
  }
}

struct AppendArgs {
  Params p;
  const uint16_t* kin;
  const uint16_t* vin;
  int64_t sb, sh, st;
  int32_t t0, n_tok;
};

__global__ void __launch_bounds__(256) append_kernel(const __grid_constant__ AppendArgs a) {
  pdl_wait();  // the previous kernel in the stream may still read the cache
  pdl_launch_dependents();
  const Params& p = a.p;
  const uint16_t* __restrict__ kin = a.kin;
  const uint16_t* __restrict__ vin = a.vin;
  const int64_t sb = a.sb, sh = a.sh, st = a.st;
  const int32_t t0 = a.t0, n_tok = a.n_tok;
  const int lane = threadIdx.x & 31;
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nrows = static_cast<int64_t>(p.B) * p.Hkv * n_tok;
  if (wid >= nrows) return;
  const int32_t i = static_cast<int32_t>(wid % n_tok);
  const int64_t bh = wid / n_tok;
  const int32_t h = static_cast<int32_t>(bh % p.Hkv);
  const int32_t b = static_cast<int32_t>(bh / p.Hkv);
  const int32_t t = t0 + i;
  const int64_t src = b * sb + h * sh + i * st + 4 * lane;
  const bool visual = t >= p.vs && t < p.ve;
  const bool prot = p.prot[h] != 0;

#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const uint16_t* in = which ? vin : kin;
    const uint2 raw = *reinterpret_cast<const uint2*>(in + src);
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
        const float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
        quantize_store(p, codes, sz, bits, x, lane);
        continue;
      }
      dst = codes;
    }
    *reinterpret_cast<uint2*>(dst + 8 * lane) = raw;
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
  if (reinterpret_cast<uintptr_t>(k_bf16) % 8 != 0 || reinterpret_cast<uintptr_t>(v_bf16) % 8 != 0)
    return KVQ_ERR_INVALID_ARG;
  if (stride_b < 0 || stride_h < 0 || stride_t < 0 || stride_b % 4 || stride_h % 4 || stride_t % 4)
    return KVQ_ERR_INVALID_ARG;
  if (t0 < 0 || n_tok < 0) return KVQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(t0) + n_tok > L->d.T_cap) return KVQ_ERR_CAPACITY;
  if (n_tok == 0) return KVQ_OK;
  kvq::Params p;
  kvq_fill_params(L, &p);
  uint8_t* base = static_cast<uint8_t*>(cache);
  for (int s = 0; s < KVQ_NSEG; ++s) p.seg[s] = base + L->off[s];
  const int64_t rows = static_cast<int64_t>(L->d.B) * L->d.H_kv * n_tok;
  const int64_t blocks = (rows + 7) / 8;
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
