// kvq_device.cuh -- small device helpers shared by the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kvq_internal.h"

namespace kvq {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Round-to-nearest-even float -> bf16 bits.
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Row pointers of one position of one unit (decode side).
struct RowRef {
  const uint8_t* k;    // K codes or bf16 row
  const uint8_t* ksz;  // K (s, z) half2 per group, or null for bf16 rows
  const uint8_t* v;
  const uint8_t* vsz;
  int kbits, vbits;    // 16 = bf16
};

__device__ __forceinline__ RowRef row_ref(const Params& p, const UnitInfo& ui, int32_t pos) {
  RowRef r;
  if (pos < p.vs || pos >= p.ve) {
    const int64_t tr = pos < p.vs ? pos : pos - p.Tv;
    const int64_t row = (static_cast<int64_t>(ui.b) * p.Hkv + ui.h) * p.T_text + tr;
    r.k = p.seg[KVQ_SEG_TEXT_K] + row * (2 * kD);
    r.v = p.seg[KVQ_SEG_TEXT_V] + row * (2 * kD);
    r.ksz = r.vsz = nullptr;
    r.kbits = r.vbits = 16;
  } else if (ui.prot) {
    const int64_t row = (static_cast<int64_t>(ui.b) * p.n_prot + ui.slot) * p.Tv + (pos - p.vs);
    r.k = p.seg[KVQ_SEG_PROT_K] + row * (2 * kD);
    r.v = p.seg[KVQ_SEG_PROT_V] + row * (2 * kD);
    r.ksz = r.vsz = nullptr;
    r.kbits = r.vbits = 16;
  } else {
    const int64_t row = (static_cast<int64_t>(ui.b) * p.n_packed + ui.slot) * p.Tv_pad + (pos - p.vs);
    r.k = p.seg[KVQ_SEG_K_CODES] + row * p.krow;
    r.v = p.seg[KVQ_SEG_V_CODES] + row * p.vrow;
    r.ksz = p.kb < 16 ? p.seg[KVQ_SEG_K_SZ] + row * p.kszrow : nullptr;
    r.vsz = p.vb < 16 ? p.seg[KVQ_SEG_V_SZ] + row * p.vszrow : nullptr;
    r.kbits = p.kb;
    r.vbits = p.vb;
  }
  return r;
}

}  // namespace kvq
