// Device helpers shared by the expert-MLP kernels (k_mlp.cu, k_mlp_ring.cu):
// 16-byte weight chunks dotted with f32 activations (chunk_dot), the warp
// reduction, activation staging and the output store.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstring>
#include <cstdint>

#include "internal.cuh"

namespace moe {
namespace mlp {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = kMlpThreads / 32;

template <int F>
struct FmtT;
template <>
struct FmtT<MOE_F32> {
  static constexpr int kElems = 4;
};
template <>
struct FmtT<MOE_BF16> {
  static constexpr int kElems = 8;
};
template <>
struct FmtT<MOE_INT4_G128> {
  static constexpr int kElems = 32;
};
template <>
struct FmtT<MOE_FP8_E4M3> {
  static constexpr int kElems = 16;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ uint4 ldw(const uint4* p) { return __ldcs(p); }

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// exact (q - 8) for a 4-bit code q: 2^23 + q as a float, minus 2^23 + 8
__device__ __forceinline__ float code_m8(uint32_t word, int sh) {
  return __uint_as_float(((word >> sh) & 0xFu) | 0x4B000000u) - 8388616.0f;
}

template <int F>
__device__ __forceinline__ float chunk_dot(const uint4 w, const float* __restrict__ x);

template <>
__device__ __forceinline__ float chunk_dot<MOE_F32>(const uint4 w, const float* __restrict__ x) {
  const float4 a = *reinterpret_cast<const float4*>(x);
  float s = __uint_as_float(w.x) * a.x;
  s = fmaf(__uint_as_float(w.y), a.y, s);
  s = fmaf(__uint_as_float(w.z), a.z, s);
  s = fmaf(__uint_as_float(w.w), a.w, s);
  return s;
}

template <>
__device__ __forceinline__ float chunk_dot<MOE_BF16>(const uint4 w, const float* __restrict__ x) {
  const float4 a = *reinterpret_cast<const float4*>(x);
  const float4 b = *reinterpret_cast<const float4*>(x + 4);
  float s = bf16_lo(w.x) * a.x;
  s = fmaf(bf16_hi(w.x), a.y, s);
  s = fmaf(bf16_lo(w.y), a.z, s);
  s = fmaf(bf16_hi(w.y), a.w, s);
  s = fmaf(bf16_lo(w.z), b.x, s);
  s = fmaf(bf16_hi(w.z), b.y, s);
  s = fmaf(bf16_lo(w.w), b.z, s);
  s = fmaf(bf16_hi(w.w), b.w, s);
  return s;
}

// 32 codes: nibble i of 32-bit word j is element 8 j + i (low nibble = even column).
__device__ __forceinline__ float int4_word_dot(uint32_t wd, const float* __restrict__ x, float s) {
  const float4 a = *reinterpret_cast<const float4*>(x);
  const float4 b = *reinterpret_cast<const float4*>(x + 4);
  s = fmaf(code_m8(wd, 0), a.x, s);
  s = fmaf(code_m8(wd, 4), a.y, s);
  s = fmaf(code_m8(wd, 8), a.z, s);
  s = fmaf(code_m8(wd, 12), a.w, s);
  s = fmaf(code_m8(wd, 16), b.x, s);
  s = fmaf(code_m8(wd, 20), b.y, s);
  s = fmaf(code_m8(wd, 24), b.z, s);
  s = fmaf(code_m8(wd, 28), b.w, s);
  return s;
}

template <>
__device__ __forceinline__ float chunk_dot<MOE_INT4_G128>(const uint4 w,
                                                         const float* __restrict__ x) {
  float s = 0.f;
  s = int4_word_dot(w.x, x, s);
  s = int4_word_dot(w.y, x + 8, s);
  s = int4_word_dot(w.z, x + 16, s);
  s = int4_word_dot(w.w, x + 24, s);
  return s;
}

// two E4M3 codes (low byte = lower element) -> two exact floats
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t two) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)(two & 0xffffu)));
  __half2 v;
  memcpy(&v, &h, 4);
  return __half22float2(v);
}

// 16 codes: byte i of 32-bit word j is element 4 j + i.  The per-tensor
// scale is applied by the caller to the whole row's dot product.
template <>
__device__ __forceinline__ float chunk_dot<MOE_FP8_E4M3>(const uint4 w, const float* __restrict__ x) {
  const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 a = e4m3x2_to_f2(wd[j]), b = e4m3x2_to_f2(wd[j] >> 16);
    s = fmaf(a.x, x[4 * j], s);
    s = fmaf(a.y, x[4 * j + 1], s);
    s = fmaf(b.x, x[4 * j + 2], s);
    s = fmaf(b.y, x[4 * j + 3], s);
  }
  return s;
}

template <int F>
__device__ __forceinline__ size_t row_bytes(int K) {
  return F == MOE_F32 ? (size_t)K * 4
                      : (F == MOE_BF16 ? (size_t)K * 2 : (F == MOE_FP8_E4M3 ? (size_t)K : (size_t)K / 2));
}

__device__ __forceinline__ float bf16_bits(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

// position of the (s+1)-th set bit of m
__device__ __forceinline__ int nth_set_bit(unsigned m, int s) {
  for (int i = 0; i < s; ++i) m &= m - 1u;
  return __ffs(m) - 1;
}

template <int F>
__device__ __forceinline__ void store_y(const MlpArgs& a, int t, int n, float v) {
  const size_t o = (size_t)t * a.H + n;
  if (F == MOE_F32) {
    if (a.residual) v += reinterpret_cast<const float*>(a.x)[o];
    reinterpret_cast<float*>(a.y)[o] = v;
  } else {
    if (a.residual) v += bf16_bits(reinterpret_cast<const uint16_t*>(a.x)[o]);
    reinterpret_cast<__nv_bfloat16*>(a.y)[o] = __float2bfloat16_rn(v);
  }
}

// x (bf16 or f32) of token t -> f32 in shared memory, 16-byte loads, by
// threads tid = 0 .. nthr - 1
template <int F>
__device__ __forceinline__ void stage_x(float* dst, const MlpArgs& a, int t, int tid, int nthr) {
  const int H = a.H;
  const void* row = reinterpret_cast<const uint8_t*>(a.x) + (size_t)t * H * (F == MOE_F32 ? 4 : 2);
  if (reinterpret_cast<uintptr_t>(row) & 15) {          // caller's x not 16-byte aligned
    for (int i = tid; i < H; i += nthr)
      dst[i] = F == MOE_F32 ? reinterpret_cast<const float*>(row)[i]
                            : bf16_bits(reinterpret_cast<const uint16_t*>(row)[i]);
    return;
  }
  if (F == MOE_F32) {
    const float4* s = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.x) + (size_t)t * H);
    for (int i = tid; i < H / 4; i += nthr) reinterpret_cast<float4*>(dst)[i] = s[i];
  } else {
    const uint4* s = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.x) + (size_t)t * H);
    for (int i = tid; i < H / 8; i += nthr) {
      const uint4 v = s[i];
      float4* d = reinterpret_cast<float4*>(dst + 8 * i);
      d[0] = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
      d[1] = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
    }
  }
}

// h of token t (k * I floats, written by other CTAs) -> shared memory, L2 reads
__device__ __forceinline__ void stage_h(float* dst, const MlpArgs& a, int t, int tid, int nthr) {
  const float* row = a.h + (size_t)t * a.k * a.I;
  if (reinterpret_cast<uintptr_t>(row) & 15) {          // caller's scratch not 16-byte aligned
    for (int i = tid; i < a.k * a.I; i += nthr) dst[i] = __ldcg(row + i);
    return;
  }
  const int n4 = a.k * a.I / 4;
  const float4* s = reinterpret_cast<const float4*>(row);
  for (int i = tid; i < n4; i += nthr) reinterpret_cast<float4*>(dst)[i] = __ldcg(s + i);
}

}  // namespace mlp
}  // namespace moe
