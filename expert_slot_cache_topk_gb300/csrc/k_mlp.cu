// Grouped expert MLP for small token counts (decode): HBM-bound GEMV.
//
// For every assignment a = t*k + j the expert block pointer asg_ptr[a] points
// at the canonical block [w13 | w2 | s13 | s2] of expert ids[t, j] -- in its
// pool slot, in bypass scratch, or in mapped pinned host memory (cold set) --
// so the kernels never see where an expert lives (vLLM PR #37190 "Run MoE
// models exceeding VRAM via expert CPU offloading with GPU cache", "How it
// works": fused_experts on slot buffers with remapped ids; "Running 125B MoE
// on Two 32 GB Cards", section 2: the GPU reads host rows through a UVA view).
//
//   up   : h[a, i] = w[a] * silu(Wg_e[i] . x_t) * (Wu_e[i] . x_t)   (w13 rows i, I+i)
//   down : y[t, n] = sum over the k experts of W2_e[n] . h[t*k + j]
//
// The router weight is folded into h, so the down pass is one dot product per
// output row over the k experts' concatenated W2 rows -- every lane of a warp
// has work even when a single expert row is short (INT4 I = 640: 20 chunks).
//
// Layout of the work: one 16-warp CTA per SM (persistent), the grid split into
// G CTAs per token; a CTA owns a contiguous share of the token's tasks (gate/up
// row pairs, or output rows), so there is no wave tail.  Weights stream once
// from HBM in 16-byte vectors; each warp's first loads are issued before x (or
// h) is staged in shared memory so the staging latency hides under them.  The
// staged activations are f32 and every lane reuses one staged chunk for all
// rows it owns.  INT4 codes become exact (code - 8) floats by integer bit
// arithmetic and are scaled once per 32-element chunk.  Each output comes from
// one warp's fixed reduction tree, so the result does not depend on where the
// expert's bytes live (pool, scratch, host): cached, bypass and cold paths are
// bitwise identical.

#include <cuda_bf16.h>
#include <cstdint>

#include "internal.cuh"

namespace moe {

namespace {

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

template <int F>
__device__ __forceinline__ size_t row_bytes(int K) {
  return F == MOE_F32 ? (size_t)K * 4 : (F == MOE_BF16 ? (size_t)K * 2 : (size_t)K / 2);
}

__device__ __forceinline__ float bf16_bits(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

template <int F>
__device__ __forceinline__ void stage_f32(float* dst, const void* src, size_t off, int n) {
  if (F == MOE_F32) {
    const float* s = reinterpret_cast<const float*>(src) + off;
    for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = s[i];
  } else {
    const uint16_t* s = reinterpret_cast<const uint16_t*>(src) + off;
    for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = bf16_bits(s[i]);
  }
}

// position of the (s+1)-th set bit of m
__device__ __forceinline__ int nth_set_bit(unsigned m, int s) {
  for (int i = 0; i < s; ++i) m &= m - 1u;
  return __ffs(m) - 1;
}

// ---------------------------------------------------------------- up (w13)
// grid (G, T).  Tasks of token t: (selected assignment, group of RP gate/up
// row pairs); CTA b of G owns tasks [b*n/G, (b+1)*n/G); warps stride them.
template <int F, int RP, int U>
__global__ void __launch_bounds__(kMlpThreads, 1) k_up(MlpArgs a) {
  extern __shared__ __align__(16) float xs[];
  constexpr int EL = FmtT<F>::kElems;
  constexpr int R = 2 * RP;
  const int H = a.H, I = a.I, k = a.k;
  const int t = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  bool mine = lane < k;
  if (mine && a.pending != nullptr) mine = a.pending[(size_t)t * k + lane] == a.phase;
  const unsigned sel = __ballot_sync(kFull, mine);
  const int P = (I + RP - 1) / RP;
  const int ntask = __popc(sel) * P;
  const int t_beg = (int)((long long)ntask * blockIdx.x / gridDim.x);
  const int t_end = (int)((long long)ntask * (blockIdx.x + 1) / gridDim.x);
  const int C = H / EL;
  const size_t rb = row_bytes<F>(H);
  const int G = H / 128;

  uint4 wv[R][U];
  float sc[R][U];
  const uint4* rp[R];
  int ri[R];
  bool rv[R];
  int asg = 0, p0 = 0;
  const uint16_t* sb = nullptr;
  unsigned long long base = 0;

  auto setup = [&](int task) {
    const int s = task / P;
    p0 = (task - s * P) * RP;
    asg = t * k + nth_set_bit(sel, s);
    base = a.asg_ptr[asg];
    const uint8_t* wb = reinterpret_cast<const uint8_t*>(base);
    sb = reinterpret_cast<const uint16_t*>(wb + a.off_s13);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int p = p0 + (r % RP);
      rv[r] = base != 0ull && p < I;
      ri[r] = (r < RP) ? p : I + p;
      rp[r] = reinterpret_cast<const uint4*>(wb + (size_t)ri[r] * rb);
    }
  };
  auto load = [&](int cbase) {   // chunks cbase + lane + 32 u (cbase is warp-uniform)
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = cbase + lane + 32 * u;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (rv[r] && c < C) {
          wv[r][u] = ldw(rp[r] + c);
          if (F == MOE_INT4_G128) sc[r][u] = bf16_bits(sb[(size_t)ri[r] * G + (c >> 2)]);
        } else {
          wv[r][u] = make_uint4(0u, 0u, 0u, 0u);
          sc[r][u] = 0.f;
        }
      }
    }
  };

  int task = t_beg + warp;
  bool have = task < t_end;
  if (have) {
    setup(task);
    load(0);
  }
  stage_f32<F>(xs, a.x, (size_t)t * H, H);
  __syncthreads();

  while (have) {
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.f;
    for (int cbase = 0;;) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = cbase + lane + 32 * u;
        if (c < C) {
          const float* xc = xs + c * EL;
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float d = chunk_dot<F>(wv[r][u], xc);
            acc[r] = (F == MOE_INT4_G128) ? fmaf(d, sc[r][u], acc[r]) : acc[r] + d;
          }
        }
      }
      cbase += 32 * U;
      if (cbase >= C) break;
      load(cbase);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = warp_sum(acc[r]);
    if (lane == 0) {
      const float wa = base != 0ull ? a.w[asg] : 0.f;
      float* hrow = a.h + (size_t)asg * I;
#pragma unroll
      for (int p = 0; p < RP; ++p) {
        if (p0 + p < I) {
          const float g = acc[p], u = acc[RP + p];
          hrow[p0 + p] = base != 0ull ? wa * (g / (1.0f + expf(-g)) * u) : 0.f;
        }
      }
    }
    task += kWarps;
    have = task < t_end;
    if (have) {
      setup(task);
      load(0);
    }
  }
}

// -------------------------------------------------------------- down (w2)
// grid (G, T).  CTA b of G owns output rows [b*H/G, (b+1)*H/G) of token t;
// each warp computes whole rows, one chunk q of the concatenated k*C chunks
// per lane and step: expert j = q / C, chunk c = q % C.
template <int F, int U>
__global__ void __launch_bounds__(kMlpThreads, 1) k_down(MlpArgs a) {
  extern __shared__ __align__(16) float hs[];
  constexpr int EL = FmtT<F>::kElems;
  const int H = a.H, I = a.I, k = a.k;
  const int t = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_beg = (int)((long long)H * blockIdx.x / gridDim.x);
  const int n_end = (int)((long long)H * (blockIdx.x + 1) / gridDim.x);
  const int C = I / EL;
  const int Q = k * C;
  const size_t rb = row_bytes<F>(I);
  const int G = I / 128;
  // lane j keeps expert j's block pointer; others fetch it by shuffle
  const unsigned long long my_base = lane < k ? a.asg_ptr[(size_t)t * k + lane] : 0ull;

  uint4 wv[U];
  float sc[U];
  auto load = [&](int n, int qbase) {   // chunks qbase + lane + 32 u (qbase is warp-uniform)
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = qbase + lane + 32 * u;
      const int j = q / C;
      const unsigned long long base = __shfl_sync(kFull, my_base, q < Q ? j : 0);
      if (q < Q && base != 0ull) {
        const int c = q - j * C;
        const uint8_t* wb = reinterpret_cast<const uint8_t*>(base);
        wv[u] = ldw(reinterpret_cast<const uint4*>(wb + a.off_w2 + (size_t)n * rb) + c);
        if (F == MOE_INT4_G128)
          sc[u] = bf16_bits(reinterpret_cast<const uint16_t*>(wb + a.off_s2)[(size_t)n * G + (c >> 2)]);
      } else {
        wv[u] = make_uint4(0u, 0u, 0u, 0u);
        sc[u] = 0.f;
      }
    }
  };

  int n = n_beg + warp;
  if (n < n_end) load(n, 0);
  for (int i = threadIdx.x; i < k * I; i += blockDim.x) hs[i] = a.h[(size_t)t * k * I + i];
  __syncthreads();

  for (; n < n_end; n += kWarps) {
    float acc = 0.f;
    for (int qbase = 0;;) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int q = qbase + lane + 32 * u;
        if (q < Q) {
          const float d = chunk_dot<F>(wv[u], hs + (size_t)q * EL);
          acc = (F == MOE_INT4_G128) ? fmaf(d, sc[u], acc) : acc + d;
        }
      }
      qbase += 32 * U;
      if (qbase >= Q) break;
      load(n, qbase);
    }
    acc = warp_sum(acc);
    if (n + kWarps < n_end) load(n + kWarps, 0);
    if (lane == 0) {
      const size_t o = (size_t)t * H + n;
      if (F == MOE_F32) {
        if (a.residual) acc += reinterpret_cast<const float*>(a.x)[o];
        reinterpret_cast<float*>(a.y)[o] = acc;
      } else {
        if (a.residual) acc += bf16_bits(reinterpret_cast<const uint16_t*>(a.x)[o]);
        reinterpret_cast<__nv_bfloat16*>(a.y)[o] = __float2bfloat16_rn(acc);
      }
    }
  }
}

template <int F>
struct Tiles;
template <>
struct Tiles<MOE_F32> {
  static constexpr int RP = 1, UU = 2, UD = 2;
};
template <>
struct Tiles<MOE_BF16> {
  static constexpr int RP = 1, UU = 8, UD = 16;
};
template <>
struct Tiles<MOE_INT4_G128> {
  static constexpr int RP = 2, UU = 3, UD = 7;
};

// Opt a kernel into more than 48 KiB of dynamic shared memory once per size,
// so launches (also inside stream capture) do not repeat the attribute call.
template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes, size_t* configured) {
  if (bytes <= *configured) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) *configured = bytes;
  return e;
}

template <int F>
struct Configured {
  static size_t up, down;
};
template <int F>
size_t Configured<F>::up = 48 * 1024;
template <int F>
size_t Configured<F>::down = 48 * 1024;

constexpr int kMaxDev = 64;
int g_sms[kMaxDev];

// CTAs per token: one 16-warp CTA per SM across the whole grid.
int ctas_per_token(int T) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) dev = 0;
  if (g_sms[dev] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = v > 0 ? v : 1;
  }
  const int g = g_sms[dev] / (T > 0 ? T : 1);
  return g > 1 ? g : 1;
}

template <int F>
cudaError_t configure_impl(int H, int I, int k) {
  cudaError_t e = allow_smem(k_up<F, Tiles<F>::RP, Tiles<F>::UU>, mlp_up_smem_bytes(H), &Configured<F>::up);
  if (e != cudaSuccess) return e;
  ctas_per_token(1);
  return allow_smem(k_down<F, Tiles<F>::UD>, mlp_down_smem_bytes(k, I), &Configured<F>::down);
}

template <int F>
cudaError_t up_impl(const MlpArgs& a, cudaStream_t s) {
  const size_t smem = mlp_up_smem_bytes(a.H);
  auto kern = k_up<F, Tiles<F>::RP, Tiles<F>::UU>;
  cudaError_t e = allow_smem(kern, smem, &Configured<F>::up);
  if (e != cudaSuccess) return e;
  dim3 grid(ctas_per_token(a.T), a.T);
  kern<<<grid, kMlpThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int F>
cudaError_t down_impl(const MlpArgs& a, cudaStream_t s) {
  const size_t smem = mlp_down_smem_bytes(a.k, a.I);
  auto kern = k_down<F, Tiles<F>::UD>;
  cudaError_t e = allow_smem(kern, smem, &Configured<F>::down);
  if (e != cudaSuccess) return e;
  dim3 grid(ctas_per_token(a.T), a.T);
  kern<<<grid, kMlpThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t mlp_up_smem_bytes(int H) { return (size_t)H * sizeof(float); }
size_t mlp_down_smem_bytes(int k, int I) { return (size_t)k * I * sizeof(float); }

cudaError_t mlp_configure(int wdtype, int H, int I, int k) {
  switch (wdtype) {
    case MOE_F32: return configure_impl<MOE_F32>(H, I, k);
    case MOE_BF16: return configure_impl<MOE_BF16>(H, I, k);
    case MOE_INT4_G128: return configure_impl<MOE_INT4_G128>(H, I, k);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_mlp_up(int wdtype, const MlpArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  switch (wdtype) {
    case MOE_F32: return up_impl<MOE_F32>(a, s);
    case MOE_BF16: return up_impl<MOE_BF16>(a, s);
    case MOE_INT4_G128: return up_impl<MOE_INT4_G128>(a, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_mlp_down(int wdtype, const MlpArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  switch (wdtype) {
    case MOE_F32: return down_impl<MOE_F32>(a, s);
    case MOE_BF16: return down_impl<MOE_BF16>(a, s);
    case MOE_INT4_G128: return down_impl<MOE_INT4_G128>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
