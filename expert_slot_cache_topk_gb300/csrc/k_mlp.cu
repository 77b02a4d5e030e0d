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
// Layout of the work: two 16-warp CTAs per SM (persistent), the grid split into
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
#include "mlp_common.cuh"

namespace moe {

namespace {

using namespace mlp;

// ------------------------------------------------------ per-warp task state
// Every kernel that produces y uses these two helpers, so the per-lane
// accumulation order (chunk c = lane + 32 m, m increasing) and the warp
// reduction tree are the same whichever kernel runs: the fused per-layer
// kernel and the standalone up/down kernels give bitwise identical outputs.

// Up task: gate rows [p0, p0 + RP) and up rows [I + p0, I + p0 + RP) of one
// assignment; writes h = w * silu(gate . x) * (up . x).
template <int F, int RP, int U>
struct UpWarp {
  static constexpr int R = 2 * RP;
  static constexpr int EL = FmtT<F>::kElems;
  uint4 wv[R][U];
  float sc[R][U];
  const uint4* rp[R];
  long long delta;       // read-through: slot address minus host address of the block
  int ri[R];
  bool rv[R];
  bool copy;
  const uint16_t* sb;
  unsigned long long base;
  int asg, p0;
  float fsg, fsu, fsd;   // FP8: gate, up and down tensor scales

  // task = (pair group, selected assignment), pair-major so that a contiguous
  // task range touches every selected expert
  __device__ __forceinline__ void setup(const MlpArgs& a, int t, unsigned sel, int nsel, int task) {
    const int g = task / nsel;
    p0 = g * RP;
    asg = t * a.k + nth_set_bit(sel, task - g * nsel);
    base = a.asg_ptr[asg];
    copy = a.readthrough && a.pending[asg] != 0 && base != 0ull;
    const unsigned long long src = copy ? a.src_ptr[asg] : base;
    const uint8_t* wb = reinterpret_cast<const uint8_t*>(src);
    delta = (long long)(base - src);
    sb = reinterpret_cast<const uint16_t*>(wb + a.off_s13);
    if (F == MOE_FP8_E4M3 && base != 0ull) {
      const float* f13 = reinterpret_cast<const float*>(wb + a.off_s13);
      fsg = __ldcg(f13);
      fsu = __ldcg(f13 + 1);
      fsd = __ldcg(reinterpret_cast<const float*>(wb + a.off_s2));
    }
    const size_t rb = row_bytes<F>(a.H);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int p = p0 + (r % RP);
      rv[r] = base != 0ull && p < a.I;
      ri[r] = (r < RP) ? p : a.I + p;
      rp[r] = reinterpret_cast<const uint4*>(wb + (size_t)ri[r] * rb);
    }
  }
  // chunks cbase + lane + 32 u; cbase is warp-uniform
  __device__ __forceinline__ void load(const MlpArgs& a, int cbase, int lane) {
    const int C = a.H / EL;
    const int G = a.H / 128;
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
  }
  // consume the loaded batch (and further batches), reduce, write h
  __device__ __forceinline__ void finish(const MlpArgs& a, const float* __restrict__ xs, int lane) {
    const int C = a.H / EL;
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
            if (copy && rv[r])
              reinterpret_cast<uint4*>(reinterpret_cast<uintptr_t>(rp[r] + c) + delta)[0] = wv[r][u];
            const float d = chunk_dot<F>(wv[r][u], xc);
            acc[r] = (F == MOE_INT4_G128) ? fmaf(d, sc[r][u], acc[r]) : acc[r] + d;
          }
        }
      }
      cbase += 32 * U;
      if (cbase >= C) break;
      load(a, cbase, lane);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = warp_sum(acc[r]);
    if (lane == 0) {
      const float wa = base != 0ull ? a.w[asg] : 0.f;
      float* hrow = a.h + (size_t)asg * a.I;
#pragma unroll
      for (int p = 0; p < RP; ++p) {
        if (p0 + p < a.I) {
          float g = acc[p], u = acc[RP + p];
          if (F == MOE_FP8_E4M3) {
            // per-tensor scales: gate and up on their dot products; the down
            // scale folded into h (the down pass mixes experts in one dot)
            g *= fsg;
            u *= fsu;
          }
          float hv = base != 0ull ? wa * (g / (1.0f + expf(-g)) * u) : 0.f;
          if (F == MOE_FP8_E4M3) hv *= fsd;
          hrow[p0 + p] = hv;
        }
      }
    }
  }
};

// Down task: half `part` of output row n of token t -- chunks
// [part * Qh, min(Q, (part + 1) * Qh)) of the k experts' concatenated W2 rows
// (Q = k * C, Qh = ceil(Q / 2)); chunk q is expert j = q / C, column chunk
// q % C.  y[t, n] = half 0 + half 1 (+ residual).
template <int F, int U>
struct DownWarp {
  static constexpr int EL = FmtT<F>::kElems;
  uint4 wv[U];
  float sc[U];
  unsigned long long my_base;   // lane j holds expert j's block pointer
  int n, q_beg, q_end;

  __device__ __forceinline__ void bases(const MlpArgs& a, int t, int lane) {
    my_base = lane < a.k ? a.asg_ptr[(size_t)t * a.k + lane] : 0ull;
  }
  __device__ __forceinline__ void setup(const MlpArgs& a, int row, int part) {
    const int Q = a.k * (a.I / EL);
    const int Qh = (Q + 1) >> 1;
    n = row;
    q_beg = part * Qh;
    q_end = part ? Q : Qh;
  }
  __device__ __forceinline__ void load(const MlpArgs& a, int qbase, int lane) {
    const int C = a.I / EL;
    const int G = a.I / 128;
    const size_t rb = row_bytes<F>(a.I);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = q_beg + qbase + lane + 32 * u;
      const int j = q / C;
      const unsigned long long b = __shfl_sync(kFull, my_base, q < q_end ? j : 0);
      if (q < q_end && b != 0ull) {
        const int c = q - j * C;
        const uint8_t* wb = reinterpret_cast<const uint8_t*>(b);
        wv[u] = __ldcg(reinterpret_cast<const uint4*>(wb + a.off_w2 + (size_t)n * rb) + c);
        if (F == MOE_INT4_G128)
          sc[u] = bf16_bits(__ldcg(reinterpret_cast<const unsigned short*>(wb + a.off_s2) + (size_t)n * G + (c >> 2)));
      } else {
        wv[u] = make_uint4(0u, 0u, 0u, 0u);
        sc[u] = 0.f;
      }
    }
  }
  // returns the half-row dot product (same value in every lane)
  __device__ __forceinline__ float finish(const MlpArgs& a, const float* __restrict__ hs, int lane) {
    float acc = 0.f;
    const int len = q_end - q_beg;
    for (int qbase = 0;;) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int q = q_beg + qbase + lane + 32 * u;
        if (q < q_end) {
          const float d = chunk_dot<F>(wv[u], hs + (size_t)q * EL);
          acc = (F == MOE_INT4_G128) ? fmaf(d, sc[u], acc) : acc + d;
        }
      }
      qbase += 32 * U;
      if (qbase >= len) break;
      load(a, qbase, lane);
    }
    return warp_sum(acc);
  }
};


__device__ __forceinline__ unsigned select_assignments(const MlpArgs& a, int t, int lane) {
  bool mine = lane < a.k;
  if (mine && a.pending != nullptr && a.phase >= 0) mine = a.pending[(size_t)t * a.k + lane] == a.phase;
  return __ballot_sync(kFull, mine);
}

// Down rounds of one token's row range [n_beg, n_end): 16 (row, half) tasks
// per round, one per warp; halves combined in a fixed order through smem.
// The first round's loads may already be in flight (prefetched = true).
template <int F, int U>
__device__ __forceinline__ void down_rounds(const MlpArgs& a, int t, int n_beg, int n_end,
                                            const float* hs, float* s_part, DownWarp<F, U>& dw,
                                            bool prefetched) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntask = 2 * (n_end - n_beg);
  for (int r0 = 0; r0 < ntask; r0 += kWarps) {
    const int task = r0 + warp;
    if (task < ntask) {
      if (!(prefetched && r0 == 0)) {
        dw.setup(a, n_beg + (task >> 1), task & 1);
        dw.load(a, 0, lane);
      }
      const float v = dw.finish(a, hs, lane);
      if (lane == 0) s_part[warp] = v;
    }
    __syncthreads();
    if (threadIdx.x < kWarps / 2 && r0 + 2 * (int)threadIdx.x < ntask) {
      const int i = threadIdx.x;
      store_y<F>(a, t, n_beg + (r0 >> 1) + i, s_part[2 * i] + s_part[2 * i + 1]);
    }
    __syncthreads();
  }
}

// ------------------------------------------------ standalone up / down kernels
// grid (G, T).  Up: CTA b of G owns tasks [b*n/G, (b+1)*n/G) of token t, a
// task being (selected assignment, group of RP row pairs).  Down: CTA b owns
// output rows [b*H/G, (b+1)*H/G) of token t.
template <int F, int RP, int U>
__global__ void __launch_bounds__(kMlpThreads, 2) k_up(MlpArgs a) {
  extern __shared__ __align__(16) float xs[];
  const int t = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned sel = select_assignments(a, t, lane);
  const int P = (a.I + RP - 1) / RP;
  const int nsel = __popc(sel);
  const int ntask = nsel * P;
  const int t_beg = (int)((long long)ntask * blockIdx.x / gridDim.x);
  const int t_end = (int)((long long)ntask * (blockIdx.x + 1) / gridDim.x);
  UpWarp<F, RP, U> uw;
  int task = t_beg + warp;
  if (task < t_end) {
    uw.setup(a, t, sel, nsel, task);
    uw.load(a, 0, lane);       // in flight while x is staged
  }
  stage_x<F>(xs, a, t, threadIdx.x, blockDim.x);
  __syncthreads();
  while (task < t_end) {
    uw.finish(a, xs, lane);
    task += kWarps;
    if (task < t_end) {
      uw.setup(a, t, sel, nsel, task);
      uw.load(a, 0, lane);
    }
  }
}

template <int F, int U>
__global__ void __launch_bounds__(kMlpThreads, 2) k_down(MlpArgs a) {
  extern __shared__ __align__(16) float hs[];
  __shared__ float s_part[kWarps];
  const int t = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_beg = (int)((long long)a.H * blockIdx.x / gridDim.x);
  const int n_end = (int)((long long)a.H * (blockIdx.x + 1) / gridDim.x);
  DownWarp<F, U> dw;
  dw.bases(a, t, lane);
  const bool pre = warp < 2 * (n_end - n_beg);
  if (pre) {
    dw.setup(a, n_beg + (warp >> 1), warp & 1);
    dw.load(a, 0, lane);
  }
  stage_h(hs, a, t, threadIdx.x, blockDim.x);
  __syncthreads();
  down_rounds<F, U>(a, t, n_beg, n_end, hs, s_part, dw, true);
}

// --------------------------------------------------- fused per-layer kernel
// Cooperative launch, every CTA resident.  Work unit u = blockIdx.x < T * Gt
// is (token u / Gt, slice u % Gt).  Phase 1 computes h for the unit's share of
// the token's up tasks; each warp then issues its first W2 loads, all CTAs meet
// at a grid barrier (bounded wait), and phase 2 computes the unit's share of
// the token's output rows.
__device__ __forceinline__ void grid_barrier(GridBar* bar, int* err) {
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile unsigned* vgen = &bar->gen;
    const unsigned gen = *vgen;
    __threadfence();
    const unsigned arrived = atomicAdd(&bar->count, 1u);
    if (arrived == gridDim.x - 1) {
      atomicExch(&bar->count, 0u);
      __threadfence();
      atomicAdd(&bar->gen, 1u);
    } else {
      unsigned it = 0;
      while (*vgen == gen) {
        if (++it > (1u << 24)) {        // ~seconds: give up, flag it, never hang
          atomicExch(err, DEVERR_BARRIER);
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
  }
  __syncthreads();
}

template <int F, int RP, int UU, int UD>
__global__ void __launch_bounds__(kMlpThreads, 2) k_mlp_fused(MlpArgs a, GridBar* bar, int* err) {
  extern __shared__ __align__(16) float sm[];
  __shared__ float s_part[kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Gt = gridDim.x / a.T;
  const int unit = blockIdx.x;
  const bool active = unit < a.T * Gt;
  const int t = active ? unit / Gt : 0;
  const int slice = active ? unit % Gt : 0;

  // pending experts of this token (read-through only)
  unsigned pend = 0;
  if (a.readthrough) pend = __ballot_sync(kFull, lane < a.k && a.pending[(size_t)t * a.k + lane] != 0 &&
                                                     a.asg_ptr[(size_t)t * a.k + lane] != 0ull);
  // phase 1: up (and, with read-through, copies of the pending experts' w2 /
  // scale bytes into their slots, 4 KiB per task, this CTA's share of them)
  if (active) {
    const unsigned sel = select_assignments(a, t, lane);
    const int P = (a.I + RP - 1) / RP;
    const int nsel = __popc(sel);
    const int ntask = nsel * P;
    const int t_beg = (int)((long long)ntask * slice / Gt);
    const int t_end = (int)((long long)ntask * (slice + 1) / Gt);
    UpWarp<F, RP, UU> uw;
    int task = t_beg + warp;
    if (pend == 0u && task < t_end) {
      uw.setup(a, t, sel, nsel, task);
      uw.load(a, 0, lane);            // in flight while x is staged
    }
    stage_x<F>(sm, a, t, threadIdx.x, blockDim.x);
    __syncthreads();
    if (pend) {
      const unsigned long long cpe = (a.tail_bytes + 4095ull) / 4096ull;
      const unsigned long long ncopy = (unsigned long long)__popc(pend) * cpe;
      const unsigned long long c_beg = ncopy * slice / Gt, c_end = ncopy * (slice + 1) / Gt;
      for (unsigned long long c = c_beg + warp; c < c_end; c += kWarps) {
        const int s = (int)(c / cpe);
        const unsigned long long off = a.tail_off + (c - (unsigned long long)s * cpe) * 4096ull;
        const int asg = t * a.k + nth_set_bit(pend, s);
        const uint4* src = reinterpret_cast<const uint4*>(a.src_ptr[asg] + off);
        uint4* dst = reinterpret_cast<uint4*>(a.asg_ptr[asg] + off);
        const unsigned long long nv = (a.tail_off + a.tail_bytes - off) / 16ull;
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const unsigned i = lane + 32u * u;
          if (i < nv) v[u] = __ldcs(src + i);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const unsigned i = lane + 32u * u;
          if (i < nv) dst[i] = v[u];
        }
      }
      if (task < t_end) {
        uw.setup(a, t, sel, nsel, task);
        uw.load(a, 0, lane);
      }
    }
    while (task < t_end) {
      uw.finish(a, sm, lane);
      task += kWarps;
      if (task < t_end) {
        uw.setup(a, t, sel, nsel, task);
        uw.load(a, 0, lane);
      }
    }
  }
  // first W2 loads go out before the barrier -- unless some of them are still
  // being copied into their slots by other CTAs
  const int n_beg = (int)((long long)a.H * slice / Gt);
  const int n_end = active ? (int)((long long)a.H * (slice + 1) / Gt) : n_beg;
  const bool prefetch = pend == 0u;
  DownWarp<F, UD> dw;
  dw.bases(a, t, lane);
  if (prefetch && warp < 2 * (n_end - n_beg)) {
    dw.setup(a, n_beg + (warp >> 1), warp & 1);
    dw.load(a, 0, lane);
  }
  __threadfence();
  grid_barrier(bar, err);
  if (!active) return;
  // phase 2: down
  stage_h(sm, a, t, threadIdx.x, blockDim.x);
  __syncthreads();
  down_rounds<F, UD>(a, t, n_beg, n_end, sm, s_part, dw, prefetch);
}

template <int F>
struct Tiles;
template <>
struct Tiles<MOE_F32> {
  static constexpr int RP = 1, UU = 2, UD = 2;
};
template <>
struct Tiles<MOE_BF16> {
  static constexpr int RP = 1, UU = 4, UD = 8;
};
template <>
struct Tiles<MOE_INT4_G128> {
  static constexpr int RP = 2, UU = 1, UD = 4;
};
template <>
struct Tiles<MOE_FP8_E4M3> {
  static constexpr int RP = 1, UU = 4, UD = 8;
};

// Opt a kernel into more than 48 KiB of dynamic shared memory once per size
// and device, so launches (also inside stream capture) do not repeat the
// attribute call.  Callers hold launch_state_mutex().
template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes, size_t* configured) {
  if (bytes <= *configured) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) *configured = bytes;
  return e;
}

// What has been configured for one weight format on one device.
struct MlpLaunchState {
  size_t up = 48 * 1024, down = 48 * 1024, fused = 48 * 1024;   // shared memory the attributes allow
  int fused_blocks_per_sm = 0;                                   // occupancy of the fused kernel ...
  size_t fused_blocks_smem = 0;                                  // ... at this shared-memory size
};
MlpLaunchState g_mlp_state[4][kMaxDevices];   // [weight format][device]

template <int F>
MlpLaunchState* mlp_state() {
  const int dev = current_device();
  return dev < 0 ? nullptr : &g_mlp_state[F][dev];
}

// CTAs per token for the standalone kernels: two 16-warp CTAs per SM overall.
int ctas_per_token(int T) {
  const int g = 2 * device_sm_count() / (T > 0 ? T : 1);
  return g > 1 ? g : 1;
}

template <int F>
size_t fused_smem(int H, int I, int k) {
  const size_t a = mlp_up_smem_bytes(H), b = mlp_down_smem_bytes(k, I);
  return a > b ? a : b;
}

template <int F>
cudaError_t configure_impl(int H, int I, int k) {
  device_sm_count();   // cache the SM count outside any capture
  std::lock_guard<std::mutex> lock(launch_state_mutex());
  MlpLaunchState* st = mlp_state<F>();
  if (!st) return cudaErrorInvalidDevice;
  cudaError_t e = allow_smem(k_up<F, Tiles<F>::RP, Tiles<F>::UU>, mlp_up_smem_bytes(H), &st->up);
  if (e != cudaSuccess) return e;
  e = allow_smem(k_down<F, Tiles<F>::UD>, mlp_down_smem_bytes(k, I), &st->down);
  if (e != cudaSuccess) return e;
  auto fk = k_mlp_fused<F, Tiles<F>::RP, Tiles<F>::UU, Tiles<F>::UD>;
  const size_t fs = fused_smem<F>(H, I, k);
  e = allow_smem(fk, fs, &st->fused);
  if (e != cudaSuccess) return e;
  if (st->fused_blocks_smem != fs) {
    int nb = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fk, kMlpThreads, fs);
    if (e != cudaSuccess) return e;
    st->fused_blocks_per_sm = nb;
    st->fused_blocks_smem = fs;
  }
  return cudaSuccess;
}

template <int F>
cudaError_t up_impl(const MlpArgs& a, cudaStream_t s) {
  const size_t smem = mlp_up_smem_bytes(a.H);
  auto kern = k_up<F, Tiles<F>::RP, Tiles<F>::UU>;
  {
    std::lock_guard<std::mutex> lock(launch_state_mutex());
    MlpLaunchState* st = mlp_state<F>();
    if (!st) return cudaErrorInvalidDevice;
    cudaError_t e = allow_smem(kern, smem, &st->up);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(ctas_per_token(a.T), a.T);
  kern<<<grid, kMlpThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int F>
cudaError_t down_impl(const MlpArgs& a, cudaStream_t s) {
  const size_t smem = mlp_down_smem_bytes(a.k, a.I);
  auto kern = k_down<F, Tiles<F>::UD>;
  {
    std::lock_guard<std::mutex> lock(launch_state_mutex());
    MlpLaunchState* st = mlp_state<F>();
    if (!st) return cudaErrorInvalidDevice;
    cudaError_t e = allow_smem(kern, smem, &st->down);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(ctas_per_token(a.T), a.T);
  kern<<<grid, kMlpThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int F>
cudaError_t fused_impl(const MlpArgs& a, GridBar* bar, int* err, cudaStream_t s) {
  const size_t smem = fused_smem<F>(a.H, a.I, a.k);
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(launch_state_mutex());
    const MlpLaunchState* st = mlp_state<F>();
    if (!st || st->fused_blocks_smem != smem || st->fused_blocks_per_sm < 1)
      return cudaErrorNotSupported;    // not configured for this shape: caller falls back
    per_sm = st->fused_blocks_per_sm;
  }
  const int grid = per_sm * device_sm_count();
  if (a.T > grid) return cudaErrorNotSupported;
  auto kern = k_mlp_fused<F, Tiles<F>::RP, Tiles<F>::UU, Tiles<F>::UD>;
  MlpArgs args = a;
  void* params[] = {&args, &bar, &err};
  const cudaError_t e = cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(kMlpThreads),
                                                    params, smem, s);
  return e;
}

}  // namespace

size_t mlp_up_smem_bytes(int H) { return (size_t)H * sizeof(float); }
size_t mlp_down_smem_bytes(int k, int I) { return (size_t)k * I * sizeof(float); }

cudaError_t mlp_configure(int wdtype, int H, int I, int k) {
  switch (wdtype) {
    case MOE_F32: return configure_impl<MOE_F32>(H, I, k);
    case MOE_BF16: return configure_impl<MOE_BF16>(H, I, k);
    case MOE_INT4_G128: return configure_impl<MOE_INT4_G128>(H, I, k);
    case MOE_FP8_E4M3: return configure_impl<MOE_FP8_E4M3>(H, I, k);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_mlp_up(int wdtype, const MlpArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  switch (wdtype) {
    case MOE_F32: return up_impl<MOE_F32>(a, s);
    case MOE_BF16: return up_impl<MOE_BF16>(a, s);
    case MOE_INT4_G128: return up_impl<MOE_INT4_G128>(a, s);
    case MOE_FP8_E4M3: return up_impl<MOE_FP8_E4M3>(a, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_mlp_fused(int wdtype, const MlpArgs& a, GridBar* bar, int* err, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  switch (wdtype) {
    case MOE_F32: return fused_impl<MOE_F32>(a, bar, err, s);
    case MOE_BF16: return fused_impl<MOE_BF16>(a, bar, err, s);
    case MOE_INT4_G128: return fused_impl<MOE_INT4_G128>(a, bar, err, s);
    case MOE_FP8_E4M3: return fused_impl<MOE_FP8_E4M3>(a, bar, err, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_mlp_down(int wdtype, const MlpArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  switch (wdtype) {
    case MOE_F32: return down_impl<MOE_F32>(a, s);
    case MOE_BF16: return down_impl<MOE_BF16>(a, s);
    case MOE_INT4_G128: return down_impl<MOE_INT4_G128>(a, s);
    case MOE_FP8_E4M3: return down_impl<MOE_FP8_E4M3>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
