// Router, prepare, miss/bypass copy and slot verification kernels for
// sm_103a.  The router and the per-layer slot bookkeeping live in
// prepare.cuh.

#include <climits>
#include <cstdint>

#include "internal.cuh"
#include "prepare.cuh"

namespace moe {

namespace {

__global__ void __launch_bounds__(256) k_router(const float* __restrict__ logits, int T, int E,
                                                int k, int renorm, int32_t* __restrict__ ids,
                                                float* __restrict__ w) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  prep::route_dispatch(logits + (size_t)t * E, E, k, renorm, ids + (size_t)t * k, w + (size_t)t * k, nullptr);
}

template <int MAXT>
__global__ void __launch_bounds__(MAXT, 1) k_prepare(PrepArgs a) {
  extern __shared__ __align__(16) unsigned char prep_smem[];
  // Launched early behind the previous kernel of the stream (programmatic
  // dependent launch): wait for it to complete before any global access.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  prep::PrepSmem S;
  prep::prep_smem_layout(a.E, a.N, a.do_route ? a.T * a.k : 0, prep_smem, &S);
  prep::prepare_body(a, S);
}

// Copy the experts of the last prepare (misses -> their slots, or on bypass
// all non-cold experts -> scratch) from the mapped pinned host store.  The
// copy list is read on the device, so no host round trip is needed.
__global__ void __launch_bounds__(kCopyThreads) k_copy(CopyArgs a) {
  const RecHdr h = *a.hdr;
  const int n = h.bypass ? h.n_noncold : h.n_misses;
  if (n == 0) return;
  const int32_t* src_list = a.lists + (h.bypass ? LST_NONCOLD : LST_MISS_E) * a.E;
  const int32_t* slot_list = a.lists + LST_MISS_SLOT * a.E;
  const unsigned long long cpe = (a.nvec + kCopyChunkVec - 1) / kCopyChunkVec;
  const unsigned long long total = (unsigned long long)n * cpe;
  for (unsigned long long c = blockIdx.x; c < total; c += gridDim.x) {
    const int which = (int)(c / cpe);
    const unsigned long long base = (c % cpe) * kCopyChunkVec + threadIdx.x;
    const int e = src_list[which];
    const uint4* src = reinterpret_cast<const uint4*>(a.host_base + (unsigned long long)e * a.stride);
    uint8_t* dst_b = h.bypass ? a.scratch_base + (unsigned long long)which * a.stride
                              : a.pool_base + (unsigned long long)slot_list[which] * a.stride;
    uint4* dst = reinterpret_cast<uint4*>(dst_b);
    uint4 v[kCopyVecPerThread];
#pragma unroll
    for (int u = 0; u < kCopyVecPerThread; ++u) {
      const unsigned long long i = base + (unsigned long long)u * kCopyThreads;
      if (i < a.nvec) v[u] = __ldcs(src + i);
    }
#pragma unroll
    for (int u = 0; u < kCopyVecPerThread; ++u) {
      const unsigned long long i = base + (unsigned long long)u * kCopyThreads;
      if (i < a.nvec) dst[i] = v[u];
    }
  }
}

// Same copies, one whole expert per CTA at a time, in list order (ascending
// expert id); once an expert's bytes are written the CTA publishes
// ready[e] = hdr->seq, so a consumer can start on that expert while later
// ones are still in flight.
__global__ void __launch_bounds__(kCopyThreads) k_copy_flagged(CopyArgs a) {
  const RecHdr h = *a.hdr;
  const int n = h.bypass ? h.n_noncold : h.n_misses;
  const int32_t* src_list = a.lists + (h.bypass ? LST_NONCOLD : LST_MISS_E) * a.E;
  const int32_t* slot_list = a.lists + LST_MISS_SLOT * a.E;
  for (int which = blockIdx.x; which < n; which += gridDim.x) {
    const int e = src_list[which];
    const uint4* src = reinterpret_cast<const uint4*>(a.host_base + (unsigned long long)e * a.stride);
    uint8_t* dst_b = h.bypass ? a.scratch_base + (unsigned long long)which * a.stride
                              : a.pool_base + (unsigned long long)slot_list[which] * a.stride;
    uint4* dst = reinterpret_cast<uint4*>(dst_b);
    for (unsigned long long base = threadIdx.x; base < a.nvec; base += (unsigned long long)kCopyChunkVec) {
      uint4 v[kCopyVecPerThread];
#pragma unroll
      for (int u = 0; u < kCopyVecPerThread; ++u) {
        const unsigned long long i = base + (unsigned long long)u * kCopyThreads;
        if (i < a.nvec) v[u] = __ldcs(src + i);
      }
#pragma unroll
      for (int u = 0; u < kCopyVecPerThread; ++u) {
        const unsigned long long i = base + (unsigned long long)u * kCopyThreads;
        if (i < a.nvec) dst[i] = v[u];
      }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a.ready + e), "r"(h.seq) : "memory");
    }
  }
}

// Plain copy of nvec 16-byte vectors (used to time the UVA path at create).
__global__ void __launch_bounds__(kCopyThreads) k_copy_raw(const uint4* __restrict__ src,
                                                           uint4* __restrict__ dst,
                                                           unsigned long long nvec) {
  const unsigned long long chunks = (nvec + kCopyChunkVec - 1) / kCopyChunkVec;
  for (unsigned long long c = blockIdx.x; c < chunks; c += gridDim.x) {
    const unsigned long long base = c * kCopyChunkVec + threadIdx.x;
    uint4 v[kCopyVecPerThread];
#pragma unroll
    for (int u = 0; u < kCopyVecPerThread; ++u) {
      const unsigned long long i = base + (unsigned long long)u * kCopyThreads;
      if (i < nvec) v[u] = __ldcs(src + i);
    }
#pragma unroll
    for (int u = 0; u < kCopyVecPerThread; ++u) {
      const unsigned long long i = base + (unsigned long long)u * kCopyThreads;
      if (i < nvec) dst[i] = v[u];
    }
  }
}

// One CTA per slot: does the slot hold exactly its expert's backing bytes?
__global__ void __launch_bounds__(256) k_verify(const int32_t* __restrict__ slot_expert,
                                                const uint8_t* __restrict__ pool_base,
                                                const uint8_t* __restrict__ host_base,
                                                unsigned long long stride, unsigned long long nvec,
                                                int* __restrict__ mismatches) {
  const int s = blockIdx.x;
  const int e = slot_expert[s];
  if (e < 0) return;
  const uint4* a = reinterpret_cast<const uint4*>(pool_base + (unsigned long long)s * stride);
  const uint4* b = reinterpret_cast<const uint4*>(host_base + (unsigned long long)e * stride);
  int bad = 0;
  for (unsigned long long i = threadIdx.x; i < nvec; i += blockDim.x) {
    const uint4 x = a[i], y = __ldcs(b + i);
    bad |= (x.x != y.x) | (x.y != y.y) | (x.z != y.z) | (x.w != y.w);
  }
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0 && bad) atomicAdd(mismatches, 1);
}

}  // namespace

cudaError_t launch_router(const float* logits, int T, int E, int k, int renorm, int32_t* ids,
                          float* w, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  k_router<<<(T + 7) / 8, 256, 0, s>>>(logits, T, E, k, renorm, ids, w);
  return cudaGetLastError();
}

cudaError_t launch_prepare(const PrepArgs& a, cudaStream_t s) {
  // one thread per expert for the ranking scans, one warp per token for the
  // fused router, plus (when it fits) E more threads so that the slot state
  // is loaded by threads that do not route
  int need = a.E > 32 * a.T ? a.E : 32 * a.T;
  if (a.do_route && a.E + 32 * a.T <= kPrepThreads && a.E + 32 * a.T > need) need = a.E + 32 * a.T;
  if (need > kPrepThreads) need = kPrepThreads;
  const int threads = (need + 31) / 32 * 32;
  if (a.do_route && a.T * a.k > prep::kMaxRoutedIds) return cudaErrorInvalidValue;
  const size_t smem = prep::prep_smem_layout(a.E, a.N, a.do_route ? a.T * a.k : 0, nullptr, nullptr);
  // programmatic dependent launch: the CTA may be scheduled while the previous
  // kernel (which triggers early) still runs, and waits for it on the device
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (threads <= 256) return cudaLaunchKernelEx(&cfg, k_prepare<256>, a);
  return cudaLaunchKernelEx(&cfg, k_prepare<kPrepThreads>, a);
}

// Every kernel of a layer step prefers the largest shared-memory carve-out,
// so that consecutive launches (one-CTA prepare, then an expert-MLP kernel
// with up to 227 KiB of shared memory per CTA) never make an SM switch its
// L1 / shared-memory split in between.
cudaError_t prepare_configure() {
  const void* kernels[] = {(const void*)k_router, (const void*)k_prepare<256>, (const void*)k_prepare<kPrepThreads>,
                           (const void*)k_copy, (const void*)k_copy_flagged};
  for (const void* k : kernels) {
    const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                               (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  for (const void* k : {(const void*)k_prepare<256>, (const void*)k_prepare<kPrepThreads>}) {
    const cudaError_t e = cudaFuncSetAttribute(
        k, cudaFuncAttributeMaxDynamicSharedMemorySize,
        (int)prep::prep_smem_layout(MOE_MAX_EXPERTS, MOE_MAX_EXPERTS, prep::kMaxRoutedIds, nullptr, nullptr));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_copy(const CopyArgs& a, int grid, cudaStream_t s) {
  k_copy<<<grid, kCopyThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_copy_flagged(const CopyArgs& a, int grid, cudaStream_t s) {
  k_copy_flagged<<<grid, kCopyThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_copy_raw(const void* src, void* dst, unsigned long long nvec, int grid,
                            cudaStream_t s) {
  k_copy_raw<<<grid, kCopyThreads, 0, s>>>(reinterpret_cast<const uint4*>(src),
                                           reinterpret_cast<uint4*>(dst), nvec);
  return cudaGetLastError();
}

cudaError_t launch_verify(const int32_t* slot_expert, int N, const uint8_t* pool_base,
                          const uint8_t* host_base, unsigned long long stride,
                          unsigned long long nvec, int* mismatches, cudaStream_t s) {
  if (N <= 0) return cudaSuccess;
  k_verify<<<N, 256, 0, s>>>(slot_expert, pool_base, host_base, stride, nvec, mismatches);
  return cudaGetLastError();
}

}  // namespace moe
