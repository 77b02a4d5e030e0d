// moe_expert_mlp_noalloc: the grouped expert MLP for callers that cannot
// allocate device memory.
//
// The regular entry point takes the gate/up intermediate h (T*k*I floats)
// from a buffer the caller allocates.  Some callers have no way to do that at
// the point of the call: plugins hosted by a framework whose caching
// allocator owns every byte of device memory, and latency-critical loops that
// must never hit cudaMalloc's implicit device synchronisation.  This variant
// keeps its scratch in a fixed-size array compiled into the library instead,
// so a call allocates nothing.
//
// Costs and rules for users:
//  * The array (MOE_NOALLOC_MAX_SCRATCH_FLOATS floats, 2 MiB) exists on every
//    GPU that loads the library and stays there until the process exits.
//  * Every call on a device shares the one array.  Two calls whose kernels
//    overlap on the GPU (different streams, no ordering between them) race on
//    it and may produce wrong results; order them on one stream or with events.
//  * The array keeps the last call's contents.  Nothing in it needs to start
//    at zero: the up kernel writes every h element the down kernel reads
//    (skipped assignments get explicit zeros).
//  * The first call on a device looks up the array's device address with
//    cudaGetSymbolAddress (a one-time set-up per device, done with that device
//    current).  Make that first call before any stream capture.
//
// Shape checks, the expert block layout and the kernels are the ones
// moe_expert_mlp uses (block_layout / chunk_elems / mlp_args), so both entry
// points accept the same shapes and give the same bits.

#include <cuda_runtime.h>

#include <mutex>

#include "internal.cuh"

using namespace moe;

namespace {

static __device__ __align__(256) float g_mlp_scratch[MOE_NOALLOC_MAX_SCRATCH_FLOATS];

std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_mlp_scratch on the current device.  In host code the
// symbol name itself is only a host-side stand-in, so it must never be passed
// to a kernel; the address comes from cudaGetSymbolAddress, once per device.
cudaError_t scratch_on_current_device(float** out) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_mlp_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" moe_status moe_expert_mlp_noalloc(int wdtype, int hidden, int inter, int top_k,
                                             const void* x_d, const uint64_t* block_ptrs_d,
                                             const float* w_d, int T, void* y_d, int flags,
                                             moe_stream_t stream) {
  size_t w13 = 0, w2 = 0, s13 = 0, s2 = 0;
  if (!block_layout(wdtype, hidden, inter, &w13, &w2, &s13, &s2) || hidden <= 0 || inter <= 0 ||
      hidden % chunk_elems(wdtype) || inter % chunk_elems(wdtype))
    return set_global_error(MOE_EINVAL, "moe_expert_mlp_noalloc: bad weight format or shape");
  if (top_k < 1 || top_k > MOE_MAX_TOPK || T < 0 || (long long)T * top_k > 65535)
    return set_global_error(MOE_EINVAL, "moe_expert_mlp_noalloc: bad top_k or T");
  if (mlp_up_smem_bytes(hidden) > 200 * 1024 || mlp_down_smem_bytes(top_k, inter) > 200 * 1024)
    return set_global_error(MOE_EINVAL, "moe_expert_mlp_noalloc: shape exceeds shared-memory staging limits");
  if ((long long)T * top_k * inter > MOE_NOALLOC_MAX_SCRATCH_FLOATS)
    return set_global_error(MOE_EINVAL,
                            "moe_expert_mlp_noalloc: T * top_k * inter exceeds the built-in scratch of "
                            "MOE_NOALLOC_MAX_SCRATCH_FLOATS (524288) floats; use moe_expert_mlp with a "
                            "caller-provided scratch buffer");
  if (flags & ~MOE_FWD_RESIDUAL) return set_global_error(MOE_EINVAL, "moe_expert_mlp_noalloc: unknown flags");
  if (T == 0) return MOE_OK;
  if (!x_d || !block_ptrs_d || !w_d || !y_d || x_d == y_d)
    return set_global_error(MOE_EINVAL, "moe_expert_mlp_noalloc: null or aliased buffer");

  float* h = nullptr;
  cudaError_t e = scratch_on_current_device(&h);
  if (e != cudaSuccess) return set_global_error(MOE_ECUDA, cudaGetErrorString(e));
  e = mlp_configure(wdtype, hidden, inter, top_k);
  if (e != cudaSuccess) return set_global_error(MOE_ECUDA, cudaGetErrorString(e));

  const MlpArgs a = mlp_args(wdtype, hidden, inter, top_k, x_d,
                             reinterpret_cast<const unsigned long long*>(block_ptrs_d), w_d, h, y_d, T,
                             flags);
  const cudaStream_t s = (cudaStream_t)stream;
  e = launch_mlp_up(wdtype, a, s);
  if (e == cudaSuccess) e = launch_mlp_down(wdtype, a, s);
  if (e != cudaSuccess) return set_global_error(MOE_ECUDA, cudaGetErrorString(e));
  return MOE_OK;
}
