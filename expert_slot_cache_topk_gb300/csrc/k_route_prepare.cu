// Router top-k, per-layer slot bookkeeping + remap, miss/bypass copy and
// slot verification kernels for sm_103a.
//
// Router: one warp per token (ids by logit, ties -> lower id: "Running 125B
// MoE on Two 32 GB Cards", section 4.2).  Prepare: one 1024-thread CTA per
// layer step keeps the whole LRU in shared memory; distinct experts are found
// with a shared-memory hit table and ranked with warp ballots, so the result
// equals an OrderedDict LRU processed in ascending id order (vLLM PR #37190
// "Run MoE models exceeding VRAM via expert CPU offloading with GPU cache",
// "How it works"), with hits touched before misses are filled.  Bypass when the
// distinct non-cold experts exceed the slots (llama.cpp discussion #28248
// "RFC: Persistent expert slot pool for MoE CPU offload", "Why not the other
// approaches on the table").

#include <climits>
#include <cstdint>

#include "internal.cuh"

namespace moe {

namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// (v, e) beats (bv, be) when v is larger, or equal with the lower id.
__device__ __forceinline__ bool beats(float v, int e, float bv, int be) {
  return v > bv || (v == bv && e < be);
}

// Top-k of one token's logits by one warp.  Lane l holds logits l + 32 i.
template <int PL>
__device__ void route_token(const float* __restrict__ row, int E, int k, int renorm,
                            int32_t* __restrict__ ids, float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  float v[PL];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + 32 * i;
    float x = (e < E) ? row[e] : -INFINITY;
    if (x != x) x = -INFINITY;   // NaN ranks below every number
    v[i] = x;
    m = fmaxf(m, x);
  }
  m = warp_max(m);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < PL; ++i)
    if (lane + 32 * i < E) s += expf(v[i] - m);
  s = warp_sum(s);

  unsigned taken = 0;
  int my_id = 0;
  float my_p = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = INT_MAX;
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && beats(v[i], e, bv, be)) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, o);
      const int oe = __shfl_xor_sync(kFull, be, o);
      if (beats(ov, oe, bv, be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) {
      my_id = be;
      my_p = expf(bv - m) / s;
    }
  }
  if (renorm) {
    const float tot = warp_sum(lane < k ? my_p : 0.f);
    my_p = my_p / tot;
  }
  if (lane < k) {
    ids[lane] = my_id;
    w[lane] = my_p;
  }
}

__device__ __forceinline__ void route_dispatch(const float* row, int E, int k, int renorm,
                                               int32_t* ids, float* w) {
  if (E <= 32) route_token<1>(row, E, k, renorm, ids, w);
  else if (E <= 64) route_token<2>(row, E, k, renorm, ids, w);
  else if (E <= 128) route_token<4>(row, E, k, renorm, ids, w);
  else if (E <= 256) route_token<8>(row, E, k, renorm, ids, w);
  else if (E <= 512) route_token<16>(row, E, k, renorm, ids, w);
  else route_token<32>(row, E, k, renorm, ids, w);
}

__global__ void __launch_bounds__(256) k_router(const float* __restrict__ logits, int T, int E,
                                                int k, int renorm, int32_t* __restrict__ ids,
                                                float* __restrict__ w) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  route_dispatch(logits + (size_t)t * E, E, k, renorm, ids + (size_t)t * k, w + (size_t)t * k);
}

// Exclusive block-wide prefix count of `flag`; *total gets the block sum.
// Every thread of the CTA must call it.
__device__ __forceinline__ int block_scan_excl(int flag, int* total, int* s_w) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const unsigned b = __ballot_sync(kFull, flag);
  const int r = __popc(b & ((1u << lane) - 1u));
  __syncthreads();
  if (lane == 0) s_w[warp] = __popc(b);
  __syncthreads();
  if (warp == 0) {
    const int v = lane < nw ? s_w[lane] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    s_w[lane] = incl - v;
    if (lane == 31) s_w[32] = incl;
  }
  __syncthreads();
  *total = s_w[32];
  return s_w[warp] + r;
}

__global__ void __launch_bounds__(kPrepThreads, 1) k_prepare(PrepArgs a) {
  __shared__ int s_w[33];
  __shared__ int s_map[MOE_MAX_EXPERTS];      // expert -> slot (-1 absent)
  __shared__ int s_rank[MOE_MAX_EXPERTS];     // rank among the step's non-cold experts
  __shared__ int s_sexp[MOE_MAX_EXPERTS];     // slot -> expert (-1 free)
  __shared__ long long s_stamp[MOE_MAX_EXPERTS];
  __shared__ int s_victim[MOE_MAX_EXPERTS];
  __shared__ unsigned char s_mark[MOE_MAX_EXPERTS];
  __shared__ unsigned char s_new[MOE_MAX_EXPERTS];  // expert copied in this step
  __shared__ int s_bad;

  const int tid = threadIdx.x;
  const int E = a.E, N = a.N;
  const int n_ids = a.T * a.k;

  const int nthr = blockDim.x;   // >= E, a multiple of 32
  if (a.do_route) {
    for (int t = tid >> 5; t < a.T; t += nthr / 32)
      route_dispatch(a.logits + (size_t)t * E, E, a.k, a.renorm, a.ids + (size_t)t * a.k,
                     a.w_out + (size_t)t * a.k);
  }
  const unsigned long long clk = a.st->clock;
  const int nfree = a.st->nfree;
  if (tid == 0) s_bad = 0;
  if (tid < E) {
    s_mark[tid] = 0;
    s_new[tid] = 0;
    s_map[tid] = a.slot_map[tid];
  }
  if (tid < N) {
    s_sexp[tid] = a.slot_expert[tid];
    s_stamp[tid] = a.slot_stamp[tid];
  }
  __syncthreads();   // also orders the fused router's ids before they are read
  for (int i = tid; i < n_ids; i += nthr) {
    const int e = a.ids[i];
    if ((unsigned)e >= (unsigned)E) s_bad = 1;
    else s_mark[e] = 1;
  }
  __syncthreads();
  if (s_bad) {
    // Reject the whole step: state untouched, every assignment skipped.
    if (tid == 0) {
      atomicExch(a.err, DEVERR_BAD_ID);
      RecHdr h = {};
      h.n_ids = n_ids;
      *a.hdr = h;
    }
    for (int i = tid; i < n_ids; i += nthr) {
      if (a.slot_ids_out) a.slot_ids_out[i] = -1;
      if (a.asg_ptr) a.asg_ptr[i] = 0ull;
      if (a.pending) a.pending[i] = 0;
    }
    return;
  }

  const int e = tid;
  const int sel = (e < E) ? s_mark[e] : 0;
  const int cold = sel && a.cold != nullptr && a.cold[e] != 0;
  const int nc = sel && !cold;
  int D, C, ND;
  const int r_nc = block_scan_excl(nc, &D, s_w);
  const int r_c = block_scan_excl(cold, &C, s_w);
  block_scan_excl(sel, &ND, s_w);
  if (nc) {
    a.lists[LST_NONCOLD * E + r_nc] = e;
    s_rank[e] = r_nc;
    if (D > N) s_new[e] = 1;   // bypass: every non-cold expert is copied to scratch
  }
  if (cold) a.lists[LST_COLD * E + r_c] = e;

  const bool bypass = D > N;
  int nh = 0, nm = 0, nvict = 0;
  if (!bypass) {
    const int hit = nc && s_map[e] >= 0;
    const int miss = nc && !hit;
    const int r_h = block_scan_excl(hit, &nh, s_w);
    const int r_m = block_scan_excl(miss, &nm, s_w);
    if (hit) {
      s_stamp[s_map[e]] = (long long)(clk + (unsigned long long)r_h);   // touch: newest stamps
      a.lists[LST_HITS * E + r_h] = e;
    }
    nvict = nm > nfree ? nm - nfree : 0;
    __syncthreads();
    if (nvict > 0 && tid < N && s_sexp[tid] >= 0) {
      // rank of this slot by recency among occupied slots (stamps are unique);
      // hits were just stamped newest, so the nvict oldest are not in this step
      const long long my = s_stamp[tid];
      int r = 0;
      for (int s2 = 0; s2 < N; ++s2) r += (s_sexp[s2] >= 0 && s_stamp[s2] < my);
      if (r < nvict) s_victim[r] = tid;
    }
    __syncthreads();
    int slot = -1, ev = -1;
    if (miss) {
      if (r_m < nfree) {
        slot = nfree - 1 - r_m;                // free list [0, nfree), popped from the end
      } else {
        slot = s_victim[r_m - nfree];          // i-th least recently used slot
        ev = s_sexp[slot];
      }
      a.lists[LST_MISS_E * E + r_m] = e;
      a.lists[LST_MISS_SLOT * E + r_m] = slot;
      a.lists[LST_MISS_EV * E + r_m] = ev;
    }
    __syncthreads();
    if (miss) {
      if (ev >= 0) s_map[ev] = -1;
      s_new[e] = 1;
      s_map[e] = slot;
      s_sexp[slot] = e;
      s_stamp[slot] = (long long)(clk + (unsigned long long)(nh + r_m));
    }
    __syncthreads();
    if (e < E) a.slot_map[e] = s_map[e];
    if (tid < N) {
      a.slot_expert[tid] = s_sexp[tid];
      a.slot_stamp[tid] = s_stamp[tid];
    }
  }
  __syncthreads();

  if (tid == 0) {
    LayerState* st = a.st;
    if (n_ids > 0) st->stats[ST_STEPS] += 1;
    st->stats[ST_COLD] += (unsigned long long)C;
    st->stats[ST_B_COLD] += (unsigned long long)C * a.expert_bytes;
    if (bypass) {
      st->stats[ST_BYPASS] += 1;
      st->stats[ST_B_BYPASS] += (unsigned long long)D * a.expert_bytes;
    } else {
      st->clock = clk + (unsigned long long)(nh + nm);
      st->nfree = nfree - (nm < nfree ? nm : nfree);
      st->stats[ST_HITS] += (unsigned long long)nh;
      st->stats[ST_MISSES] += (unsigned long long)nm;
      st->stats[ST_EVICT] += (unsigned long long)nvict;
      st->stats[ST_B_MISS] += (unsigned long long)nm * a.expert_bytes;
    }
    RecHdr h;
    h.n_ids = n_ids;
    h.bypass = bypass ? 1 : 0;
    h.n_distinct = ND;
    h.n_cold = C;
    h.n_noncold = D;
    h.n_hits = nh;
    h.n_misses = nm;
    h.n_evictions = nvict;
    *a.hdr = h;
  }

  for (int i = tid; i < n_ids; i += nthr) {
    const int x = a.ids[i];
    int v;
    unsigned long long p;
    if (a.cold != nullptr && a.cold[x]) {
      v = (int)(MOE_SLOT_COLD | (unsigned)x);
      p = a.host_base + (unsigned long long)x * a.stride;
    } else if (bypass) {
      const int r = s_rank[x];
      v = (int)(MOE_SLOT_SCRATCH | (unsigned)r);
      p = a.scratch_base + (unsigned long long)r * a.stride;
    } else {
      const int s = s_map[x];
      v = (int)(MOE_SLOT_POOL | (unsigned)s);
      p = a.pool_base + (unsigned long long)s * a.stride;
    }
    if (a.slot_ids_out) a.slot_ids_out[i] = v;
    if (a.asg_ptr) a.asg_ptr[i] = p;
    if (a.pending) a.pending[i] = s_new[x];
  }
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
  // fused router (at most 32 warps)
  int need = a.E > 32 * a.T ? a.E : 32 * a.T;
  if (need > kPrepThreads) need = kPrepThreads;
  const int threads = (need + 31) / 32 * 32;
  k_prepare<<<1, threads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_copy(const CopyArgs& a, int grid, cudaStream_t s) {
  k_copy<<<grid, kCopyThreads, 0, s>>>(a);
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
