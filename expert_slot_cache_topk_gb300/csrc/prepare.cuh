// Router top-k and per-layer slot bookkeeping as device functions, used by
// the prepare kernel (k_route_prepare.cu).
//
// Router: one warp per token; a logit is turned into an order-preserving
// 32-bit key, and each of the k rounds takes two warp max-reductions (largest
// key, then among equal keys the lowest id), so ties go to the lower id
// ("Running 125B MoE on Two 32 GB Cards", section 4.2).
//
// Prepare: one CTA with one thread per expert keeps the whole LRU in shared
// memory.  Distinct experts are found with a shared-memory hit table and ranked
// with warp ballots (five flags in one block scan), so the result equals an
// OrderedDict LRU processed in ascending id order (vLLM PR #37190 "Run MoE
// models exceeding VRAM via expert CPU offloading with GPU cache", "How it
// works"), with hits touched before misses are filled.  Bypass when the
// distinct non-cold experts exceed the slots (llama.cpp discussion #28248
// "RFC: Persistent expert slot pool for MoE CPU offload", "Why not the other
// approaches on the table").  Latency-bound: every global read is issued up
// front and the routed ids stay in shared memory.
#pragma once

#include <climits>
#include <cstdint>

#include "internal.cuh"

namespace moe {
namespace prep {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kMaxRoutedIds = 64 * MOE_MAX_TOPK;   // in-kernel router: T <= 64

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
  return v;
}

// Order-preserving key of a logit: larger logit -> larger key.  NaN ranks as
// -inf, and -0.0 equals +0.0 (they compare equal, so the lower id wins).
__device__ __forceinline__ unsigned logit_key(float v) {
  if (v != v) v = -INFINITY;
  if (v == 0.0f) v = 0.0f;
  const unsigned b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_logit(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-k of one token's logits by one warp.  Lane l holds logits l + 32 i.
// Writes ids / w to global and, when s_ids is given, ids to shared memory.
template <int PL>
__device__ __forceinline__ void route_token(const float* __restrict__ row, int E, int k, int renorm,
                            int32_t* __restrict__ ids, float* __restrict__ w, int32_t* s_ids) {
  const int lane = threadIdx.x & 31;
  unsigned key[PL];
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + 32 * i;
    key[i] = (e < E) ? logit_key(row[e]) : 0u;
  }
  unsigned km = 0;
#pragma unroll
  for (int i = 0; i < PL; ++i) km = key[i] > km ? key[i] : km;
  const float m = key_logit(__reduce_max_sync(kFullMask, km));
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < PL; ++i)
    if (lane + 32 * i < E) s += expf(key_logit(key[i]) - m);
  s = warp_sum_f(s);

  unsigned taken = 0;
  int my_id = 0;
  float my_p = 0.f;
  for (int j = 0; j < k; ++j) {
    unsigned bk = 0, bi = 0;   // best key, and ~id (larger = lower id); 0/0 = none
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      const int e = lane + 32 * i;
      const unsigned ii = ~(unsigned)e;
      if (e < E && !((taken >> i) & 1u) && (key[i] > bk || (key[i] == bk && ii > bi))) {
        bk = key[i];
        bi = ii;
      }
    }
    const unsigned mk = __reduce_max_sync(kFullMask, bk);
    const unsigned mi = __reduce_max_sync(kFullMask, bk == mk ? bi : 0u);
    const int be = (int)~mi;
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) {
      my_id = be;
      my_p = expf(key_logit(mk) - m) / s;
    }
  }
  if (renorm) {
    const float tot = warp_sum_f(lane < k ? my_p : 0.f);
    my_p = my_p / tot;
  }
  if (lane < k) {
    ids[lane] = my_id;
    w[lane] = my_p;
    if (s_ids) s_ids[lane] = my_id;
  }
}

__device__ __forceinline__ void route_dispatch(const float* row, int E, int k, int renorm,
                                               int32_t* ids, float* w, int32_t* s_ids) {
  if (E <= 32) route_token<1>(row, E, k, renorm, ids, w, s_ids);
  else if (E <= 64) route_token<2>(row, E, k, renorm, ids, w, s_ids);
  else if (E <= 128) route_token<4>(row, E, k, renorm, ids, w, s_ids);
  else if (E <= 256) route_token<8>(row, E, k, renorm, ids, w, s_ids);
  else if (E <= 512) route_token<16>(row, E, k, renorm, ids, w, s_ids);
  else route_token<32>(row, E, k, renorm, ids, w, s_ids);
}

// Exclusive block-wide prefix counts of NF flags at once; s_c is [NF][33].
// Every thread of the CTA must call it.  tot[f] gets the block totals.
template <int NF>
__device__ __forceinline__ void block_scan_multi(const int (&flag)[NF], int (&rank)[NF], int (&tot)[NF],
                                                 int (*s_c)[33]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  unsigned b[NF];
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    b[f] = __ballot_sync(kFullMask, flag[f]);
    if (lane == 0) s_c[f][warp] = __popc(b[f]);
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int f = 0; f < NF; ++f) {
      const int v = lane < nw ? s_c[f][lane] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += t;
      }
      s_c[f][lane] = incl - v;
      if (lane == 31) s_c[f][32] = incl;
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    rank[f] = s_c[f][warp] + __popc(b[f] & lt);
    tot[f] = s_c[f][32];
  }
}

// Shared state of one prepare CTA, carved out of dynamic shared memory at
// sizes for this layer (E experts, N slots, n_ids routed ids), so that a small
// layer needs a few KiB and its prepare CTA fits on an SM beside a resident
// expert-MLP CTA.
struct PrepSmem {
  long long* stamp;                  // [N]
  unsigned long long (*red)[32];     // [2][32] block reductions of the move decision
  unsigned long long* stats;         // [ST_COUNT] the layer's counters, read at the start
  int (*c)[33];                      // [5][33] block scan
  int* map;                          // [E] expert -> slot (-1 absent)
  int* rank;                         // [E] rank among the step's non-cold experts
  int* nsel;                         // [E] assignments of each expert in this step
  float* counts;                     // [E] use counts for run-time moves
  int* sexp;                         // [N] slot -> expert (-1 free)
  int* victim;                       // [N]
  int* fstack;                       // [N] free-slot stack (the next miss takes fstack[nfree - 1])
  int* aux;                          // [N] LFU use count, or SLRU segment (1 = protected)
  int* hl;                           // [N] this step's hits, ascending
  int32_t* ids;                      // [n_ids] routed ids (fused router)
  int* bad;                          // an id out of range
  unsigned char* used;               // [N] slot hit in this step
  unsigned char* newf;               // [E] expert copied in this step
  unsigned char* cold;               // [E]
};

// Byte size of the state for (E, N, n_ids); with base != null also points the
// fields of S into base (16-byte aligned).
__host__ __device__ inline size_t prep_smem_layout(int E, int N, int n_ids, unsigned char* base, PrepSmem* S) {
  const size_t e = E > 0 ? (size_t)E : 1, n = N > 0 ? (size_t)N : 1, t = n_ids > 0 ? (size_t)n_ids : 1;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = (o + bytes + 15) / 16 * 16;
    return base ? base + at : nullptr;
  };
  unsigned char* p_stamp = take(n * 8);
  unsigned char* p_red = take(2 * 32 * 8);
  unsigned char* p_stats = take(ST_COUNT * 8);
  unsigned char* p_c = take(5 * 33 * 4);
  unsigned char* p_map = take(e * 4);
  unsigned char* p_rank = take(e * 4);
  unsigned char* p_nsel = take(e * 4);
  unsigned char* p_counts = take(e * 4);
  unsigned char* p_sexp = take(n * 4);
  unsigned char* p_victim = take(n * 4);
  unsigned char* p_fstack = take(n * 4);
  unsigned char* p_aux = take(n * 4);
  unsigned char* p_hl = take(n * 4);
  unsigned char* p_ids = take(t * 4);
  unsigned char* p_bad = take(4);
  unsigned char* p_used = take(n);
  unsigned char* p_newf = take(e);
  unsigned char* p_cold = take(e);
  if (base && S) {
    S->stamp = reinterpret_cast<long long*>(p_stamp);
    S->red = reinterpret_cast<unsigned long long(*)[32]>(p_red);
    S->stats = reinterpret_cast<unsigned long long*>(p_stats);
    S->c = reinterpret_cast<int(*)[33]>(p_c);
    S->map = reinterpret_cast<int*>(p_map);
    S->rank = reinterpret_cast<int*>(p_rank);
    S->nsel = reinterpret_cast<int*>(p_nsel);
    S->counts = reinterpret_cast<float*>(p_counts);
    S->sexp = reinterpret_cast<int*>(p_sexp);
    S->victim = reinterpret_cast<int*>(p_victim);
    S->fstack = reinterpret_cast<int*>(p_fstack);
    S->aux = reinterpret_cast<int*>(p_aux);
    S->hl = reinterpret_cast<int*>(p_hl);
    S->ids = reinterpret_cast<int32_t*>(p_ids);
    S->bad = reinterpret_cast<int*>(p_bad);
    S->used = p_used;
    S->newf = p_newf;
    S->cold = p_cold;
  }
  return o;
}

// Eviction order of an occupied slot (lower = evicted first): recency stamp
// (LRU), insertion stamp (FIFO), (steps used, insertion stamp) (LFU),
// (segment, recency stamp) with the probationary segment first (SLRU).
// Stamps stay below 2^40 (each step advances the clock by at most 2E) and
// LFU counts below 2^24.
__device__ __forceinline__ unsigned long long evict_key(int pol, long long stamp, int aux) {
  const unsigned long long st = (unsigned long long)stamp;
  if (pol == MOE_EVICT_LFU) return ((unsigned long long)(unsigned)aux << 40) | st;
  if (pol == MOE_EVICT_SLRU) return ((unsigned long long)(aux != 0) << 62) | st;
  return st;
}

// Max (is_max) or min of one 64-bit value per thread over the CTA; every
// thread must call it; the result is valid in thread 0.  buf holds 32 words.
__device__ __forceinline__ unsigned long long block_reduce_u64(unsigned long long v, bool is_max,
                                                               unsigned long long* buf) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(kFullMask, v, o);
    v = is_max ? (w > v ? w : v) : (w < v ? w : v);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = (blockDim.x + 31) >> 5;
  __syncthreads();
  if (lane == 0) buf[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < nw ? buf[lane] : (is_max ? 0ull : ~0ull);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long w = __shfl_xor_sync(kFullMask, v, o);
      v = is_max ? (w > v ? w : v) : (w < v ? w : v);
    }
  }
  return v;
}

// One layer step's bookkeeping by the calling CTA (blockDim.x >= E, a multiple
// of 32; do_route needs T <= 64).
__device__ __forceinline__ void prepare_body(const PrepArgs& a, const PrepSmem& S) {
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;   // >= E, a multiple of 32
  const int E = a.E, N = a.N;
  const int n_ids = a.T * a.k;
  const bool ids_in_smem = a.do_route != 0;

  // every global read the step needs, issued before anything waits.  With
  // the fused router the first a.T warps route (their logits loads go out at
  // once) and the threads after them load the slot state, so the two
  // latencies overlap.
  const unsigned long long clk = a.st->clock;
  const int nfree = a.st->nfree;
  const int l0 = (a.do_route && nthr >= 32 * a.T + 32) ? 32 * a.T : 0;   // first state-loading thread
  const bool moving = a.move_interval > 0 && a.counts != nullptr && a.T <= a.move_count_tokens;
  const unsigned counted = moving ? a.st->counted + 1u : 0u;
  for (int q = tid - l0; q >= 0 && q < E; q += nthr - l0) {
    S.map[q] = a.slot_map[q];
    S.cold[q] = a.cold != nullptr ? a.cold[q] : 0;
    S.nsel[q] = 0;
    S.newf[q] = 0;
    if (moving) S.counts[q] = a.counts[q];
  }
  for (int q = tid - l0; q >= 0 && q < N; q += nthr - l0) {
    S.sexp[q] = a.slot_expert[q];
    S.stamp[q] = a.slot_stamp[q];
    S.fstack[q] = a.free_stack[q];
    S.aux[q] = a.slot_aux[q];
    S.used[q] = 0;
  }
  if (tid - l0 >= 0 && tid - l0 < ST_COUNT) S.stats[tid - l0] = a.st->stats[tid - l0];
  if (a.ring_cnt != nullptr)
    for (int q = tid; q < 3 * MOE_MAX_TOPK; q += nthr) a.ring_cnt[q] = 0u;
  if (tid == 0) *S.bad = 0;
  if (a.do_route) {
    for (int t = tid >> 5; t < a.T; t += nthr / 32)
      route_dispatch(a.logits + (size_t)t * E, E, a.k, a.renorm, a.ids + (size_t)t * a.k,
                     a.w_out + (size_t)t * a.k, S.ids + t * a.k);
  }
  __syncthreads();
  for (int i = tid; i < n_ids; i += nthr) {
    const int e = ids_in_smem ? S.ids[i] : a.ids[i];
    if ((unsigned)e >= (unsigned)E) *S.bad = 1;
    else atomicAdd(&S.nsel[e], 1);
  }
  __syncthreads();
  if (*S.bad) {
    // Reject the whole step: state untouched, every assignment skipped.
    if (tid == 0) {
      atomicExch(a.err, DEVERR_BAD_ID);
      RecHdr h = {};
      h.n_ids = n_ids;
      h.seq = a.seq_ctr ? atomicAdd(a.seq_ctr, 1u) + 1u : 0u;
      *a.hdr = h;
    }
    for (int i = tid; i < n_ids; i += nthr) {
      if (a.slot_ids_out) a.slot_ids_out[i] = -1;
      if (a.asg_ptr) a.asg_ptr[i] = 0ull;
      if (a.src_ptr) a.src_ptr[i] = 0ull;
      if (a.pending) a.pending[i] = 0;
    }
    return;
  }

  const int e = tid;
  const int sel = (e < E) ? (S.nsel[e] > 0) : 0;
  const int cold = sel && S.cold[e];
  const int nc = sel && !cold;
  const int hit = nc && S.map[e] >= 0;
  int flag[5] = {nc, cold, sel, hit, nc && !hit};
  int rank[5], tot[5];
  block_scan_multi<5>(flag, rank, tot, S.c);
  const int D = tot[0], C = tot[1], ND = tot[2];
  const bool bypass = D > N;
  if (nc) {
    a.lists[LST_NONCOLD * E + rank[0]] = e;
    S.rank[e] = rank[0];
    if (bypass) S.newf[e] = 1;   // bypass: every non-cold expert is copied to scratch
  }
  if (cold) a.lists[LST_COLD * E + rank[1]] = e;

  int nh = 0, nm = 0, nvict = 0;
  if (!bypass) {
    const int miss = flag[4];
    const int r_h = rank[3], r_m = rank[4];
    nh = tot[3];
    nm = tot[4];
    const int pol = a.policy;
    if (hit) {
      const int hs = S.map[e];
      S.used[hs] = 1;
      if (pol == MOE_EVICT_LRU) S.stamp[hs] = (long long)(clk + (unsigned long long)r_h);   // touch: newest
      else if (pol == MOE_EVICT_LFU) S.aux[hs] += 1;                                        // one more step used
      a.lists[LST_HITS * E + r_h] = e;
      S.hl[r_h] = e;
    }
    nvict = nm > nfree ? nm - nfree : 0;
    __syncthreads();
    if (pol == MOE_EVICT_SLRU && tid < 32 && nh > 0) {
      // warp 0 takes the hits in ascending id order: a probationary expert
      // moves to the protected MRU end, and if that overflows the protected
      // segment (floor(4N/5)), the protected LRU expert moves to the
      // probationary MRU end; a protected expert moves to its MRU end
      const int cap = (4 * N) / 5;
      int np = 0;
      for (int s2 = tid; s2 < N; s2 += 32) np += (S.sexp[s2] >= 0 && S.aux[s2] == 1);
      int nprot = __reduce_add_sync(0xffffffffu, np);
      unsigned long long c2 = clk;
      for (int r = 0; r < nh; ++r) {
        const int hs = S.map[S.hl[r]];
        const bool promote = S.aux[hs] == 0;
        __syncwarp();
        if (tid == 0) {
          S.stamp[hs] = (long long)c2;
          S.aux[hs] = 1;
        }
        ++c2;
        __syncwarp();
        if (promote && ++nprot > cap) {
          unsigned long long lo = ~0ull;   // (stamp << 10 | slot) of the protected LRU expert
          for (int s2 = tid; s2 < N; s2 += 32)
            if (S.sexp[s2] >= 0 && S.aux[s2] == 1) {
              const unsigned long long v = ((unsigned long long)S.stamp[s2] << 10) | (unsigned)s2;
              lo = v < lo ? v : lo;
            }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long u = __shfl_xor_sync(0xffffffffu, lo, o);
            lo = u < lo ? u : lo;
          }
          if (tid == 0) {
            const int ls = (int)(lo & 1023u);
            S.aux[ls] = 0;
            S.stamp[ls] = (long long)c2;
          }
          ++c2;
          --nprot;
          __syncwarp();
        }
      }
    }
    __syncthreads();
    if (nvict > 0 && tid < N && S.sexp[tid] >= 0 && !S.used[tid]) {
      // rank of this slot among the occupied slots not used in this step, by
      // the policy's key (unique): the nvict lowest are the victims
      const unsigned long long my = evict_key(pol, S.stamp[tid], S.aux[tid]);
      int r = 0;
      for (int s2 = 0; s2 < N; ++s2)
        r += (S.sexp[s2] >= 0 && !S.used[s2] && evict_key(pol, S.stamp[s2], S.aux[s2]) < my);
      if (r < nvict) S.victim[r] = tid;
    }
    __syncthreads();
    int slot = -1, ev = -1;
    if (miss) {
      if (r_m < nfree) {
        slot = S.fstack[nfree - 1 - r_m];      // free-slot stack, popped from the end
      } else {
        slot = S.victim[r_m - nfree];          // i-th victim of the policy
        ev = S.sexp[slot];
      }
      a.lists[LST_MISS_E * E + r_m] = e;
      a.lists[LST_MISS_SLOT * E + r_m] = slot;
      a.lists[LST_MISS_EV * E + r_m] = ev;
    }
    __syncthreads();
    if (miss) {
      if (ev >= 0) S.map[ev] = -1;
      S.newf[e] = 1;
      S.map[e] = slot;
      S.sexp[slot] = e;
      S.stamp[slot] = (long long)(clk + (unsigned long long)(2 * nh + r_m));   // insertion: newest
      S.aux[slot] = a.policy == MOE_EVICT_LFU ? 1 : 0;                        // used in one step; probationary
    }
  }
  __syncthreads();
  if (!bypass) {
    if (e < E) a.slot_map[e] = S.map[e];
    if (tid < N) {
      a.slot_expert[tid] = S.sexp[tid];
      a.slot_stamp[tid] = S.stamp[tid];
      a.slot_aux[tid] = S.aux[tid];
    }
  }

  if (tid == 0) {
    LayerState* st = a.st;
    unsigned long long sv[ST_COUNT];
#pragma unroll
    for (int i = 0; i < ST_COUNT; ++i) sv[i] = S.stats[i];
    if (n_ids > 0) sv[ST_STEPS] += 1;
    sv[ST_COLD] += (unsigned long long)C;
    sv[ST_B_COLD] += (unsigned long long)C * a.expert_bytes;
    if (bypass) {
      sv[ST_BYPASS] += 1;
      sv[ST_B_BYPASS] += (unsigned long long)D * a.expert_bytes;
    } else {
      st->clock = clk + (unsigned long long)(2 * nh + nm);
      st->nfree = nfree - (nm < nfree ? nm : nfree);
      sv[ST_HITS] += (unsigned long long)nh;
      sv[ST_MISSES] += (unsigned long long)nm;
      sv[ST_EVICT] += (unsigned long long)nvict;
      sv[ST_B_MISS] += (unsigned long long)nm * a.expert_bytes;
    }
#pragma unroll
    for (int i = 0; i < ST_COUNT; ++i) st->stats[i] = sv[i];
    RecHdr h;
    h.n_ids = n_ids;
    h.bypass = bypass ? 1 : 0;
    h.n_distinct = ND;
    h.n_cold = C;
    h.n_noncold = D;
    h.n_hits = nh;
    h.n_misses = nm;
    h.n_evictions = nvict;
    h.seq = a.seq_ctr ? atomicAdd(a.seq_ctr, 1u) + 1u : 0u;
    *a.hdr = h;
  }

  for (int i = tid; i < n_ids; i += nthr) {
    const int x = ids_in_smem ? S.ids[i] : a.ids[i];
    int v;
    unsigned long long p;
    const unsigned long long host = a.host_base + (unsigned long long)x * a.stride;
    if (S.cold[x]) {
      v = (int)(MOE_SLOT_COLD | (unsigned)x);
      p = host;
    } else if (bypass) {
      const int r = S.rank[x];
      v = (int)(MOE_SLOT_SCRATCH | (unsigned)r);
      p = a.scratch_base + (unsigned long long)r * a.stride;
    } else {
      const int s = S.map[x];
      v = (int)(MOE_SLOT_POOL | (unsigned)s);
      p = a.pool_base + (unsigned long long)s * a.stride;
    }
    if (a.slot_ids_out) a.slot_ids_out[i] = v;
    if (a.asg_ptr) a.asg_ptr[i] = p;
    if (a.src_ptr) a.src_ptr[i] = host;
    if (a.pending) a.pending[i] = S.newf[x];
  }

  // Run-time moves between the cold set and the pool, after the step's own
  // bookkeeping ("Running 125B MoE on Two 32 GB Cards", section 4.4: decayed
  // use counts, the most used host expert and the least used GPU-side expert
  // trade places).  float32 with explicit rounding, as the oracle does.
  if (moving) {
    float cnt = 0.f;
    if (e < E) {
      cnt = S.counts[e];
      if (S.nsel[e] > 0) cnt = __fadd_rn(cnt, (float)S.nsel[e]);
    }
    const bool decide = counted % (unsigned)a.move_interval == 0u;
    if (decide && e < E) cnt = __fmul_rn(cnt, a.move_decay);
    if (e < E) a.counts[e] = cnt;
    if (decide) {
      // counts are >= 0, so their bits order like the values; ties to the lower id
      unsigned long long kc = 0ull, kh = ~0ull;
      if (e < E) {
        const unsigned long long fb = (unsigned long long)__float_as_uint(cnt) << 32;
        if (S.cold[e]) kc = fb | (0xFFFFFFFFull - (unsigned)e);
        else kh = fb | (unsigned)e;
      }
      kc = block_reduce_u64(kc, true, S.red[0]);
      kh = block_reduce_u64(kh, false, S.red[1]);
      if (tid == 0 && kc != 0ull && kh != ~0ull) {
        const int c = (int)(0xFFFFFFFFull - (kc & 0xFFFFFFFFull));
        const int h = (int)(kh & 0xFFFFFFFFull);
        const float fc = __uint_as_float((unsigned)(kc >> 32)), fh = __uint_as_float((unsigned)(kh >> 32));
        if (__fsub_rn(fc, fh) > a.move_threshold) {
          a.cold[c] = 0;
          a.cold[h] = 1;
          const int slot = S.map[h];
          if (slot >= 0) {
            // h leaves the pool: its slot goes on top of the free-slot stack
            const int nf = bypass ? nfree : nfree - (nm < nfree ? nm : nfree);
            a.slot_map[h] = -1;
            a.slot_expert[slot] = -1;
            a.free_stack[nf] = slot;
            a.st->nfree = nf + 1;
          }
          atomicAdd(&a.st->stats[ST_MOVES], 1ull);
        }
      }
    }
    if (tid == 0) a.st->counted = counted;
  }
}


}  // namespace prep
}  // namespace moe
