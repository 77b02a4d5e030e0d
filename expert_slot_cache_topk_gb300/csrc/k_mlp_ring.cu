// One-token (decode) expert MLP with the weight bytes staged in shared memory.
//
// Same arithmetic as k_mlp.cu -- up: h[j, i] = w_j * silu(Wg_j[i] . x) *
// (Wu_j[i] . x); down: y[n] = sum over the k experts' concatenated W2 rows
// n . h -- but organised for a batch-1 step, where every weight byte is used
// once and the step is a stream of k * B_e bytes out of HBM (vLLM PR #37190
// "Run MoE models exceeding VRAM via expert CPU offloading with GPU cache",
// "How it works": the experts run on slot buffers through remapped ids).
//
// One persistent CTA per SM, cooperative launch, ten warps:
//   * warp 0 (producer) walks this CTA's share of the work -- first its run
//     of gate/up row pairs (expert-major), then its output rows -- and for
//     every stage issues cp.async.bulk copies of the weight rows that live in
//     HBM into a ring of shared-memory stages, signalled by mbarriers;
//   * warps 1..8 (consumers) take every stage in order: up stages produce h,
//     then all CTAs meet at a grid barrier (h complete), then down stages
//     produce y.  The producer never waits for the grid barrier, so W2 rows
//     keep streaming into the ring while the grid synchronises;
//   * warp 9 (copier) moves the blocks of experts missed in this step from
//     pinned host memory into their slots ("Running 125B MoE on Two 32 GB
//     Cards", section 2: the GPU reads host rows through a UVA view), in
//     chunks spread over the grid, counting landed chunks per expert.  The
//     producer takes a missed expert's items last and issues their bulk
//     copies (from the slot) once the chunks they need are counted, so the
//     host-link transfer overlaps the HBM-resident experts' work.
// Rows of blocks that stay in mapped host memory (cold experts) are not
// bulk-copied: the consumers read them with plain 16-byte loads.
//
// The consumer warps keep the token's activations in registers (x in the up
// phase, one part of h in the down phase; see RingTile), so shared memory
// carries only weight bytes.  Each output is reduced in a fixed order that
// does not depend on where an expert's bytes live, so pool, scratch and host
// homes give bitwise identical y; the order differs from k_mlp.cu's, so the
// two kernels agree to rounding, not bitwise.
//
// Ring protocol: stage s of the ring holds work item i with i % NS == s.
// full[s] completes once per item (producer arrive + the bulk bytes),
// empty[s] once per item (one arrive per consumer warp).  Every consumer warp
// takes every item in order, so no waiter is ever more than one phase ahead
// of a barrier.  Waits are bounded by the global timer; a wait that runs out
// sets DEVERR_RING and the CTA stops, after the producer has waited (bounded)
// for its own copies in flight.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "internal.cuh"
#include "mlp_common.cuh"

namespace moe {

namespace {

using namespace mlp;

constexpr int kConsumers = 8;                       // consumer warps
constexpr int kRingThreads = 32 * (2 + kConsumers);  // producer, consumers, copier
constexpr int kCopierWarp = 1 + kConsumers;
constexpr unsigned long long kCopyChunk = 16384;    // copier: bytes per counted chunk
constexpr int kCopyBatch = 16;                      // copier: 16-byte loads per lane in flight
constexpr int kMaxStages = 12;
constexpr int kMaxRows = 64;                        // output rows per CTA whose residual is kept in shared memory
constexpr int kHRep = 8;                            // copies of h in global memory (read spread over L2)
constexpr int kParts = 4;                           // parts per output row in the down phase
static_assert(kParts == 4, "down_store sums four parts");
constexpr int kRowsPerPass = kConsumers / kParts;   // output rows the consumer warps take at once
constexpr unsigned long long kWaitNs = 500000000ull;  // 0.5 s
constexpr size_t kSmemLimit = 227 * 1024;

enum { SRC_RING = 0, SRC_PLAIN = 1, SRC_NONE = 2 };

struct RingDesc {
  int kind;        // 0 = up, 1 = down
  int asg;         // up: assignment index
  int p0;          // up: first row pair; down: first output row
  int n;           // up: pairs; down: rows
  unsigned src;    // up: SRC_*; down: bit j set = expert j not in the ring
};

struct RingShared {
  unsigned long long full[kMaxStages];
  unsigned long long empty[kMaxStages];
  RingDesc desc[kMaxStages];
  unsigned long long base[MOE_MAX_TOPK];   // block pointer of each assignment
  float wt[MOE_MAX_TOPK];                  // router weight of each assignment
  float xres[kMaxRows];                    // residual x of this CTA's output rows
  float part[kMaxRows * kParts];           // down: the part sums of each of the CTA's rows
  float gu[kMaxStages][kConsumers / 2][2]; // up, half-size items: gate / up sums of each pair
  int cnt[kMaxStages][kConsumers / 2];     // up, half-size items: rows of the pair finished
  int stop;                                // set when a wait ran out: skip the rest
  int jorder[MOE_MAX_TOPK];                // producer: assignments in item order (pending ones last)
  float fsc[MOE_MAX_TOPK][3];              // FP8: gate, up and down tensor scales of each assignment
};

struct RingCfg {
  int up_pairs;           // row pairs per up item: 2 * kConsumers (INT4, FP8), kConsumers or kConsumers / 2
  int nstages;            // ring stages
  unsigned stage_bytes;   // bytes per stage (multiple of 128)
  int down_rows;          // output rows per down item (<= kConsumers)
  int down_group;         // CTA row ranges start at multiples of this (8 for INT4 scale rows)
};

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// true if the phase with this parity has completed; if not, the thread is
// suspended in hardware (not spinning) until it completes or a system time
// limit (a few microseconds) passes
__device__ __forceinline__ bool mbar_try(uint32_t bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// true once the phase with this parity has completed; false after kWaitNs
// (the clock is read only when the first try finds the phase still open)
__device__ __forceinline__ bool mbar_wait(uint32_t bar, unsigned parity) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (mbar_try(bar, parity)) return true;
    if (global_ns() - t0 > kWaitNs) return false;
  }
}
// bytes (multiple of 16) from global src (16-byte aligned) to shared dst
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, unsigned bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(__cvta_generic_to_global(src)), "r"(bytes), "r"(bar)
      : "memory");
}
// the same, with an L2 eviction-priority policy for the source lines
__device__ __forceinline__ void bulk_copy_hint(uint32_t dst, const void* src, unsigned bytes, uint32_t bar,
                                               unsigned long long policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(__cvta_generic_to_global(src)), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
// weight rows read once per launch go first when L2 needs room
__device__ __forceinline__ unsigned long long evict_first_policy() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// bytes (multiple of 16) from global src (16-byte aligned) into L2, no wait
__device__ __forceinline__ void prefetch_l2(const void* src, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(__cvta_generic_to_global(src)), "r"(bytes)
               : "memory");
}
// true once *p >= target (acquire); false after kWaitNs
__device__ __forceinline__ bool wait_count(const unsigned* p, unsigned target) {
  unsigned long long t0 = 0ull;
  for (unsigned it = 0;; ++it) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= target) return true;
    if (it == 0) t0 = global_ns();
    else if (global_ns() - t0 > kWaitNs) return false;
    __nanosleep(100);
  }
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers) : "memory");
}

__device__ __forceinline__ bool in_host(const MlpArgs& a, unsigned long long p) {
  return p >= a.host_lo && p < a.host_hi;
}

// Grid barrier among the consumer warps of every CTA (the producer warps do
// not take part).  The CTA's writes are ordered before its arrival by the CTA
// barrier plus one thread's release add (release is cumulative); that thread
// polls the arrival count with acquire loads until every CTA of this launch
// has arrived -- one atomic per CTA, no reset.  Bounded: gives up after ~1 s
// and flags DEVERR_BARRIER.
__device__ __forceinline__ void consumer_grid_barrier(GridBar* bar, int* err, int ctid) {
  consumer_sync();
  if (ctid == 0) {
    const unsigned long long G = gridDim.x;
    unsigned long long old;
    asm volatile("atom.release.gpu.global.add.u64 %0, [%1], 1;" : "=l"(old) : "l"(&bar->arrivals) : "memory");
    const unsigned long long target = (old / G + 1ull) * G;
    const unsigned long long t0 = global_ns();
    for (unsigned it = 0;; ++it) {
      unsigned long long v;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(&bar->arrivals) : "memory");
      if (v >= target) break;
      if ((it & 255u) == 255u && global_ns() - t0 > 1000000000ull) {
        atomicExch(err, DEVERR_BARRIER);
        break;
      }
    }
  }
  consumer_sync();
}

// 16 bytes of data written by other CTAs in this launch (after a grid
// barrier): read at L2, never from this SM's L1
__device__ __forceinline__ float4 ld_l2_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// x[0, n] as f32, and y[0, n] = v (bf16 unless F is f32)
template <int F>
__device__ __forceinline__ float x_at(const MlpArgs& a, int n) {
  return F == MOE_F32 ? reinterpret_cast<const float*>(a.x)[n] : bf16_bits(reinterpret_cast<const uint16_t*>(a.x)[n]);
}
template <int F>
__device__ __forceinline__ void store_out(const MlpArgs& a, int n, float v) {
  if (F == MOE_F32) reinterpret_cast<float*>(a.y)[n] = v;
  else reinterpret_cast<__nv_bfloat16*>(a.y)[n] = __float2bfloat16_rn(v);
}

// ------------------------------------------------------------- consumers
// Per-format register tiling of the consumer warps.  Lane l owns the 16-byte
// chunks c = l + 32 m (m < XM) of every w13 row and keeps the matching x
// values in registers for the whole up phase.  In the down phase every
// output row is cut into kParts parts of Qp = ceil(Q / kParts) chunks of the
// k experts' concatenated W2 rows (Q chunks); warp w owns part w % kParts of
// its rows -- chunks q = part * Qp + l + 32 m (m < HM) -- and keeps those h
// values in registers.  Shared memory then only carries the weight bytes.
template <int F>
struct RingTile;
template <>
struct RingTile<MOE_F32> {
  static constexpr int XM = 8, HM = 8;
};
template <>
struct RingTile<MOE_BF16> {
  static constexpr int XM = 8, HM = 8;
};
template <>
struct RingTile<MOE_INT4_G128> {
  static constexpr int XM = 3, HM = 2;
};
template <>
struct RingTile<MOE_FP8_E4M3> {
  static constexpr int XM = 4, HM = 4;
};

// ---- activations in registers
// bf16 / f32 / FP8: a chunk's EL activations as f32.  INT4: a chunk of 32
// activations as 16-bit integers at a power-of-two scale (Q4Act below), so that
// a 16-byte chunk of packed codes is dotted in exact integer arithmetic.
template <int EL>
struct FAct {
  float v[EL];
};

// INT4 activation chunk.  With s chosen so that the chunk's largest magnitude
// times 2^s lies in [2^13, 2^14): even elements X = rint(x 2^s) (|X| <= 2^14),
// odd elements Y = rint(x 2^(s-4)) (|Y| <= 2^10), i.e. the odd element's
// integer is 16 Y.  A 32-bit weight word holds the codes of elements 8k .. 8k+7,
// byte i = q[2i] + 16 q[2i+1] (low nibble = even column).  dp2a (two 16-bit x
// 8-bit products per instruction) of the raw bytes with (Y_{2i+1}) pairs gives
// Y q_even + 16 Y q_odd, and of the even codes (word & 0x0F0F0F0F) with
// (X_{2i} - Y_{2i+1}) pairs completes X q_even: four dp2a and one LOP3 per word
// give sum q X over its eight elements.  The offset of the codes enters as the
// starting value -8 sum X, so the chunk's D = sum (q - 8) X is exact in int32
// (|D| <= 2^22, exact in f32 too), and the chunk's dot is D * 2^-s.  Activations
// keep 14 significant bits (even) and 10 (odd) relative to the chunk's largest,
// i.e. every bf16 x at least 1/4 of the chunk's largest is exact.
struct Q4Act {
  uint32_t p[16];   // word k: (Y1,Y3), (Y5,Y7), (X0-Y1, X2-Y3), (X4-Y5, X6-Y7) of elements 8k + i
  int off;          // -8 * sum of the 32 integers
  float sc;         // 2^-s (NaN when the chunk holds a NaN or an infinity)
};

// FP8 activation chunk: 16 values as eight f16 pairs at a power-of-two scale
// 2^s chosen so that the chunk's largest magnitude times 2^s lies in [8, 16):
// a product with an E4M3 code (|code| <= 448) stays below 7168 and a half-lane
// sum of eight below 57344, inside f16.  Codes become f16 pairs exactly
// (cvt.rn.f16x2.e4m3x2), each 32-bit word of codes meets its activations in
// two HFMA2, and the chunk's f16 pair of partial sums (eight products each) is
// summed in f32 and scaled by 2^-s.  x is bf16 (8 significant bits) and fits
// f16's 11 exactly unless it is below 2^-14 after scaling (2^-18 of the
// chunk's largest); h (f32) is rounded to 11 bits.
struct F8Act {
  uint32_t p[8];   // f16 pairs (x[2i], x[2i + 1]) * 2^s
  float sc;        // 2^-s (NaN when the chunk holds a NaN or an infinity)
};

template <int F>
struct ActSel {
  using type = FAct<FmtT<F>::kElems>;
};
template <>
struct ActSel<MOE_INT4_G128> {
  using type = Q4Act;
};
template <>
struct ActSel<MOE_FP8_E4M3> {
  using type = F8Act;
};
template <int F>
using ActT = typename ActSel<F>::type;

__device__ __forceinline__ uint32_t pack_s16x2(int lo, int hi) {
  return ((uint32_t)lo & 0xffffu) | ((uint32_t)hi << 16);
}

// 32 activations (f32) -> Q4Act
__device__ __forceinline__ void q4_pack(const float (&x)[32], Q4Act& a) {
  float mx = 0.f;
  bool finite = true;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float v = fabsf(x[i]);
    finite = finite && v <= 3.402823466e38f;   // false for NaN and infinities
    mx = fmaxf(mx, v);
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) a.p[i] = 0u;
  a.off = 0;
  a.sc = 1.f;
  if (!finite) {
    a.sc = __int_as_float(0x7fc00000);   // the chunk's dot becomes NaN, as in float arithmetic
    return;
  }
  if (mx < 5.421010862e-20f) return;      // below 2^-64: contributes nothing measurable
  const int e = (int)((__float_as_uint(mx) >> 23) & 0xffu) - 127;   // mx normal here
  const int sh = 13 - e;                                            // in [-114, 77]
  const float up = __uint_as_float((uint32_t)(127 + sh) << 23);
  const float up16 = __uint_as_float((uint32_t)(127 + sh - 4) << 23);
  a.sc = __uint_as_float((uint32_t)(127 - sh) << 23);
  int sum = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float* xk = x + 8 * k;
    const int X0 = __float2int_rn(xk[0] * up), X2 = __float2int_rn(xk[2] * up);
    const int X4 = __float2int_rn(xk[4] * up), X6 = __float2int_rn(xk[6] * up);
    const int Y1 = __float2int_rn(xk[1] * up16), Y3 = __float2int_rn(xk[3] * up16);
    const int Y5 = __float2int_rn(xk[5] * up16), Y7 = __float2int_rn(xk[7] * up16);
    sum += X0 + X2 + X4 + X6 + 16 * (Y1 + Y3 + Y5 + Y7);
    a.p[4 * k + 0] = pack_s16x2(Y1, Y3);
    a.p[4 * k + 1] = pack_s16x2(Y5, Y7);
    a.p[4 * k + 2] = pack_s16x2(X0 - Y1, X2 - Y3);
    a.p[4 * k + 3] = pack_s16x2(X4 - Y5, X6 - Y7);
  }
  a.off = -8 * sum;
}

// 16 activations (f32) -> F8Act
__device__ __forceinline__ void f8_pack(const float (&x)[16], F8Act& a) {
  float mx = 0.f;
  bool finite = true;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float v = fabsf(x[i]);
    finite = finite && v <= 3.402823466e38f;
    mx = fmaxf(mx, v);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) a.p[i] = 0u;
  a.sc = 1.f;
  if (!finite) {
    a.sc = __int_as_float(0x7fc00000);
    return;
  }
  if (mx < 5.421010862e-20f) return;      // below 2^-64: contributes nothing measurable
  const int e = (int)((__float_as_uint(mx) >> 23) & 0xffu) - 127;
  const int sh = 3 - e;                                              // mx * 2^sh in [8, 16)
  const float up = __uint_as_float((uint32_t)(127 + sh) << 23);
  a.sc = __uint_as_float((uint32_t)(127 - sh) << 23);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __half2 h2 = __floats2half2_rn(x[2 * i] * up, x[2 * i + 1] * up);
    a.p[i] = *reinterpret_cast<const uint32_t*>(&h2);
  }
}

// sum over the chunk of code * x * 2^s, as f32 (the caller scales by 2^-s)
__device__ __forceinline__ float f8_dot(const uint4 w, const F8Act& a) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  __half2 acc = __float2half2_rn(0.f);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t lo, hi;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"((unsigned short)(ws[j] & 0xffffu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"((unsigned short)(ws[j] >> 16)));
    acc = __hfma2(*reinterpret_cast<const __half2*>(&lo), *reinterpret_cast<const __half2*>(&a.p[2 * j]), acc);
    acc = __hfma2(*reinterpret_cast<const __half2*>(&hi), *reinterpret_cast<const __half2*>(&a.p[2 * j + 1]), acc);
  }
  const float2 f = __half22float2(acc);
  return f.x + f.y;
}

__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// sum over the chunk of (q - 8) X, exact
__device__ __forceinline__ int q4_dot(const uint4 w, const Q4Act& a) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  int d = a.off;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t ev = ws[k] & 0x0F0F0F0Fu;
    d = dp2a_lo(a.p[4 * k + 0], ws[k], d);
    d = dp2a_hi(a.p[4 * k + 1], ws[k], d);
    d = dp2a_lo(a.p[4 * k + 2], ev, d);
    d = dp2a_hi(a.p[4 * k + 3], ev, d);
  }
  return d;
}

// dot product of one 16-byte weight chunk with a chunk of activations in
// registers (INT4: before the group scale, which the caller applies)
template <int F>
__device__ __forceinline__ float chunk_dot_r(const uint4 w, const ActT<F>& x) {
  if constexpr (F == MOE_INT4_G128) return (float)q4_dot(w, x) * x.sc;
  else if constexpr (F == MOE_FP8_E4M3) return f8_dot(w, x) * x.sc;
  else return chunk_dot<F>(w, x.v);
}

// an all-zero activation chunk (past the end of x or of this warp's part of h)
template <int F>
__device__ __forceinline__ void act_zero(ActT<F>& a) {
  if constexpr (F == MOE_INT4_G128) {
#pragma unroll
    for (int i = 0; i < 16; ++i) a.p[i] = 0u;
    a.off = 0;
    a.sc = 1.f;
  } else if constexpr (F == MOE_FP8_E4M3) {
#pragma unroll
    for (int i = 0; i < 8; ++i) a.p[i] = 0u;
    a.sc = 1.f;
  } else {
#pragma unroll
    for (int e = 0; e < FmtT<F>::kElems; ++e) a.v[e] = 0.f;
  }
}

// EL activations as f32 -> the register form
template <int F>
__device__ __forceinline__ void act_set(ActT<F>& a, const float (&v)[FmtT<F>::kElems]) {
  if constexpr (F == MOE_INT4_G128) q4_pack(v, a);
  else if constexpr (F == MOE_FP8_E4M3) f8_pack(v, a);
  else {
#pragma unroll
    for (int e = 0; e < FmtT<F>::kElems; ++e) a.v[e] = v[e];
  }
}

// activation chunk (EL values) -> registers; x is bf16 unless F is f32
template <int F>
__device__ __forceinline__ void load_x_chunk(ActT<F>& act, const void* x, int c) {
  constexpr int EL = FmtT<F>::kElems;
  float dst[EL];
  if (F == MOE_F32) {
    const float4 v = reinterpret_cast<const float4*>(x)[c];
    dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
  } else {
#pragma unroll
    for (int i = 0; i < EL / 8; ++i) {
      const uint4 v = reinterpret_cast<const uint4*>(x)[(size_t)c * (EL / 8) + i];
      float* d = dst + 8 * i;
      d[0] = bf16_lo(v.x); d[1] = bf16_hi(v.x); d[2] = bf16_lo(v.y); d[3] = bf16_hi(v.y);
      d[4] = bf16_lo(v.z); d[5] = bf16_hi(v.z); d[6] = bf16_lo(v.w); d[7] = bf16_hi(v.w);
    }
  }
  act_set<F>(act, dst);
}

// Dot products of NR weight rows with the token's x (registers), reduced
// over the warp; every lane gets the sums.  Row r's 16-byte chunks come from
// the stage (ring) or from global memory (plain loads; with `copy`, also
// stored to cpy[r], the row's place in the expert's slot).  INT4 scales come
// from srow[r] (bf16, one per 128 elements).
template <int F, int NR>
__device__ __forceinline__ void rows_dot(const uint4* const (&row)[NR], const uint16_t* const (&srow)[NR],
                                         uint4* const (&cpy)[NR], bool ring, bool copy, int C,
                                         const ActT<F> (&xr)[RingTile<F>::XM], int lane,
                                         float (&out)[NR]) {
  constexpr int XM = RingTile<F>::XM;
  uint4 wv[NR][XM];
  float sc[NR][XM];
  if (ring) {
    // branch-free: chunks past the row end re-read its last chunk; their x is
    // zero, so they add nothing
#pragma unroll
    for (int m = 0; m < XM; ++m) {
      const int c = min(lane + 32 * m, C - 1);
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        wv[r][m] = row[r][c];
        sc[r][m] = F == MOE_INT4_G128 ? bf16_bits(srow[r][c >> 2]) : 0.f;
      }
    }
  } else {
#pragma unroll
    for (int m = 0; m < XM; ++m) {
      const int c = lane + 32 * m;
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        wv[r][m] = make_uint4(0u, 0u, 0u, 0u);
        sc[r][m] = 0.f;
        if (c < C) {
          wv[r][m] = __ldcs(row[r] + c);
          if (F == MOE_INT4_G128) sc[r][m] = bf16_bits(srow[r][c >> 2]);
        }
      }
    }
  }
  if (copy) {
#pragma unroll
    for (int m = 0; m < XM; ++m) {
      const int c = lane + 32 * m;
#pragma unroll
      for (int r = 0; r < NR; ++r)
        if (c < C) cpy[r][c] = wv[r][m];
    }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float acc = 0.f;
#pragma unroll
    for (int m = 0; m < XM; ++m) {
      const float dd = chunk_dot_r<F>(wv[r][m], xr[m]);
      acc = (F == MOE_INT4_G128) ? fmaf(dd, sc[r][m], acc) : acc + dd;
    }
    out[r] = warp_sum(acc);
  }
}

// h = w * silu(g) * u.  FP8: the gate and up tensor scales apply to the dot
// products, and the down scale is folded into h (a down dot mixes experts).
template <int F>
__device__ __forceinline__ float swiglu_h(const RingShared& S, unsigned long long base, int asg, float g, float u) {
  if (F == MOE_FP8_E4M3) {
    g *= S.fsc[asg][0];
    u *= S.fsc[asg][1];
  }
  const float h = base != 0ull ? S.wt[asg] * (g / (1.0f + expf(-g)) * u) : 0.f;
  return F == MOE_FP8_E4M3 ? h * S.fsc[asg][2] : h;
}

// Up item of P = d.n row pairs (pairs d.p0 .. d.p0 + P - 1 of assignment
// d.asg).  The stage holds [gate rows (P) | up rows (P) | gate scales (P) |
// up scales (P)], so stage row r is gate row p0 + r for r < P, else up row
// I + p0 + r - P.
//   P == 2 * kConsumers (INT4, FP8): warp cw takes pairs cw and cw + kConsumers.
//   P == kConsumers: warp cw takes pair cw, both of its rows.
//   P == kConsumers / 2: warp cw takes stage row cw alone; the two warps of a
//   pair meet through S.gu / S.cnt of this stage (the second one to finish
//   writes h), so no barrier is needed.
template <int F>
__device__ __forceinline__ void up_item(const MlpArgs& a, RingShared& S, const RingDesc& d, int s,
                                        const uint8_t* stage, const ActT<F> (&xr)[RingTile<F>::XM],
                                        int cw, int lane) {
  const int P = d.n;
  const int C = a.H / FmtT<F>::kElems;
  const int G = a.H / 128;
  const size_t rb = row_bytes<F>(a.H);
  const unsigned long long base = S.base[d.asg];
  const bool ring = d.src == SRC_RING;
  const bool copy = d.src == SRC_PLAIN && a.readthrough && a.pending[d.asg] != 0;
  const unsigned long long blk = copy ? a.src_ptr[d.asg] : base;
  // stage row r -> weight row of the expert block
  auto wrow = [&](int r) { return r < P ? d.p0 + r : a.I + d.p0 + r - P; };
  auto rowp = [&](int r) -> const uint4* {
    return ring ? reinterpret_cast<const uint4*>(stage + (size_t)r * rb)
                : reinterpret_cast<const uint4*>(blk + (size_t)wrow(r) * rb);
  };
  auto srowp = [&](int r) -> const uint16_t* {
    return ring ? reinterpret_cast<const uint16_t*>(stage + 2 * (size_t)P * rb) + (size_t)r * G
                : reinterpret_cast<const uint16_t*>(blk + a.off_s13) + (size_t)wrow(r) * G;
  };
  auto cpyp = [&](int r) { return reinterpret_cast<uint4*>(base + (size_t)wrow(r) * rb); };
  if ((F == MOE_INT4_G128 || F == MOE_FP8_E4M3) && P == 2 * kConsumers) {
    // (INT4, FP8) warp cw takes pairs cw and cw + kConsumers, all four rows
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    const int c2 = cw + kConsumers;
    if (d.src != SRC_NONE) {
      const uint4* const rows[4] = {rowp(cw), rowp(c2), rowp(P + cw), rowp(P + c2)};
      const uint16_t* const srows[4] = {srowp(cw), srowp(c2), srowp(P + cw), srowp(P + c2)};
      uint4* const cpys[4] = {copy ? cpyp(cw) : nullptr, copy ? cpyp(c2) : nullptr, copy ? cpyp(P + cw) : nullptr,
                              copy ? cpyp(P + c2) : nullptr};
      if constexpr (F == MOE_INT4_G128 || F == MOE_FP8_E4M3) rows_dot<F, 4>(rows, srows, cpys, ring, copy, C, xr, lane, v);
    }
    if (lane < kHRep) {
      float* hrow = a.h + (size_t)lane * a.k * a.I + (size_t)d.asg * a.I + d.p0;
      hrow[cw] = swiglu_h<F>(S, base, d.asg, v[0], v[2]);
      hrow[c2] = swiglu_h<F>(S, base, d.asg, v[1], v[3]);
    }
  } else if (P == kConsumers) {
    float v[2] = {0.f, 0.f};
    if (d.src != SRC_NONE) {
      const uint4* const rows[2] = {rowp(cw), rowp(P + cw)};
      const uint16_t* const srows[2] = {srowp(cw), srowp(P + cw)};
      uint4* const cpys[2] = {copy ? cpyp(cw) : nullptr, copy ? cpyp(P + cw) : nullptr};
      rows_dot<F, 2>(rows, srows, cpys, ring, copy, C, xr, lane, v);
    }
    // every lane holds the sums: lanes 0..kHRep-1 write one copy of h each
    if (lane < kHRep)
      a.h[(size_t)lane * a.k * a.I + (size_t)d.asg * a.I + d.p0 + cw] = swiglu_h<F>(S, base, d.asg, v[0], v[1]);
  } else {
    float v[1] = {0.f};
    if (d.src != SRC_NONE) {
      const uint4* const rows[1] = {rowp(cw)};
      const uint16_t* const srows[1] = {srowp(cw)};
      uint4* const cpys[1] = {copy ? cpyp(cw) : nullptr};
      rows_dot<F, 1>(rows, srows, cpys, ring, copy, C, xr, lane, v);
    }
    if (lane == 0) {
      const int pr = cw % P, role = cw / P;   // role 0 = gate, 1 = up
      S.gu[s][pr][role] = v[0];
      __threadfence_block();
      if (atomicAdd(&S.cnt[s][pr], 1) == 1) {
        __threadfence_block();
        const float g = S.gu[s][pr][0], u = S.gu[s][pr][1];
        S.cnt[s][pr] = 0;
        const float hv = swiglu_h<F>(S, base, d.asg, g, u);
        for (int r = 0; r < kHRep; ++r) a.h[(size_t)r * a.k * a.I + (size_t)d.asg * a.I + d.p0 + pr] = hv;
      }
    }
  }
}

// Down item: output rows d.p0 + r, r < d.n.  Consumer warp cw takes part
// cw % kParts of rows r = cw / kParts + kRowsPerPass i, two rows at a time
// (independent accumulators, one chunk decode for both).  The stage holds,
// per expert j in the ring, its d.n W2 rows at j * d.n * rb2, then (INT4) its
// scale rows after all the weight rows.  qj[m] packs (expert << 16 | chunk in
// expert row) of this lane's chunk m, or -1.
template <int F>
__device__ __forceinline__ void down_rows(const MlpArgs& a, const RingShared& S, const RingDesc& d,
                                          const uint8_t* stage, const ActT<F> (&hr)[RingTile<F>::HM],
                                          const int (&qj)[RingTile<F>::HM], float* part, int cw, int lane) {
  constexpr int HM = RingTile<F>::HM;
  const int G2 = a.I / 128;
  const size_t rb2 = row_bytes<F>(a.I);
  const size_t wbytes = (size_t)d.n * rb2;
  const size_t sbytes = (size_t)d.n * G2 * 2;
  const uint8_t* sring = stage + (size_t)a.k * wbytes;
  // per chunk: byte offset of row 0 in the stage (or -1: not in the ring)
  uint32_t off[HM], soff[HM];
#pragma unroll
  for (int m = 0; m < HM; ++m) {
    const int e = qj[m];
    off[m] = 0xffffffffu;
    soff[m] = 0u;
    if (e >= 0) {
      const int j = e >> 16, c = e & 0xffff;
      if (S.base[j] != 0ull && !((d.src >> j) & 1u)) {
        off[m] = (uint32_t)((size_t)j * wbytes + (size_t)c * 16);
        soff[m] = (uint32_t)((size_t)j * sbytes + (size_t)(c >> 2) * 2);
      }
    }
  }
  if (d.src == 0u) {
    // every expert of the item is in the ring: branch-free loads (chunks past
    // the part's end read offset 0; their h is zero, so they add nothing)
    for (int r0 = cw / kParts; r0 < d.n; r0 += 2 * kRowsPerPass) {
      const int r1 = r0 + kRowsPerPass;
      const bool two = r1 < d.n;
      const int r1c = two ? r1 : r0;
      uint4 w0[HM], w1[HM];
      float s0[HM], s1[HM];
#pragma unroll
      for (int m = 0; m < HM; ++m) {
        const uint32_t o = off[m] == 0xffffffffu ? 0u : off[m];
        w0[m] = *reinterpret_cast<const uint4*>(stage + o + (size_t)r0 * rb2);
        w1[m] = *reinterpret_cast<const uint4*>(stage + o + (size_t)r1c * rb2);
        if (F == MOE_INT4_G128) {
          const uint16_t* sp = reinterpret_cast<const uint16_t*>(sring + soff[m]);
          s0[m] = bf16_bits(sp[(size_t)r0 * G2]);
          s1[m] = bf16_bits(sp[(size_t)r1c * G2]);
        }
      }
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int m = 0; m < HM; ++m) {
        const float d0 = chunk_dot_r<F>(w0[m], hr[m]);
        const float d1 = chunk_dot_r<F>(w1[m], hr[m]);
        if (F == MOE_INT4_G128) {
          acc0 = fmaf(d0, s0[m], acc0);
          acc1 = fmaf(d1, s1[m], acc1);
        } else {
          acc0 += d0;
          acc1 += d1;
        }
      }
      acc0 = warp_sum(acc0);
      acc1 = warp_sum(acc1);
      if (lane == 0) {
        part[kParts * r0 + cw % kParts] = acc0;
        if (two) part[kParts * r1 + cw % kParts] = acc1;
      }
    }
    return;
  }
  for (int r0 = cw / kParts; r0 < d.n; r0 += 2 * kRowsPerPass) {
    const int r1 = r0 + kRowsPerPass;
    const bool two = r1 < d.n;
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int m = 0; m < HM; ++m) {
      uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = w0;
      float s0 = 0.f, s1 = 0.f;
      if (off[m] != 0xffffffffu) {
        w0 = *reinterpret_cast<const uint4*>(stage + off[m] + (size_t)r0 * rb2);
        if (two) w1 = *reinterpret_cast<const uint4*>(stage + off[m] + (size_t)r1 * rb2);
        if (F == MOE_INT4_G128) {
          const uint16_t* sp = reinterpret_cast<const uint16_t*>(sring + soff[m]);
          s0 = bf16_bits(sp[(size_t)r0 * G2]);
          if (two) s1 = bf16_bits(sp[(size_t)r1 * G2]);
        }
      } else if (qj[m] >= 0) {
        // expert read from global memory: missing, host-resident or read through
        const int j = qj[m] >> 16, c = qj[m] & 0xffff;
        const unsigned long long blk = S.base[j];
        if (blk != 0ull) {
          const uint4* wrow = reinterpret_cast<const uint4*>(blk + a.off_w2) + c;
          const unsigned short* srow = reinterpret_cast<const unsigned short*>(blk + a.off_s2) + (c >> 2);
          const size_t n0 = (size_t)(d.p0 + r0), n1 = (size_t)(d.p0 + r1);
          w0 = __ldcg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(wrow) + n0 * rb2));
          if (two) w1 = __ldcg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(wrow) + n1 * rb2));
          if (F == MOE_INT4_G128) {
            s0 = bf16_bits(__ldcg(srow + n0 * G2));
            if (two) s1 = bf16_bits(__ldcg(srow + n1 * G2));
          }
        }
      }
      const float d0 = chunk_dot_r<F>(w0, hr[m]);
      const float d1 = chunk_dot_r<F>(w1, hr[m]);
      if (F == MOE_INT4_G128) {
        acc0 = fmaf(d0, s0, acc0);
        acc1 = fmaf(d1, s1, acc1);
      } else {
        acc0 += d0;
        acc1 += d1;
      }
    }
    acc0 = warp_sum(acc0);
    acc1 = warp_sum(acc1);
    if (lane == 0) {
      part[kParts * r0 + cw % kParts] = acc0;
      if (two) part[kParts * r1 + cw % kParts] = acc1;
    }
  }
}

// ------------------------------------------------------------- copier
// A pending block is copied in chunks of at most kCopyChunk bytes, phase A
// first (w13, then the gate/up scales: what the up items read), then phase B
// (w2, then the down scales).
__device__ __forceinline__ int chunk_count(unsigned long long bytes) {
  return (int)((bytes + kCopyChunk - 1) / kCopyChunk);
}
__device__ __forceinline__ int phase_chunks(const MlpArgs& a, bool b) {
  return b ? chunk_count(a.off_s13 - a.off_w2) + chunk_count(a.blk_bytes - a.off_s2)
           : chunk_count(a.off_w2) + chunk_count(a.off_s2 - a.off_s13);
}
// byte range [lo, hi) of chunk c of phase b
__device__ __forceinline__ void chunk_range(const MlpArgs& a, bool b, int c, unsigned long long* lo,
                                            unsigned long long* hi) {
  const unsigned long long r0 = b ? a.off_w2 : 0ull, r0e = b ? a.off_s13 : a.off_w2;
  const unsigned long long r1 = b ? a.off_s2 : a.off_s13, r1e = b ? a.blk_bytes : a.off_s2;
  const int n0 = chunk_count(r0e - r0);
  const unsigned long long base = c < n0 ? r0 : r1, end = c < n0 ? r0e : r1e;
  *lo = base + (unsigned long long)(c < n0 ? c : c - n0) * kCopyChunk;
  *hi = *lo + kCopyChunk < end ? *lo + kCopyChunk : end;
}

// Copier warp: the chunks of the pending blocks, spread over the grid (chunk
// b, b + G, ... of the global list: every phase A chunk of every pending
// assignment, then every phase B chunk), host -> slot with plain 16-byte
// loads and stores; each landed chunk is counted with a release add.
__device__ __forceinline__ void copier(const MlpArgs& a, const RingShared& S, int lane) {
  // the same blocks the producer waits for (pending, in HBM, 16-byte aligned)
  const unsigned long long b = lane < a.k ? S.base[lane] : 0ull;
  const unsigned pend = __ballot_sync(
      kFull, lane < a.k && a.pending[lane] != 0 && b != 0ull && !in_host(a, b) && (b & 15ull) == 0ull);
  const long long np = __popc(pend);
  // timing record (see MlpArgs::copy_span): header, then this CTA's span
  unsigned long long* rec = (a.copy_span != nullptr && gridDim.x <= (unsigned)kSpanMaxCtas)
                                ? a.copy_span + 2 + 2 * (size_t)blockIdx.x : nullptr;
  if (rec != nullptr && blockIdx.x == 0 && lane == 0) {
    a.copy_span[0] = (unsigned long long)np;
    a.copy_span[1] = gridDim.x;
  }
  if (pend == 0u) {
    if (rec != nullptr && lane == 0) rec[0] = rec[1] = 0ull;
    return;
  }
  const int nA = phase_chunks(a, false), nB = phase_chunks(a, true);
  const long long total = np * (nA + nB);
  // timing: when this warp issued its first chunk (warp-uniform)
  const unsigned long long t_first = (rec != nullptr && blockIdx.x < total) ? global_ns() : 0ull;
  for (long long ci = blockIdx.x; ci < total; ci += gridDim.x) {
    const bool pb = ci >= np * nA;
    const long long cc = pb ? ci - np * nA : ci;
    const int per = pb ? nB : nA;
    const int pj = (int)(cc / per), c = (int)(cc - (long long)pj * per);
    const int j = nth_set_bit(pend, pj);
    unsigned long long lo, hi;
    chunk_range(a, pb, c, &lo, &hi);
    const uint4* src = reinterpret_cast<const uint4*>(a.src_ptr[j] + lo);
    uint4* dst = reinterpret_cast<uint4*>(S.base[j] + lo);
    const int nv = (int)((hi - lo) / 16ull);
    for (int v0 = 0; v0 < nv; v0 += 32 * kCopyBatch) {
      uint4 v[kCopyBatch];
#pragma unroll
      for (int u = 0; u < kCopyBatch; ++u) {
        const int q = v0 + lane + 32 * u;
        if (q < nv) v[u] = __ldcs(src + q);
      }
#pragma unroll
      for (int u = 0; u < kCopyBatch; ++u) {
        const int q = v0 + lane + 32 * u;
        if (q < nv) dst[q] = v[u];
      }
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) {
      if (!pb) red_release_add(a.copy_cnt + j, 1u);
      red_release_add(a.copy_cnt + MOE_MAX_TOPK + j, 1u);
    }
  }
  if (rec != nullptr && lane == 0) {
    // every chunk of this warp has landed (fenced above)
    rec[0] = t_first;
    rec[1] = blockIdx.x < total ? global_ns() : 0ull;
  }
}

// ------------------------------------------------------------- producer
// Items of CTA b of G: up items = groups of P = up_pairs consecutive row
// pairs of one assignment, groups b, b + G, b + 2 G, ... of the NG = k * I / P
// groups (expert-major); then down items = runs of down_rows output rows of
// the CTA's row range (whole groups of down_group rows).
struct Share {
  int g0, gstride;    // up groups g0, g0 + gstride, ... (below ng)
  int n0, n1;         // output rows
  int n_up, n_items;
};

__device__ __forceinline__ Share cta_share(const MlpArgs& a, const RingCfg& rc) {
  Share w;
  const long long G = gridDim.x, b = blockIdx.x;
  const long long ng = (long long)a.k * (a.I / rc.up_pairs);
  // groups round-robin over the CTAs, so that every expert -- in particular
  // one read from host memory in this step -- is spread over many CTAs
  w.g0 = (int)b;
  w.gstride = (int)G;
  w.n_up = b < ng ? (int)((ng - 1 - b) / G + 1) : 0;
  const long long nrg = a.H / rc.down_group;
  w.n0 = (int)(nrg * b / G) * rc.down_group;
  w.n1 = (int)(nrg * (b + 1) / G) * rc.down_group;
  w.n_items = w.n_up + (w.n1 - w.n0 + rc.down_rows - 1) / rc.down_rows;
  return w;
}

template <int F>
__device__ __forceinline__ void produce(const MlpArgs& a, const RingCfg& rc, RingShared& S, uint8_t* ring,
                                        int lane, int* err) {
  const Share w = cta_share(a, rc);
  const int NS = rc.nstages;
  const size_t rb1 = row_bytes<F>(a.H), rb2 = row_bytes<F>(a.I);
  const size_t srb1 = F == MOE_INT4_G128 ? (size_t)(a.H / 128) * 2 : 0;
  const size_t srb2 = F == MOE_INT4_G128 ? (size_t)(a.I / 128) * 2 : 0;
  const int P = rc.up_pairs;
  const int gpe = a.I / P;   // groups per expert
  // experts that are not bulk-copied: no block, host blocks, blocks filled by
  // read-through in this step, or (defensively) blocks not 16-byte aligned
  const unsigned long long myb = lane < a.k ? S.base[lane] : 0ull;
  // with the copier, a pending block is bulk-copied from its slot once its
  // chunks have landed; without it, the consumers read it through
  const bool cp_mode = a.readthrough && a.copy_cnt != nullptr;
  const bool pend = lane < a.k && a.readthrough && a.pending[lane] != 0;
  const bool plain = lane < a.k && (myb == 0ull || in_host(a, myb) || (myb & 15ull) != 0ull || (pend && !cp_mode));
  const unsigned plain_mask = __ballot_sync(kFull, plain);
  const unsigned k_mask = a.k >= 32 ? kFull : ((1u << a.k) - 1u);
  const int n_ring = __popc(k_mask & ~plain_mask);
  const unsigned wait_mask = cp_mode ? __ballot_sync(kFull, pend && !plain) : 0u;
  // item order: the assignments that wait for the copier come last
  if (lane < a.k) {
    const unsigned lt = (1u << lane) - 1u, early = k_mask & ~wait_mask;
    S.jorder[(wait_mask >> lane) & 1u ? __popc(early) + __popc(wait_mask & lt) : __popc(early & lt)] = lane;
  }
  __syncwarp();
  const int nA = cp_mode ? phase_chunks(a, false) : 0, nAll = cp_mode ? nA + phase_chunks(a, true) : 0;
  unsigned landed = 0u;   // assignments whose phase A chunks have all landed
  const unsigned long long pol_first = evict_first_policy();
  int i = 0;
  for (; i < w.n_items; ++i) {
    if (i == w.n_up && w.n_items - w.n_up > NS && lane < a.k && !plain && !((wait_mask >> lane) & 1u)) {
      // the W2 rows of the down items that wait for a free stage: into L2 now,
      // while the grid meets, so that their copies after the barrier are short
      const int nr0 = w.n0 + NS * rc.down_rows;
      const uint8_t* blk = reinterpret_cast<const uint8_t*>(myb);
      prefetch_l2(blk + a.off_w2 + (size_t)nr0 * rb2, (unsigned)((size_t)(w.n1 - nr0) * rb2));
      if (srb2 != 0) prefetch_l2(blk + a.off_s2 + (size_t)nr0 * srb2, (unsigned)((size_t)(w.n1 - nr0) * srb2));
    }
    const int s = i % NS;
    const uint32_t full = smem_u32(&S.full[s]);
    uint8_t* st = ring + (size_t)s * rc.stage_bytes;
    bool ok = true;
    if (lane == 0 && i >= NS) ok = mbar_wait(smem_u32(&S.empty[s]), (unsigned)((i / NS) - 1) & 1u);
    ok = __shfl_sync(kFull, ok, 0);
    if (!ok) {
      if (lane == 0) {
        atomicExch(err, DEVERR_RING);
        *reinterpret_cast<volatile int*>(&S.stop) = 1;
      }
      break;
    }
    if (i < w.n_up) {
      const int gg = w.g0 + i * w.gstride;
      const int jj = gg / gpe;
      const int p0 = (gg - jj * gpe) * P;
      const int j = S.jorder[jj];
      if ((wait_mask >> j) & 1u & ~(landed >> j)) {
        // the block's w13 (and gate/up scales) must be in its slot first
        bool got = true;
        if (lane == 0) got = wait_count(a.copy_cnt + j, (unsigned)nA);
        if (!__shfl_sync(kFull, got, 0)) {
          if (lane == 0) {
            atomicExch(err, DEVERR_RING);
            *reinterpret_cast<volatile int*>(&S.stop) = 1;
          }
          break;
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");   // copier stores -> bulk copy reads
        landed |= 1u << j;
      }
      const unsigned long long blk = __shfl_sync(kFull, myb, j);
      const bool pl = (plain_mask >> j) & 1u;
      const unsigned src = blk == 0ull ? SRC_NONE : (pl ? SRC_PLAIN : SRC_RING);
      if (lane == 0) S.desc[s] = RingDesc{0, j, p0, P, src};
      if (src == SRC_RING) {
        const unsigned wb = (unsigned)(P * rb1), sb = (unsigned)(P * srb1);
        if (lane == 0) mbar_arrive_tx(full, 2u * (wb + sb));
        __syncwarp();
        const uint8_t* w13 = reinterpret_cast<const uint8_t*>(blk);
        if (lane == 0) bulk_copy_hint(smem_u32(st), w13 + (size_t)p0 * rb1, wb, full, pol_first);
        if (lane == 1) bulk_copy_hint(smem_u32(st + wb), w13 + (size_t)(a.I + p0) * rb1, wb, full, pol_first);
        if (sb != 0u) {
          const uint8_t* s13 = w13 + a.off_s13;
          if (lane == 2) bulk_copy_hint(smem_u32(st + 2 * wb), s13 + (size_t)p0 * srb1, sb, full, pol_first);
          if (lane == 3) bulk_copy_hint(smem_u32(st + 2 * wb + sb), s13 + (size_t)(a.I + p0) * srb1, sb, full, pol_first);
        }
      } else if (lane == 0) {
        mbar_arrive(full);
      }
    } else {
      if (i == w.n_up && wait_mask != 0u) {
        // every pending block whole in its slot before its W2 rows are read
        const bool got = !((wait_mask >> lane) & 1u) || wait_count(a.copy_cnt + MOE_MAX_TOPK + lane, (unsigned)nAll);
        if (!__all_sync(kFull, got)) {
          if (lane == 0) {
            atomicExch(err, DEVERR_RING);
            *reinterpret_cast<volatile int*>(&S.stop) = 1;
          }
          break;
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      const int n = w.n0 + (i - w.n_up) * rc.down_rows;
      const int nr = min(rc.down_rows, w.n1 - n);
      if (lane == 0) S.desc[s] = RingDesc{1, 0, n, nr, plain_mask};
      const unsigned wb = (unsigned)(nr * rb2), sb = (unsigned)(nr * srb2);
      const unsigned bytes = (unsigned)n_ring * (wb + sb);
      if (lane == 0) {
        if (bytes) mbar_arrive_tx(full, bytes);
        else mbar_arrive(full);
      }
      __syncwarp();
      if (lane < a.k && !plain) {
        const uint8_t* blk = reinterpret_cast<const uint8_t*>(myb);
        // W2 rows are read once per launch too: evict-first, so that they do
        // not push the slot state and the prepare code out of L2
        bulk_copy_hint(smem_u32(st + (size_t)lane * wb), blk + a.off_w2 + (size_t)n * rb2, wb, full, pol_first);
        if (sb != 0u)
          bulk_copy_hint(smem_u32(st + (size_t)a.k * wb + (size_t)lane * sb), blk + a.off_s2 + (size_t)n * srb2, sb,
                         full, pol_first);
      }
    }
  }
  // every copy this CTA issued has landed before it may exit
  if (lane == 0) {
    for (int q = i > NS ? i - NS : 0; q < i; ++q)
      if (!mbar_wait(smem_u32(&S.full[q % NS]), (unsigned)(q / NS) & 1u)) atomicExch(err, DEVERR_RING);
  }
  __syncwarp();
}

// y for output rows n0 + r, r < nr, from their part sums (part + kParts r),
// one consumer thread per row, parts summed in a fixed order
template <int F>
__device__ __forceinline__ void down_store(const MlpArgs& a, const RingShared& S, const float* part, int n0, int nr,
                                           int cta_n0, int ctid) {
  for (int r = ctid; r < nr; r += 32 * kConsumers) {
    const float* pr = part + kParts * r;
    const int n = n0 + r;
    float v = (pr[0] + pr[1]) + (pr[2] + pr[3]);
    if (a.residual) v += n - cta_n0 < kMaxRows ? S.xres[n - cta_n0] : x_at<F>(a, n);
    store_out<F>(a, n, v);
  }
}

// ------------------------------------------------------- consumer driver
template <int F>
__device__ __forceinline__ void consume(const MlpArgs& a, const RingCfg& rc, RingShared& S, const uint8_t* ring,
                                        GridBar* bar, int* err, int cw, int lane) {
  constexpr int EL = FmtT<F>::kElems;
  constexpr int XM = RingTile<F>::XM, HM = RingTile<F>::HM;
  const Share w = cta_share(a, rc);
  const int NS = rc.nstages;
  const int ctid = cw * 32 + lane;
  volatile int* stop = &S.stop;
  // read-through: copies of the missed experts' bytes after w13 (w2 and
  // scales) into their slots, 4 KiB per task, an equal share per CTA.  They
  // complete before the grid barrier, so the down items may read them from
  // the slots.
  if (a.readthrough && a.copy_cnt == nullptr) {
    const unsigned pend = __ballot_sync(kFull, lane < a.k && a.pending[lane] != 0 && S.base[lane] != 0ull);
    if (pend) {
      const unsigned long long cpe = (a.tail_bytes + 4095ull) / 4096ull;
      const unsigned long long ncopy = (unsigned long long)__popc(pend) * cpe;
      const unsigned long long c_beg = ncopy * blockIdx.x / gridDim.x;
      const unsigned long long c_end = ncopy * (blockIdx.x + 1) / gridDim.x;
      const unsigned long long nv_all = a.tail_bytes / 16ull;
      for (unsigned long long c = c_beg + cw; c < c_end; c += kConsumers) {
        const int sidx = (int)(c / cpe);
        const unsigned long long v0 = (c - (unsigned long long)sidx * cpe) * 256ull;   // 4 KiB = 256 vectors
        const int j = nth_set_bit(pend, sidx);
        const uint4* src = reinterpret_cast<const uint4*>(a.src_ptr[j] + a.tail_off);
        uint4* dst = reinterpret_cast<uint4*>(S.base[j] + a.tail_off);
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const unsigned long long q = v0 + lane + 32u * u;
          if (q < nv_all) v[u] = __ldcs(src + q);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const unsigned long long q = v0 + lane + 32u * u;
          if (q < nv_all) dst[q] = v[u];
        }
      }
    }
  }
  bool dead = false;
  int i = 0;
  // ---- up items: x of the token in registers
  {
    ActT<F> xr[XM];
    const int C = a.H / EL;
#pragma unroll
    for (int m = 0; m < XM; ++m) {
      const int c = lane + 32 * m;
      if (c < C) load_x_chunk<F>(xr[m], a.x, c);
      else act_zero<F>(xr[m]);
    }
    for (; i < w.n_up; ++i) {
      const int s = i % NS;
      if (!dead && *stop) dead = true;
      if (!dead) {
        const bool ok = mbar_wait(smem_u32(&S.full[s]), (unsigned)(i / NS) & 1u);
        if (!__all_sync(kFull, ok)) {
          dead = true;
          if (lane == 0) {
            atomicExch(err, DEVERR_RING);
            *stop = 1;
          }
        }
      }
      if (!dead) {
        const RingDesc d = S.desc[s];
        if (cw < 2 * d.n) up_item<F>(a, S, d, s, ring + (size_t)s * rc.stage_bytes, xr, cw, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.empty[s]));
    }
  }
  // h complete everywhere; W2 rows keep landing in the ring meanwhile
  consumer_grid_barrier(bar, err, ctid);
  if (i >= w.n_items) return;
  // ---- down items: this warp's half of h in registers
  {
    const int C2 = a.I / EL;
    const int Q = a.k * C2;
    const int Qp = (Q + kParts - 1) / kParts;
    const int pt = cw % kParts;
    const int q_end = min(Q, (pt + 1) * Qp);
    // this warp's part of h (k * I f32, written by every CTA) -> registers,
    // straight from L2
    ActT<F> hr[HM];
    int qj[HM];
#pragma unroll
    for (int m = 0; m < HM; ++m) {
      const int q = pt * Qp + lane + 32 * m;
      qj[m] = -1;
      if (q < q_end) {
        const int j = q / C2;
        qj[m] = (j << 16) | (q - j * C2);
        // every CTA reads all of h: copy blockIdx % kHRep, so that the reads
        // of the grid spread over kHRep times as many L2 lines
        const float* src = a.h + (size_t)(blockIdx.x % kHRep) * a.k * a.I + (size_t)q * EL;
        float hv[EL];
#pragma unroll
        for (int e = 0; e < EL / 4; ++e) {
          const float4 v = ld_l2_f4(src + 4 * e);
          hv[4 * e] = v.x;
          hv[4 * e + 1] = v.y;
          hv[4 * e + 2] = v.z;
          hv[4 * e + 3] = v.w;
        }
        act_set<F>(hr[m], hv);
      } else {
        act_zero<F>(hr[m]);
      }
    }
    for (; i < w.n_items; ++i) {
      const int s = i % NS;
      if (!dead && *stop) dead = true;
      if (!dead) {
        const bool ok = mbar_wait(smem_u32(&S.full[s]), (unsigned)(i / NS) & 1u);
        if (!__all_sync(kFull, ok)) {
          dead = true;
          if (lane == 0) {
            atomicExch(err, DEVERR_RING);
            *stop = 1;
          }
        }
      }
      const RingDesc d = S.desc[s];
      // part sums go to the row's place in S.part; a CTA with more rows than
      // that holds reuses it from the start, one item at a time
      const bool all_rows = w.n1 - w.n0 <= kMaxRows;
      float* part = S.part + (all_rows ? kParts * (d.p0 - w.n0) : 0);
      if (!dead) down_rows<F>(a, S, d, ring + (size_t)s * rc.stage_bytes, hr, qj, part, cw, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.empty[s]));
      if (!all_rows) {
        consumer_sync();   // every part of every row of the item is in part[]
        if (!dead) down_store<F>(a, S, part, d.p0, d.n, w.n0, ctid);
        consumer_sync();   // part[] is free for the next item
      }
    }
    if (w.n1 - w.n0 <= kMaxRows) {
      consumer_sync();     // every part of every row of the CTA is in S.part
      if (!dead) down_store<F>(a, S, S.part, w.n0, w.n1 - w.n0, w.n0, ctid);
    }
  }
}

template <int F>
__global__ void __launch_bounds__(kRingThreads, 1) k_mlp_ring(MlpArgs a, RingCfg rc, GridBar* bar, int* err) {
  extern __shared__ __align__(1024) uint8_t ring[];
  __shared__ RingShared S;
  // the next kernel of the stream (a prepare launched as a programmatic
  // dependent) may be scheduled now: it waits for this grid to complete
  // before it touches memory.  Its CTA takes an SM as soon as one of this
  // grid's CTAs exits (beside one it would need more than the SM's registers).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < a.k) {
    S.base[threadIdx.x] = a.asg_ptr[threadIdx.x];
    S.wt[threadIdx.x] = a.w[threadIdx.x];
    if (F == MOE_FP8_E4M3) {
      // the block's scales: from its host copy while the copier is still moving it
      const unsigned long long b = (a.readthrough && a.pending[threadIdx.x] != 0) ? a.src_ptr[threadIdx.x]
                                                                                  : a.asg_ptr[threadIdx.x];
      float g = 0.f, u = 0.f, dn = 0.f;
      if (b != 0ull) {
        const float* f13 = reinterpret_cast<const float*>(b + a.off_s13);
        g = __ldcg(f13);
        u = __ldcg(f13 + 1);
        dn = __ldcg(reinterpret_cast<const float*>(b + a.off_s2));
      }
      S.fsc[threadIdx.x][0] = g;
      S.fsc[threadIdx.x][1] = u;
      S.fsc[threadIdx.x][2] = dn;
    }
  }
  if (a.residual) {
    const Share w = cta_share(a, rc);
    for (int r = threadIdx.x; r < w.n1 - w.n0 && r < kMaxRows; r += blockDim.x) S.xres[r] = x_at<F>(a, w.n0 + r);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < rc.nstages; ++s) {
      mbar_init(smem_u32(&S.full[s]), 1u);
      mbar_init(smem_u32(&S.empty[s]), (unsigned)kConsumers);
    }
    S.stop = 0;
    for (int q = 0; q < kMaxStages * (kConsumers / 2); ++q) (&S.cnt[0][0])[q] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  if (warp == 0) produce<F>(a, rc, S, ring, lane, err);
  else if (warp == kCopierWarp) {
    if (a.readthrough && a.copy_cnt != nullptr) copier(a, S, lane);
  } else {
    consume<F>(a, rc, S, ring, bar, err, warp - 1, lane);
  }
}

// ------------------------------------------------------------------ host
size_t host_row_bytes(int F, int K) {
  return F == MOE_F32 ? (size_t)K * 4
                      : (F == MOE_BF16 ? (size_t)K * 2 : (F == MOE_FP8_E4M3 ? (size_t)K : (size_t)K / 2));
}

// Stage geometry for a shape, or false if the staged kernel cannot take it.
bool ring_geometry(int F, int H, int I, int k, RingCfg* rc, size_t* dyn_smem) {
  if (k < 1 || k > MOE_MAX_TOPK || H < 1) return false;
  const size_t rb1 = host_row_bytes(F, H), rb2 = host_row_bytes(F, I);
  const int el = F == MOE_F32 ? 4 : (F == MOE_BF16 ? 8 : (F == MOE_FP8_E4M3 ? 16 : 32));
  if (H % el || I % el || rb1 % 16 || rb2 % 16) return false;
  const bool q = F == MOE_INT4_G128;
  if (q && (H % 128 || I % 128)) return false;
  // the consumers hold x (H / el chunks) and one part of h (ceil(k * I / el /
  // kParts) chunks) in registers: at most 32 * XM and 32 * HM chunks per warp
  const int xm = q ? RingTile<MOE_INT4_G128>::XM
                   : (F == MOE_FP8_E4M3 ? RingTile<MOE_FP8_E4M3>::XM : RingTile<MOE_BF16>::XM);
  const int hm = q ? RingTile<MOE_INT4_G128>::HM
                   : (F == MOE_FP8_E4M3 ? RingTile<MOE_FP8_E4M3>::HM : RingTile<MOE_BF16>::HM);
  if (H / el > 32 * xm || (k * I / el + kParts - 1) / kParts > 32 * hm) return false;
  const size_t srb1 = q ? (size_t)(H / 128) * 2 : 0, srb2 = q ? (size_t)(I / 128) * 2 : 0;
  // up items of kConsumers pairs (one pair per warp) while they stay small;
  // otherwise half as many (one row per warp), so that more, smaller stages
  // fit and a CTA's whole share of W2 can be in flight before the grid barrier
  int P = kConsumers;
  if ((size_t)2 * P * (rb1 + srb1) > 64 * 1024) P = kConsumers / 2;
  // INT4 / FP8: items of 2 * kConsumers pairs (two pairs per warp) while a stage stays
  // within 64 KiB: a warp's rows of one item are four independent dot
  // products, and half as many items each wait for a stage
  if ((q || F == MOE_FP8_E4M3) && (size_t)2 * (2 * kConsumers) * (rb1 + srb1) <= 64 * 1024 &&
      I % (2 * kConsumers) == 0)
    P = 2 * kConsumers;
  if (I % P) return false;
  size_t sb = (size_t)2 * P * (rb1 + srb1);
  int down_rows, down_group;
  if (q) {
    // 8 rows of bf16 scales per expert and item keep every scale copy 16-byte aligned
    down_group = 8;
    down_rows = 8;
    if (H % 8) return false;
    sb = sb > (size_t)8 * k * (rb2 + srb2) ? sb : (size_t)8 * k * (rb2 + srb2);
  } else {
    down_group = 1;
    if (sb < (size_t)k * rb2) sb = (size_t)k * rb2;
    down_rows = (int)(sb / ((size_t)k * rb2));
    if (down_rows > kConsumers) down_rows = kConsumers;
  }
  sb = (sb + 127) / 128 * 128;
  // static shared memory (the ring starts 1024-byte aligned after it) + reserve
  const size_t fixed = (sizeof(RingShared) + 1023) / 1024 * 1024 + 1024;
  if (fixed + 2 * sb > kSmemLimit) return false;
  size_t ns = (kSmemLimit - fixed) / sb;
  if (ns > (size_t)kMaxStages) ns = kMaxStages;
  rc->up_pairs = P;
  rc->nstages = (int)ns;
  rc->stage_bytes = (unsigned)sb;
  rc->down_rows = down_rows;
  rc->down_group = down_group;
  *dyn_smem = ns * sb;
  return true;
}

// Shared memory the attribute allows and the occupancy at that size, per
// weight format and device (guarded by launch_state_mutex()).
struct RingLaunchState {
  size_t smem = 0;
  int blocks_per_sm = 0;
};
RingLaunchState g_ring_state[4][kMaxDevices];

template <int F>
cudaError_t ring_configure_impl(int H, int I, int k) {
  RingCfg rc;
  size_t smem = 0;
  if (!ring_geometry(F, H, I, k, &rc, &smem)) return cudaSuccess;   // not used for this shape
  device_sm_count();   // cache the SM count outside any capture
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(launch_state_mutex());
  RingLaunchState& st = g_ring_state[F][dev];
  if (st.smem < smem) {
    cudaError_t e = cudaFuncSetAttribute(k_mlp_ring<F>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_mlp_ring<F>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    st.smem = smem;
  }
  int nb = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k_mlp_ring<F>, kRingThreads, smem);
  if (e != cudaSuccess) return e;
  st.blocks_per_sm = nb;
  return cudaSuccess;
}

template <int F>
cudaError_t ring_impl(const MlpArgs& a, GridBar* bar, int* err, cudaStream_t s) {
  RingCfg rc;
  size_t smem = 0;
  if (a.T != 1 || !ring_geometry(F, a.H, a.I, a.k, &rc, &smem)) return cudaErrorNotSupported;
  const int dev = current_device();
  if (dev < 0) return cudaErrorNotSupported;
  {
    std::lock_guard<std::mutex> lock(launch_state_mutex());
    const RingLaunchState& st = g_ring_state[F][dev];
    if (st.smem < smem || st.blocks_per_sm < 1) return cudaErrorNotSupported;
  }
  MlpArgs args = a;
  void* params[] = {&args, &rc, &bar, &err};
  return cudaLaunchCooperativeKernel((const void*)k_mlp_ring<F>, dim3(device_sm_count()), dim3(kRingThreads),
                                     params, smem, s);
}

}  // namespace

size_t mlp_ring_h_floats(int k, int I) { return (size_t)kHRep * k * I; }

cudaError_t mlp_ring_configure(int wdtype, int H, int I, int k) {
  switch (wdtype) {
    case MOE_F32: return ring_configure_impl<MOE_F32>(H, I, k);
    case MOE_BF16: return ring_configure_impl<MOE_BF16>(H, I, k);
    case MOE_INT4_G128: return ring_configure_impl<MOE_INT4_G128>(H, I, k);
    case MOE_FP8_E4M3: return ring_configure_impl<MOE_FP8_E4M3>(H, I, k);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_mlp_ring(int wdtype, const MlpArgs& a, GridBar* bar, int* err, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  switch (wdtype) {
    case MOE_F32: return ring_impl<MOE_F32>(a, bar, err, s);
    case MOE_BF16: return ring_impl<MOE_BF16>(a, bar, err, s);
    case MOE_INT4_G128: return ring_impl<MOE_INT4_G128>(a, bar, err, s);
    case MOE_FP8_E4M3: return ring_impl<MOE_FP8_E4M3>(a, bar, err, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
