// Grouped expert MLP for steps with several tokens per expert (batched
// decode, prefill) on the sm_103a tensor cores, weights on the MMA's N side.
//
// With T tokens and top-k routing there are n = T * k assignments; expert e
// serves the M_e assignments that chose it (vLLM PR #37190 "Run MoE models
// exceeding VRAM via expert CPU offloading with GPU cache", "How it works":
// fused_experts over the remapped ids).  k_group lays the assignments out
// expert by expert and cuts each expert's run into tiles of at most 64;
// k_gather copies the tiles' activation rows into that order.  A work item is
// (tile, WN weight rows), WN = 256 (128 where the shape does not divide):
//   up:   D[128 x WN] = X . [WN/2 gate rows | WN/2 up rows of features f0 ..]^T,
//         epilogue h = w * silu(gate) * up, stored bf16 in tile order;
//   down: D[128 x WN] = H . [WN W2 rows]^T, epilogue: f32 rows per assignment;
// k_combine then sums the k rows of each token in j order.
//
// Why weights on N: on this GPU one tcgen05.mma of kind::f16 (M = 64 or 128,
// K = 16) takes the same time for every N up to 256, so the instruction count
// sets the cost.  With the weights on N one instruction covers 256 weight
// rows, with the tokens (a few to 64 per tile) on M = 128; the rows of M past
// the tile's tokens compute values nobody reads.
//
// Warp roles (16 warps, one CTA per SM, items b, b + G, ... of the grid):
//   warps 0-1  epilogue: tensor-memory lane quadrants 0 and 1 hold the tile's
//              64 token rows of the accumulator (tcgen05.ld), one token a lane;
//   warp 2     TMA producer: per stage (one or two K steps of 64) boxes of the
//              weight rows (bf16, or raw INT4 / FP8 bytes) from tensor maps
//              over the pool and the bypass scratch, and of the tile's
//              activation rows; experts in mapped host memory (the cold set,
//              "Running 125B MoE on Two 32 GB Cards", section 2) are read
//              with plain 16-byte loads instead; per item a record for the
//              other roles and (INT4) a bulk copy of the item's scales;
//   warp 3     MMA issuer: four tcgen05.mma (K = 16) per K step into one of
//              two accumulators in tensor memory;
//   warps 4-15 (INT4 / FP8) three dequantisation groups of four warps; group
//              g turns the raw codes of K steps g, g + 3, ... into a bf16
//              weight tile in shared memory, two rows a thread.
// All hand-offs are mbarriers; no CTA-wide barrier runs inside the item loop.
// Every wait is bounded by the global timer and sets DEVERR_RING when it runs
// out; the other roles then stop at their next wait.
//
// Shared-memory operands are K-major rows of 64 bf16 (128 bytes) in the
// 128-byte swizzle (16-byte chunk c of row r at chunk c ^ (r % 8), 8-row
// groups 1024 bytes apart); raw codes arrive as 64-byte rows in the 64-byte
// swizzle (chunk c of row r at c ^ ((r / 2) % 4)).  Wide rows keep every TMA
// request 64 or 128 bytes long.
//
// Rounding: INT4 weights are dequantised to bf16 once ((q - 8) * scale,
// rounded once), FP8 codes are exact in bf16 and their tensor scales apply in
// the up epilogue, h is rounded to bf16 between the GEMMs; each output element
// is one tensor-core dot product over K whose value does not depend on the
// tile's other tokens.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <new>

#include "internal.cuh"
#include "mlp_common.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace mlp;

constexpr int kDqGroups = 3;           // INT4 / FP8 dequantisation groups of four warps
constexpr int kWProd = 2, kWMma = 3, kWDq = 4;   // warps 0 and 1: epilogue
constexpr int kTWarps = kWDq + 4 * kDqGroups;
constexpr int kTThreads = 32 * kTWarps;
constexpr int kTileTok = 64;           // tokens per tile (MMA M = 128)
constexpr int kM = 128;
constexpr int kKS = 64;                // K elements per K step (one row of 128 bytes)
constexpr int kATile = kTileTok * 128; // activation rows of one K step (8 KB)
constexpr int kAPad = (kM - kTileTok) * 128;   // the MMA reads 128 rows: room past the last activation tile
constexpr int kMaxWN = 256;
constexpr int kMaxStagesT = 8;
constexpr int kRecSlots = 8;           // item records in flight
constexpr int kScSlots = 2;            // INT4: items whose scales are in shared memory
constexpr unsigned long long kTWaitNs = 500000000ull;   // 0.5 s
static_assert(kTWarps * 32 <= 1024, "block size");
static_assert((kWDq & 3) == 0, "a dequantisation group spans the four lane quadrants");

// Per weight format: K steps per stage and raw bytes per weight row and stage
// (0: bf16, whose rows the MMA reads in place)
template <int F>
struct GT;
template <>
struct GT<MOE_BF16> {
  static constexpr int kSub = 1, kRawRow = 0;
};
template <>
struct GT<MOE_INT4_G128> {
  static constexpr int kSub = 2, kRawRow = 64;
};
template <>
struct GT<MOE_FP8_E4M3> {
  static constexpr int kSub = 1, kRawRow = 64;
};
// bytes per weight row in a stage
template <int F>
__host__ __device__ constexpr int wrow_bytes() { return GT<F>::kRawRow ? GT<F>::kRawRow : 128; }
template <int F>
__host__ __device__ constexpr int stage_bytes(int wn) { return wn * wrow_bytes<F>() + GT<F>::kSub * kATile; }

// weight rows per item of a phase: 256 where the rows split evenly, else 128
__host__ __device__ inline int phase_wn(int ph, int H, int I) {
  return ph == 0 ? (I % 128 == 0 ? 256 : 128) : (H % 256 == 0 ? 256 : 128);
}

// Dynamic shared memory of a phase: stages, the pad the MMA may read past the
// last activation tile, the dequantised tiles, the INT4 scale slots.
struct TLayout {
  int ns = 0;              // stages
  int wn = 0;              // weight rows per item
  unsigned sc_bytes = 0;   // INT4 scale bytes per slot
  size_t bytes = 0;
};
template <int F>
bool tma_layout(int ph, int H, int I, size_t budget, TLayout* L) {
  const int wn = phase_wn(ph, H, I);
  const int K = ph == 0 ? H : I;
  const size_t sb = (size_t)stage_bytes<F>(wn);
  const size_t sc = F == MOE_INT4_G128 ? (size_t)wn * (K / 128) * 2 : 0;
  const size_t tiles = F == MOE_BF16 ? 0 : (size_t)kDqGroups * wn * 128;
  const size_t fixed = (size_t)kAPad + tiles + (size_t)kScSlots * sc + 1024;   // + alignment slack
  if (budget < fixed + 2 * sb) return false;
  size_t n = (budget - fixed) / sb;
  if (n > (size_t)kMaxStagesT) n = kMaxStagesT;
  L->ns = (int)n;
  L->wn = wn;
  L->sc_bytes = (unsigned)sc;
  L->bytes = n * sb + fixed;
  return true;
}

enum { PH_UP = 0, PH_DOWN = 1 };
enum { REG_POOL = 0, REG_SCRATCH = 1, REG_NONE = 2 };

// the maps a kernel reads: weights of the pool and the scratch, and the
// activation rows with boxes of 16, 32 and 64 rows
struct TmaMaps {
  CUtensorMap w[2];     // [REG_POOL], [REG_SCRATCH]: weight rows of this phase
  CUtensorMap b[3];     // activations, box rows 16 << i
};

struct TArgs {
  const int32_t* order;        // [n] assignment of each position (expert-major)
  const int4* tiles;           // {first position, rows, expert, 0}
  const int* ntiles;
  const unsigned long long* asg_ptr;
  const float* w;
  int k, H, I;
  unsigned long long off_w2, off_s13, off_s2;
  uint16_t* hb;                // [n, I] bf16 h in position order (up writes, down reads through its map)
  float* out;                  // [n, H] f32 rows per assignment (down)
  // device address ranges of the pool and the scratch: an address a is in
  // region q iff reg_lo <= a < reg_hi and (a - reg_lo) % reg_pitch < reg_part
  // (a layer's device rows, when host rows sit between two layers' pools)
  unsigned long long reg_lo[2], reg_hi[2], reg_pitch[2], reg_part[2];
  int* err;
  const uint8_t* pending;      // [n] or null: the assignment's expert is copied in this step
  const unsigned* ready;       // [E]: ready[e] == hdr->seq once expert e has landed
  const RecHdr* hdr;
  int ns;                      // stages
  int wn;                      // weight rows per item (MMA N)
  unsigned sc_bytes;           // INT4 scale bytes of one slot (wn rows x K / 128 bf16)
};

// What the producer tells the epilogue and the dequantisation warps about an item
struct ItemRec {
  unsigned long long blk;      // expert block (0: the tile's assignments are invalid)
  int4 td;                     // the tile: first position, rows, expert
};

struct TShared {
  unsigned long long full[kMaxStagesT];   // TMA bytes (and the producer's arrive) of a stage
  unsigned long long empty[kMaxStagesT];  // the MMAs that read a stage are done
  unsigned long long tfull[kDqGroups];    // group g filled its bf16 weight tile
  unsigned long long tempty[kDqGroups];   // the MMAs that read it are done
  unsigned long long rfull[kRecSlots];    // item record written
  unsigned long long rempty[kRecSlots];   // read by the epilogue and the dequantisation warps
  unsigned long long sfull[kScSlots];     // INT4 scales of an item landed
  unsigned long long sempty[kScSlots];    // read by the dequantisation warps
  unsigned long long accf[2];             // accumulator b complete
  unsigned long long acce[2];             // accumulator b read by the epilogue
  ItemRec rec[kRecSlots];
  uint32_t tmem;
  int stop;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<unsigned long long>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// contiguous bytes global -> shared (16-byte aligned, a multiple of 16 bytes)
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, unsigned bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// shared-memory descriptor, K-major, 128-byte swizzle: rows of 128 bytes
// (64 bf16 of K), 8-row groups 1024 bytes apart; the K = 16 slice j of the
// rows starts 32 * j bytes in (the swizzle applies to the resulting address)
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;                  // leading byte offset: not used when K fits in the swizzle row
  d |= (uint64_t)(1024u >> 4) << 32;       // stride byte offset
  d |= (uint64_t)1 << 46;                  // descriptor version (tcgen05)
  d |= (uint64_t)2 << 61;                  // 128-byte swizzle
  return d;
}

// physical 16-byte chunk of logical chunk c in row r of a swizzled tile with
// row_bytes-byte rows (the tile starts on a 1024-byte boundary)
__host__ __device__ __forceinline__ int swz_chunk(int c, int r, int row_bytes) {
  return row_bytes == 128 ? (c ^ (r & 7)) : (c ^ ((r >> 1) & 3));
}

__device__ __forceinline__ uint32_t pack_bf16x2_t(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// Eight 4-bit codes (nibble i of wd is element i) -> bf16 (q - 8) * scale in
// element order, two per 32-bit word: a code in the mantissa of a bf16 whose
// exponent is that of 128 is the value 128 + q exactly; subtracting 136 leaves
// q - 8 exactly and the product with the scale is the only rounding.
__device__ __forceinline__ uint4 int4x8_bf16(uint32_t wd, uint32_t scale2) {
  const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162*>(&scale2);
  const uint32_t off_bits = 0x43084308u;   // bf16x2 {136, 136}
  const __nv_bfloat162 off = *reinterpret_cast<const __nv_bfloat162*>(&off_bits);
  uint32_t v[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t p = ((wd >> (4 * j)) & 0x000F000Fu) | 0x43004300u;   // {128 + q_j, 128 + q_j+4}
    const __nv_bfloat162 d = __hmul2(__hsub2(*reinterpret_cast<const __nv_bfloat162*>(&p), off), s2);
    v[j] = *reinterpret_cast<const uint32_t*>(&d);
  }
  return make_uint4(__byte_perm(v[0], v[1], 0x5410), __byte_perm(v[2], v[3], 0x5410),
                    __byte_perm(v[0], v[1], 0x7632), __byte_perm(v[2], v[3], 0x7632));
}

// Eight E4M3 codes (byte i of the pair of words is element i) -> bf16, exact
__device__ __forceinline__ uint4 fp8x8_bf16(uint32_t w0, uint32_t w1) {
  const float2 a = e4m3x2_to_f2(w0), b = e4m3x2_to_f2(w0 >> 16), c = e4m3x2_to_f2(w1), d = e4m3x2_to_f2(w1 >> 16);
  return make_uint4(pack_bf16x2_t(a.x, a.y), pack_bf16x2_t(b.x, b.y), pack_bf16x2_t(c.x, c.y),
                    pack_bf16x2_t(d.x, d.y));
}

// The item's weight rows: row of tile row r (0 .. wn - 1) in the expert block
template <int PH>
__device__ __forceinline__ int wrow_of(int r, int mt, int I, int wn) {
  const int half = wn >> 1;
  return PH == PH_UP ? (r < half ? mt * half + r : I + mt * half + (r - half)) : mt * wn + r;
}

// Pauses between tries of a wait, by role: the MMA issuer is on the critical
// path and retries at once; the others sleep a little so that waiting warps
// leave the issue slots to the dequantisation warps.
constexpr unsigned kSleepNone = 0, kSleepShort = 64, kSleepLong = 256;

// bounded wait; on a time-out flags the error and asks every role to stop
__device__ __forceinline__ bool wait_or_stop(TShared& S, uint32_t bar, unsigned parity, int* err,
                                             unsigned sleep_ns = kSleepNone) {
  if (*reinterpret_cast<volatile int*>(&S.stop)) return false;
  if (tc::mbar_wait(bar, parity, kTWaitNs, sleep_ns)) return true;
  atomicExch(err, DEVERR_RING);
  *reinterpret_cast<volatile int*>(&S.stop) = 1;
  return false;
}
// lane 0 waits, the warp follows (memory ordering through the warp barrier)
__device__ __forceinline__ bool warp_wait(TShared& S, uint32_t bar, unsigned parity, int* err, int lane,
                                          unsigned sleep_ns) {
  bool ok = true;
  if (lane == 0) ok = wait_or_stop(S, bar, parity, err, sleep_ns);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok;
}

template <int F, int PH>
__global__ void __launch_bounds__(kTThreads, 1)
    k_moe_gemm_tma(const __grid_constant__ TmaMaps maps, TArgs g) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ TShared S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool kDq = F != MOE_BF16;
  constexpr int kSub = GT<F>::kSub;               // K steps per stage
  constexpr int RB = wrow_bytes<F>();             // bytes per weight row in a stage
  constexpr unsigned kRecReaders = 2 + (kDq ? 4 * kDqGroups : 0);
  const int NS = g.ns;
  const int WN = g.wn;
  const int SB = stage_bytes<F>(WN);
  const int WB = WN * RB;                         // weight part of a stage
  uint8_t* base = smem + ((1024u - (tc::smem_u32(smem) & 1023u)) & 1023u);
  uint8_t* tiles = base + (size_t)NS * SB + kAPad;                                  // [kDqGroups][WN rows x 128 B]
  uint8_t* scb = tiles + (kDq ? (size_t)kDqGroups * WN * 128 : 0);                  // [kScSlots][sc_bytes]
  const int K = PH == PH_UP ? g.H : g.I;
  const int nk = K / kKS;
  const int NT = PH == PH_UP ? g.I / (WN >> 1) : g.H / WN;
  const int ntiles = *g.ntiles;
  const int items = ntiles * NT;
  const size_t wrb = F == MOE_BF16 ? (size_t)K * 2 : (F == MOE_FP8_E4M3 ? (size_t)K : (size_t)K / 2);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(tc::smem_u32(&S.full[s]), 1u);
      tc::mbar_init(tc::smem_u32(&S.empty[s]), 1u);
    }
    for (int b = 0; b < kDqGroups; ++b) {
      tc::mbar_init(tc::smem_u32(&S.tfull[b]), 4u);
      tc::mbar_init(tc::smem_u32(&S.tempty[b]), 1u);
    }
    for (int b = 0; b < kRecSlots; ++b) {
      tc::mbar_init(tc::smem_u32(&S.rfull[b]), 1u);
      tc::mbar_init(tc::smem_u32(&S.rempty[b]), kRecReaders);
    }
    for (int b = 0; b < kScSlots; ++b) {
      tc::mbar_init(tc::smem_u32(&S.sfull[b]), 1u);
      tc::mbar_init(tc::smem_u32(&S.sempty[b]), 4u * kDqGroups);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(tc::smem_u32(&S.accf[b]), 1u);
      tc::mbar_init(tc::smem_u32(&S.acce[b]), 2u);
    }
    S.stop = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kWMma) tc::tmem_alloc(tc::smem_u32(&S.tmem), 2u * kMaxWN);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = S.tmem;

  if (warp == kWProd) {
    // ------------------------------------------------------------ producer
    unsigned gst = 0;   // stages issued
    int it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < items && ok; item += gridDim.x, ++it) {
      const int tile = item / NT, mt = item - tile * NT;
      const int4 td = g.tiles[tile];
      const int asg0 = g.order[td.x];
      const unsigned long long blk = g.asg_ptr[asg0];
      const unsigned long long wblk = blk + (PH == PH_UP ? 0ull : g.off_w2);
      int reg = REG_NONE;
      for (int q = 0; q < 2; ++q)
        if (blk >= g.reg_lo[q] && blk < g.reg_hi[q] && (blk - g.reg_lo[q]) % g.reg_pitch[q] < g.reg_part[q] &&
            ((wblk - g.reg_lo[q]) % wrb) == 0ull)
          reg = q;
      const int row_base = reg == REG_NONE ? 0 : (int)((wblk - g.reg_lo[reg]) / wrb);
      // tile rows -> the smallest activation box that holds them
      const int bi = td.y <= 16 ? 0 : (td.y <= 32 ? 1 : 2);
      const int brows = 16 << bi;
      if (PH == PH_UP && g.pending != nullptr && g.pending[asg0] != 0 && lane == 0) {
        // the expert is being copied in this step: wait (bounded) until its copy is published
        const unsigned want = g.hdr->seq;
        const unsigned long long t0 = tc::global_ns();
        for (;;) {
          unsigned v;
          asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(g.ready + td.z) : "memory");
          if (v == want) break;
          if (tc::global_ns() - t0 > 2000000000ull) {
            atomicExch(g.err, DEVERR_RING);
            S.stop = 1;
            ok = false;
            break;
          }
          __nanosleep(256);
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");   // copy-kernel stores -> TMA reads
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      // the item's record for the epilogue and the dequantisation warps
      const int rsl = it % kRecSlots;
      if (it >= kRecSlots &&
          !warp_wait(S, tc::smem_u32(&S.rempty[rsl]), ((it / kRecSlots) - 1) & 1, g.err, lane, kSleepLong)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        S.rec[rsl].blk = blk;
        S.rec[rsl].td = td;
        mbar_arrive(tc::smem_u32(&S.rfull[rsl]));
      }
      if (F == MOE_INT4_G128) {
        // the scales of the item's WN rows, K / 128 bf16 per row: up = WN/2
        // gate rows from mt * WN/2 and WN/2 up rows from I + mt * WN/2;
        // down = WN rows from mt * WN
        const int ssl = it % kScSlots;
        if (it >= kScSlots &&
            !warp_wait(S, tc::smem_u32(&S.sempty[ssl]), ((it / kScSlots) - 1) & 1, g.err, lane, kSleepShort)) {
          ok = false;
          break;
        }
        const uint32_t sfull = tc::smem_u32(&S.sfull[ssl]);
        if (blk != 0ull) {
          const int gpr = K / 128;
          const int half = WN >> 1;
          const uint8_t* s0 = reinterpret_cast<const uint8_t*>(blk + (PH == PH_UP ? g.off_s13 : g.off_s2));
          const uint8_t* src0 = s0 + (size_t)(PH == PH_UP ? mt * half : mt * WN) * gpr * 2;
          const uint8_t* src1 = s0 + (size_t)(g.I + mt * half) * gpr * 2;
          const unsigned chunk = (unsigned)((PH == PH_UP ? half : WN) * gpr * 2);
          uint8_t* dst = scb + (size_t)ssl * g.sc_bytes;
          const bool bulk = reg != REG_NONE &&
                            ((reinterpret_cast<uintptr_t>(src0) | reinterpret_cast<uintptr_t>(src1)) & 15u) == 0;
          if (bulk) {
            if (lane == 0) {
              mbar_arrive_tx(sfull, PH == PH_UP ? 2 * chunk : chunk);
              bulk_g2s(tc::smem_u32(dst), src0, chunk, sfull);
              if (PH == PH_UP) bulk_g2s(tc::smem_u32(dst) + chunk, src1, chunk, sfull);
            }
          } else {
            for (unsigned v = (unsigned)lane * 2; v < chunk; v += 64) {
              *reinterpret_cast<uint16_t*>(dst + v) = __ldcg(reinterpret_cast<const uint16_t*>(src0 + v));
              if (PH == PH_UP)
                *reinterpret_cast<uint16_t*>(dst + chunk + v) = __ldcg(reinterpret_cast<const uint16_t*>(src1 + v));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sfull);
          }
        } else {
          __syncwarp();
          if (lane == 0) mbar_arrive(sfull);
        }
      }
      for (int kt = 0; kt < nk / kSub; ++kt, ++gst) {
        const int s = (int)(gst % (unsigned)NS);
        if (gst >= (unsigned)NS &&
            !warp_wait(S, tc::smem_u32(&S.empty[s]), ((gst / NS) - 1u) & 1u, g.err, lane, kSleepShort)) {
          ok = false;
          break;
        }
        uint8_t* st = base + (size_t)s * SB;
        const uint32_t w_u = tc::smem_u32(st), a_u = w_u + (uint32_t)WB;
        const uint32_t full = tc::smem_u32(&S.full[s]);
        const int k0 = kt * kSub * kKS;                 // first K element of the stage
        const unsigned abytes = (unsigned)(kSub * brows * 128);
        const unsigned wbytes = reg == REG_NONE ? 0u : (unsigned)WB;
        if (reg == REG_NONE && blk != 0ull) {
          // weights in host memory (or not addressable through a map): plain
          // loads, stored in the layout the TMA would write
          const uint8_t* wb = reinterpret_cast<const uint8_t*>(wblk);
          constexpr int cpr = RB / 16;
          for (int v = lane; v < WN * cpr; v += 32) {
            const int r = v / cpr, c = v - r * cpr;
            const uint4 q = __ldcg(reinterpret_cast<const uint4*>(
                wb + (size_t)wrow_of<PH>(r, mt, g.I, WN) * wrb + (kDq ? (size_t)kt * RB : (size_t)k0 * 2) + c * 16));
            *reinterpret_cast<uint4*>(st + (size_t)r * RB + swz_chunk(c, r, RB) * 16) = q;
          }
          if (!kDq) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic stores -> MMA reads
          __syncwarp();
        }
        if (lane == 0) mbar_arrive_tx(full, abytes + wbytes);
        __syncwarp();
        // activation rows of the tile: one box of brows x 64 elements per K step
        if (lane < kSub) tma_load_2d(a_u + (uint32_t)lane * kATile, &maps.b[bi], k0 + kKS * lane, td.x, full);
        if (reg != REG_NONE) {
          const CUtensorMap* wm = &maps.w[reg];
          const int x = kDq ? kt * RB : k0;             // bytes of raw codes, or bf16 elements
          const int half = WN >> 1;
          if (PH == PH_UP) {
            // WN/2 gate rows, then WN/2 up rows of features mt * WN/2 ..
            if (lane == 8) tma_load_2d(w_u, wm, x, row_base + mt * half, full);
            if (lane == 9) tma_load_2d(w_u + (uint32_t)(half * RB), wm, x, row_base + g.I + mt * half, full);
          } else {
            if (lane == 8) tma_load_2d(w_u, wm, x, row_base + mt * WN, full);
          }
        }
      }
    }
  } else if (warp == kWMma) {
    // ----------------------------------------------------------------- MMA
    const uint32_t idesc = tc::idesc_bf16(kM, (uint32_t)WN);
    unsigned gs = 0;   // K steps issued
    int it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < items && ok; item += gridDim.x, ++it) {
      const int buf = it & 1;
      if (it >= 2 && !warp_wait(S, tc::smem_u32(&S.acce[buf]), ((it >> 1) - 1) & 1, g.err, lane, kSleepNone)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t d_tmem = tmem + (uint32_t)(buf * kMaxWN);
      for (int ks = 0; ks < nk; ++ks, ++gs) {
        const unsigned gt = gs / kSub;                 // its stage
        const int u = (int)(gs % kSub);
        const int s = (int)(gt % (unsigned)NS);
        const int tb = (int)(gs % kDqGroups);
        if (lane == 0) {
          ok = wait_or_stop(S, tc::smem_u32(&S.full[s]), (gt / NS) & 1u, g.err);
          if (ok && kDq) ok = wait_or_stop(S, tc::smem_u32(&S.tfull[tb]), (gs / kDqGroups) & 1u, g.err);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc::fence_after_sync();
        if (lane == 0) {
          const uint32_t st_u = tc::smem_u32(base + (size_t)s * SB);
          const uint32_t a_u = st_u + (uint32_t)WB + (uint32_t)(u * kATile);
          const uint32_t b_u = kDq ? tc::smem_u32(tiles + (size_t)tb * WN * 128) : st_u;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc::mma_bf16(d_tmem, desc_sw128(a_u + (uint32_t)j * 32u), desc_sw128(b_u + (uint32_t)j * 32u), idesc,
                         (ks | j) != 0 ? 1u : 0u);
          if (u == kSub - 1) tc::mma_commit(tc::smem_u32(&S.empty[s]));   // the stage's last K step
          if (kDq) tc::mma_commit(tc::smem_u32(&S.tempty[tb]));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc::mma_commit(tc::smem_u32(&S.accf[buf]));
      __syncwarp();
    }
    // every MMA issued has completed before tensor memory is freed
    if (gs > 0 && lane == 0) {
      const unsigned last = (gs - 1u) / kSub;          // the last stage
      tc::mbar_wait(tc::smem_u32(&S.empty[last % (unsigned)NS]), (last / NS) & 1u, kTWaitNs);
    }
    __syncwarp();
  } else if (warp >= kWDq) {
    // ------------------------------------------------- dequantisation warps
    // group grp takes the K steps q with q % kDqGroups == grp and writes them
    // into its bf16 tile; warp w of the group converts rows w * WN / 4 ..,
    // WN / 128 a thread
    if (kDq) {
      const int grp = (warp - kWDq) >> 2;
      const int wq = (warp - kWDq) & 3;
      const int gpr = K / 128;                              // INT4 scale groups per row
      uint8_t* tile_g = tiles + (size_t)grp * WN * 128;
      unsigned gs = 0;
      int it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < items && ok; item += gridDim.x, ++it) {
        const int rsl = it % kRecSlots, ssl = it % kScSlots;
        if (!warp_wait(S, tc::smem_u32(&S.rfull[rsl]), (it / kRecSlots) & 1, g.err, lane, kSleepShort)) {
          ok = false;
          break;
        }
        const unsigned long long blk = S.rec[rsl].blk;
        __syncwarp();
        if (lane == 0) mbar_arrive(tc::smem_u32(&S.rempty[rsl]));
        if (F == MOE_INT4_G128 &&
            !warp_wait(S, tc::smem_u32(&S.sfull[ssl]), (it / kScSlots) & 1, g.err, lane, kSleepShort)) {
          ok = false;
          break;
        }
        const uint16_t* sct = reinterpret_cast<const uint16_t*>(scb + (size_t)ssl * g.sc_bytes);
        for (int ks = (int)((unsigned)(grp + kDqGroups) - gs % kDqGroups) % kDqGroups; ks < nk; ks += kDqGroups) {
          const unsigned q = gs + (unsigned)ks;        // K step; stage q / kSub, part q % kSub
          const unsigned qt = q / kSub;
          const int u = (int)(q % kSub);
          const int s = (int)(qt % (unsigned)NS);
          if (lane == 0) {
            ok = wait_or_stop(S, tc::smem_u32(&S.full[s]), (qt / NS) & 1u, g.err, kSleepShort);
            // the tile free: the MMAs that read its previous contents are done
            if (ok && q >= (unsigned)kDqGroups)
              ok = wait_or_stop(S, tc::smem_u32(&S.tempty[grp]), ((q / kDqGroups) - 1u) & 1u, g.err, kSleepShort);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          __syncwarp();
          if (blk != 0ull) {
            const uint8_t* st = base + (size_t)s * SB;
#pragma unroll 1
            for (int h = 0; h < WN / 128; ++h) {
              const int r = wq * (WN / 4) + h * 32 + lane;   // weight row of the item (< WN)
              const uint8_t* raw = st + (size_t)r * RB;
              uint4 o[8];
              if (F == MOE_INT4_G128) {
                const uint32_t sb = sct[(size_t)r * gpr + (ks >> 1)];
                const uint32_t s2 = sb | (sb << 16);
                const uint4 q0 = reinterpret_cast<const uint4*>(raw)[swz_chunk(2 * u, r, RB)];
                const uint4 q1 = reinterpret_cast<const uint4*>(raw)[swz_chunk(2 * u + 1, r, RB)];
                o[0] = int4x8_bf16(q0.x, s2);
                o[1] = int4x8_bf16(q0.y, s2);
                o[2] = int4x8_bf16(q0.z, s2);
                o[3] = int4x8_bf16(q0.w, s2);
                o[4] = int4x8_bf16(q1.x, s2);
                o[5] = int4x8_bf16(q1.y, s2);
                o[6] = int4x8_bf16(q1.z, s2);
                o[7] = int4x8_bf16(q1.w, s2);
              } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                  const uint4 v = reinterpret_cast<const uint4*>(raw)[swz_chunk(c, r, RB)];
                  o[2 * c] = fp8x8_bf16(v.x, v.y);
                  o[2 * c + 1] = fp8x8_bf16(v.z, v.w);
                }
              }
              uint8_t* trow = tile_g + (size_t)r * 128;
#pragma unroll
              for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(trow + swz_chunk(c, r, 128) * 16) = o[c];
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic stores -> MMA reads
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(tc::smem_u32(&S.tfull[grp]));
        }
        if (!ok) break;
        gs += (unsigned)nk;
        if (F == MOE_INT4_G128) {
          __syncwarp();
          if (lane == 0) mbar_arrive(tc::smem_u32(&S.sempty[ssl]));
        }
      }
    }
  } else if (warp < 2) {
    // ------------------------------------------------------------ epilogue
    // warp q reads lane quadrant q of the accumulator: token rows 32 q .. 32 q + 31
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int half = WN >> 1;
    int it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < items && ok; item += gridDim.x, ++it) {
      const int mt = item % NT;
      const int rsl = it % kRecSlots;
      if (!warp_wait(S, tc::smem_u32(&S.rfull[rsl]), (it / kRecSlots) & 1, g.err, lane, kSleepLong)) {
        ok = false;
        break;
      }
      const int4 td = S.rec[rsl].td;
      const unsigned long long blk = S.rec[rsl].blk;
      __syncwarp();
      if (lane == 0) mbar_arrive(tc::smem_u32(&S.rempty[rsl]));
      const int t = warp * 32 + lane;                  // token row of the tile
      const bool valid = t < td.y;
      const int pos = td.x + t;
      const int a = valid ? g.order[pos] : 0;          // the row's assignment
      const int buf = it & 1;
      float fsg = 1.f, fsu = 1.f, fsd = 1.f;           // FP8: the expert's gate, up and down tensor scales
      float wa = 0.f;
      if (PH == PH_UP) {
        if (valid && blk != 0ull) wa = g.w[a];
        if (F == MOE_FP8_E4M3 && blk != 0ull) {
          if (g.pending != nullptr && g.pending[g.order[td.x]] != 0) {
            // the expert was copied in this step: its published flag before its scales
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(g.ready + td.z) : "memory");
          }
          const float* f13 = reinterpret_cast<const float*>(blk + g.off_s13);
          fsg = __ldcg(f13);
          fsu = __ldcg(f13 + 1);
          fsd = __ldcg(reinterpret_cast<const float*>(blk + g.off_s2));
        }
      }
      if (!warp_wait(S, tc::smem_u32(&S.accf[buf]), (it >> 1) & 1, g.err, lane, kSleepLong)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t acc = tmem + lane_base + (uint32_t)(buf * kMaxWN);
      if (PH == PH_UP) {
        // columns c (gate of feature mt * half + c) and half + c (its up)
        __nv_bfloat16* hrow = reinterpret_cast<__nv_bfloat16*>(g.hb) + (size_t)pos * g.I + mt * half;
        for (int c0 = 0; c0 < half; c0 += 16) {
          uint32_t gv[16], uv[16];
          tc::tmem_ld16(acc + (uint32_t)c0, gv);
          tc::tmem_ld16(acc + (uint32_t)(half + c0), uv);
          if (valid) {
            uint32_t pk[8];
#pragma unroll
            for (int c = 0; c < 16; c += 2) {
              float hv[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float gg = __uint_as_float(gv[c + e]) * fsg, uu = __uint_as_float(uv[c + e]) * fsu;
                hv[e] = blk != 0ull ? wa * (gg / (1.0f + expf(-gg)) * uu) * fsd : 0.f;
              }
              pk[c >> 1] = pack_bf16x2_t(hv[0], hv[1]);
            }
            uint4* dst = reinterpret_cast<uint4*>(hrow + c0);
#pragma unroll
            for (int v = 0; v < 2; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      } else {
        float* orow = g.out + (size_t)a * g.H + (size_t)mt * WN;
        for (int c0 = 0; c0 < WN; c0 += 32) {
          uint32_t v[32];
          tc::tmem_ld32(acc + (uint32_t)c0, v);
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(orow + c0);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = blk != 0ull ? make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(tc::smem_u32(&S.acce[buf]));
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kWMma) tc::tmem_free(tmem, 2u * kMaxWN);
}

// positions -> activation rows: xg[p] = x[order[p] / k] (bf16, H per row),
// for the positions k_group filled in this step (a step with invalid ids
// fills fewer than n; entries past them are left from earlier steps)
__global__ void __launch_bounds__(256) k_gather_x(const int32_t* __restrict__ order, const int4* __restrict__ tiles,
                                                  const int* __restrict__ ntiles, const uint4* __restrict__ x,
                                                  uint4* __restrict__ xg, int n, int k, int H) {
  const int nt = *ntiles;
  const int4 last = nt > 0 ? tiles[nt - 1] : make_int4(0, 0, 0, 0);
  const int filled = nt > 0 ? last.x + last.y : 0;
  const int vpr = H / 8;   // 16-byte vectors per row
  const long long total = (long long)filled * vpr;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(i / vpr), v = (int)(i - (long long)p * vpr);
    const int a = order[p];
    if (a >= 0 && a < n) xg[i] = x[(size_t)(a / k) * vpr + v];
  }
}

// ------------------------------------------------------------------ host

struct TLaunchState {
  bool configured = false;
  size_t budget = 0;   // dynamic shared memory a CTA may use
};
TLaunchState g_tma_state[4][kMaxDevices];

template <int F>
cudaError_t tma_configure_impl() {
  device_sm_count();
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(launch_state_mutex());
  TLaunchState& st = g_tma_state[F][dev];
  if (st.configured) return cudaSuccess;
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  const void* kernels[] = {(const void*)k_moe_gemm_tma<F, PH_UP>, (const void*)k_moe_gemm_tma<F, PH_DOWN>};
  size_t static_bytes = 0;
  for (const void* kf : kernels) {
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, kf);
    if (e != cudaSuccess) return e;
    if (fa.sharedSizeBytes > static_bytes) static_bytes = fa.sharedSizeBytes;
  }
  if ((size_t)optin <= static_bytes) return cudaErrorNotSupported;
  const size_t budget = (size_t)optin - static_bytes;
  for (const void* kf : kernels) {
    e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)budget);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kf, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  st.budget = budget;
  st.configured = true;
  return cudaSuccess;
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static bool tried = false;
  std::lock_guard<std::mutex> lock(launch_state_mutex());
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

// rows x cols elements of `dtype` (elem bytes) at `base`, row pitch `pitch`
// bytes, boxes of box_rows x box_cols
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dtype, const void* base, unsigned long long rows,
               unsigned long long cols, unsigned long long pitch, unsigned box_rows, unsigned box_cols,
               CUtensorMapSwizzle swz) {
  EncodeFn fn = encode_fn();
  if (!fn || rows == 0 || cols == 0 || rows > (1ull << 32) || cols > (1ull << 32) || pitch % 16 ||
      (reinterpret_cast<uintptr_t>(base) & 15))
    return false;
  const cuuint64_t dim[2] = {cols, rows};
  const cuuint64_t stride[1] = {pitch};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dtype, 2, const_cast<void*>(base), dim, stride, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

struct MoeTmaMaps {
  TmaMaps up, down;
  bool ok = false;
};

bool moe_gemm_tma_supported(int wdtype, int H, int I, int k) {
  if (wdtype != MOE_BF16 && wdtype != MOE_INT4_G128 && wdtype != MOE_FP8_E4M3) return false;
  if (k < 1 || k > MOE_MAX_TOPK || H % 128 || I % 64) return false;
  if (wdtype == MOE_INT4_G128 && I % 128) return false;   // stages of two K steps, scale groups of 128
  // shared memory of a GB300 CTA (227 KB) less a margin for the static part
  constexpr size_t kBudget = 232448 - 4096;
  TLayout up, dn;
  switch (wdtype) {
    case MOE_BF16:
      return tma_layout<MOE_BF16>(0, H, I, kBudget, &up) && tma_layout<MOE_BF16>(1, H, I, kBudget, &dn);
    case MOE_INT4_G128:
      return tma_layout<MOE_INT4_G128>(0, H, I, kBudget, &up) && tma_layout<MOE_INT4_G128>(1, H, I, kBudget, &dn);
    case MOE_FP8_E4M3:
      return tma_layout<MOE_FP8_E4M3>(0, H, I, kBudget, &up) && tma_layout<MOE_FP8_E4M3>(1, H, I, kBudget, &dn);
  }
  return false;
}

// Tensor maps over the weight regions (the pool of every layer and the bypass
// scratch) and over the position-ordered activation buffers.  Weights are
// addressed as rows of the phase's K: the maps cover each region as a matrix
// of such rows, so an expert block's rows are found from its offset in the
// region (the kernel checks that the offset is a whole number of rows).
MoeTmaMaps* moe_gemm_tma_maps(int wdtype, int H, int I, const void* pool, size_t pool_bytes, const void* scratch,
                              size_t scratch_bytes, const void* xg, const void* hb, size_t n_rows) {
  MoeTmaMaps* m = new (std::nothrow) MoeTmaMaps();
  if (!m) return nullptr;
  const bool bf = wdtype == MOE_BF16;
  const CUtensorMapDataType wt = bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  // boxes of 64 columns: bf16 rows of 128 bytes (128-byte swizzle), or 64
  // bytes of raw codes (64-byte swizzle: two INT4 or one FP8 K step)
  const CUtensorMapSwizzle wsw = bf ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  bool ok = true;
  for (int ph = 0; ph < 2; ++ph) {
    const unsigned long long K = ph == 0 ? (unsigned long long)H : (unsigned long long)I;
    const unsigned long long rb = bf ? K * 2 : (wdtype == MOE_FP8_E4M3 ? K : K / 2);
    const unsigned long long cols = bf ? K : rb;
    // up: the gate (or up) half of an item's weight rows; down: all of them
    const unsigned box_rows = ph == 0 ? (unsigned)phase_wn(0, H, I) / 2 : (unsigned)phase_wn(1, H, I);
    const unsigned box_cols = 64;
    TmaMaps& t = ph == 0 ? m->up : m->down;
    const void* regs[2] = {pool, scratch};
    const size_t bytes[2] = {pool_bytes, scratch_bytes};
    for (int q = 0; q < 2; ++q) {
      const unsigned long long rows = bytes[q] / rb;
      if (regs[q] == nullptr || rows < box_rows) {
        // a region that does not exist (or holds less than a box): a map of
        // one box over the other region, never used (no block lies in it)
        const int o = 1 - q;
        ok = ok && regs[o] != nullptr && bytes[o] / rb >= box_rows &&
             encode_2d(&t.w[q], wt, regs[o], box_rows, cols, rb, box_rows, box_cols, wsw);
      } else {
        ok = ok && encode_2d(&t.w[q], wt, regs[q], rows, cols, rb, box_rows, box_cols, wsw);
      }
    }
    const void* act = ph == 0 ? xg : hb;
    for (int i = 0; i < 3; ++i)
      ok = ok && n_rows >= kTileTok && encode_2d(&t.b[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, act, n_rows, K, K * 2,
                                                 16u << i, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  m->ok = ok;
  return m;
}

void moe_gemm_tma_maps_free(MoeTmaMaps* m) { delete m; }

bool moe_gemm_tma_maps_ok(const MoeTmaMaps* m) { return m != nullptr && m->ok; }

cudaError_t moe_gemm_tma_configure(int wdtype) {
  switch (wdtype) {
    case MOE_BF16: return tma_configure_impl<MOE_BF16>();
    case MOE_INT4_G128: return tma_configure_impl<MOE_INT4_G128>();
    case MOE_FP8_E4M3: return tma_configure_impl<MOE_FP8_E4M3>();
  }
  return cudaErrorNotSupported;
}

namespace {
template <int F>
cudaError_t tma_impl(const MlpArgs& a, const GemmBuffers& b, const MoeTmaMaps& m, const TmaRegions& r, cudaStream_t s) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorNotSupported;
  size_t budget = 0;
  {
    std::lock_guard<std::mutex> lock(launch_state_mutex());
    if (!g_tma_state[F][dev].configured) return cudaErrorNotSupported;
    budget = g_tma_state[F][dev].budget;
  }
  TLayout lu, ld;
  if (!tma_layout<F>(PH_UP, a.H, a.I, budget, &lu) || !tma_layout<F>(PH_DOWN, a.H, a.I, budget, &ld))
    return cudaErrorNotSupported;
  const int n = a.T * a.k;
  cudaError_t e = launch_group(b.ids, n, b.E, b.order, b.tiles, b.ntiles, b.work, kTileTok, s);
  if (e != cudaSuccess) return e;
  const int sms = device_sm_count();
  k_gather_x<<<sms * 4, 256, 0, s>>>(b.order, b.tiles, b.ntiles, reinterpret_cast<const uint4*>(a.x),
                                     reinterpret_cast<uint4*>(r.xg), n, a.k, a.H);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  TArgs g{};
  g.order = b.order;
  g.tiles = b.tiles;
  g.ntiles = b.ntiles;
  g.asg_ptr = a.asg_ptr;
  g.w = a.w;
  g.k = a.k;
  g.H = a.H;
  g.I = a.I;
  g.off_w2 = a.off_w2;
  g.off_s13 = a.off_s13;
  g.off_s2 = a.off_s2;
  g.hb = b.hb;
  g.out = b.out;
  g.reg_lo[0] = r.pool_lo;
  g.reg_hi[0] = r.pool_hi;
  g.reg_pitch[0] = r.pool_pitch ? r.pool_pitch : 1ull;
  g.reg_part[0] = r.pool_part;
  g.reg_lo[1] = r.scratch_lo;
  g.reg_hi[1] = r.scratch_hi;
  g.reg_pitch[1] = r.scratch_hi > r.scratch_lo ? r.scratch_hi - r.scratch_lo : 1ull;
  g.reg_part[1] = r.scratch_hi - r.scratch_lo;
  g.err = b.err;
  g.pending = b.pending;
  g.ready = b.ready;
  g.hdr = b.hdr;
  g.ns = lu.ns;
  g.wn = lu.wn;
  g.sc_bytes = lu.sc_bytes;
  k_moe_gemm_tma<F, PH_UP><<<sms, kTThreads, lu.bytes, s>>>(m.up, g);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  g.pending = nullptr;   // every expert has landed before the up kernel ended
  g.ns = ld.ns;
  g.wn = ld.wn;
  g.sc_bytes = ld.sc_bytes;
  k_moe_gemm_tma<F, PH_DOWN><<<sms, kTThreads, ld.bytes, s>>>(m.down, g);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_combine(F, b.out, a.x, a.y, a.T, a.k, a.H, a.residual, s);
}
}  // namespace

cudaError_t launch_moe_gemm_tma(int wdtype, const MlpArgs& a, const GemmBuffers& b, const MoeTmaMaps* m,
                                const TmaRegions& r, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (m == nullptr || !m->ok || !moe_gemm_tma_supported(wdtype, a.H, a.I, a.k) || a.x == nullptr || r.xg == nullptr)
    return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(a.x) | reinterpret_cast<uintptr_t>(a.y)) & 15) return cudaErrorNotSupported;
  switch (wdtype) {
    case MOE_BF16: return tma_impl<MOE_BF16>(a, b, *m, r, s);
    case MOE_INT4_G128: return tma_impl<MOE_INT4_G128>(a, b, *m, r, s);
    case MOE_FP8_E4M3: return tma_impl<MOE_FP8_E4M3>(a, b, *m, r, s);
  }
  return cudaErrorNotSupported;
}

}  // namespace moe
