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
//   up:   D[64 x WN] = X . [WN/2 gate rows | WN/2 up rows of features f0 ..]^T,
//         epilogue h = w * silu(gate) * up, stored bf16 in tile order;
//   down: D[64 x WN] = H . [WN W2 rows]^T, epilogue: f32 rows per assignment;
// k_combine then sums the k rows of each token in j order.
//
// Why weights on N: on this GPU one tcgen05.mma of kind::f16 (M = 64 or 128,
// K = 16) takes the same time for every N up to 256, so the instruction count
// sets the cost.  With the weights on N one instruction covers 256 weight
// rows, with the tile's tokens (a few to 64) on M = 64.
//
// Warp roles (19 warps, one CTA per SM, items b, b + G, ... of the grid):
//   warps 0-3  epilogue: with M = 64 the accumulator's row 16 q + i sits in
//              tensor-memory lane 32 q + i, so warp q reads 16 token rows;
//   warp 4     weight producer: per item a record for the other roles and
//              (INT4) a bulk copy of the item's scales; bf16 weight tiles, or
//              stages of raw INT4 / FP8 codes, by cp.async.bulk.tensor from
//              tensor maps over the pool and the bypass scratch; experts in
//              mapped host memory (the cold set, "Running 125B MoE on Two
//              32 GB Cards", section 2) are read with plain 16-byte loads;
//   warp 5     activation producer: the tile's activation rows, one K step a box;
//   warp 6     MMA issuer: four tcgen05.mma (K = 16) per K step into one of
//              two accumulators in tensor memory;
//   warps 7-18 (INT4 / FP8) three dequantisation groups of four warps; group
//              g turns the raw codes of K steps g, g + 3, ... into a bf16
//              weight tile in the MMA's layout (a ring of four tiles).
// Weight tiles, raw stages and activation tiles are three rings, each freed
// by its own reader, so raw codes stream ahead of the dequantisation and the
// dequantisation ahead of the MMA.
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
// warps 0-3: epilogue (tensor-memory lane quadrants 0-3)
constexpr int kWProdW = 4, kWProdA = 5, kWMma = 6, kWDq = 7;
constexpr int kTWarps = kWDq + 4 * kDqGroups;
constexpr int kTThreads = 32 * kTWarps;
constexpr int kTileTok = 64;           // tokens per tile (MMA M = 64)
constexpr int kM = 64;
constexpr int kKS = 64;                // K elements per K step
constexpr int kATile = kTileTok * 128; // activation rows of one K step: 64 rows of 128 bytes (8 KB)
constexpr int kARing = 4;              // activation tiles in flight
constexpr int kMaxWN = 256;
constexpr int kMaxTiles = 8;           // weight tiles (bf16, in the MMA's layout)
constexpr int kMaxRaw = 8;             // raw-code stages (INT4 / FP8)
constexpr int kRecSlots = 8;           // item records in flight
constexpr int kScSlots = 2;            // INT4: items whose scales are in shared memory
constexpr unsigned long long kTWaitNs = 500000000ull;   // 0.5 s
static_assert(kTWarps * 32 <= 1024, "block size");

// Per weight format.  Weight tiles hold one K step (rows of 64 bf16, 128
// bytes, 128-byte swizzle): bf16 tiles land by TMA; INT4 / FP8 raw codes land
// by TMA in stages of 64-byte rows (two INT4 K steps or one FP8 K step,
// 64-byte swizzle) and the dequantisation warps write the tiles.
template <int F>
struct GT;
template <>
struct GT<MOE_BF16> {
  static constexpr int kRawSteps = 0;
};
template <>
struct GT<MOE_INT4_G128> {
  static constexpr int kRawSteps = 2;
};
template <>
struct GT<MOE_FP8_E4M3> {
  static constexpr int kRawSteps = 1;
};
constexpr int kTRB = 128;              // bytes per weight-tile row

// weight rows per item of a phase: 256 where the rows split evenly, else 128
__host__ __device__ inline int phase_wn(int ph, int H, int I) {
  return ph == 0 ? (I % 128 == 0 ? 256 : 128) : (H % 256 == 0 ? 256 : 128);
}

// Dynamic shared memory of a phase, in this order: weight tiles, raw stages,
// activation tiles, INT4 scale slots.
struct TLayout {
  int wn = 0;              // weight rows per item (MMA N)
  int nt = 0;              // weight tiles
  int nr = 0;              // raw stages
  unsigned sc_bytes = 0;   // INT4 scale bytes per slot
  size_t bytes = 0;
};
template <int F>
bool tma_layout(int ph, int H, int I, size_t budget, TLayout* L) {
  const int wn = phase_wn(ph, H, I);
  const int K = ph == 0 ? H : I;
  const size_t tb = (size_t)wn * kTRB;
  const size_t rb = (size_t)wn * 64;
  const size_t sc = F == MOE_INT4_G128 ? (size_t)wn * (K / 128) * 2 : 0;
  const size_t fixed = (size_t)kARing * kATile + (size_t)kScSlots * sc + 1024;   // + alignment slack
  if (budget < fixed) return false;
  size_t nt = 0, nr = 0;
  if (F == MOE_BF16) {
    nt = (budget - fixed) / tb;
    if (nt > (size_t)kMaxTiles) nt = kMaxTiles;
  } else {
    nt = 4;   // four K steps of dequantised weights
    if (budget < fixed + nt * tb) return false;
    nr = (budget - fixed - nt * tb) / rb;
    if (nr > (size_t)kMaxRaw) nr = kMaxRaw;
    if (nr < 2) return false;
  }
  if (nt < 3) return false;
  L->wn = wn;
  L->nt = (int)nt;
  L->nr = (int)nr;
  L->sc_bytes = (unsigned)sc;
  L->bytes = nt * tb + nr * rb + fixed;
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
  int wn;                      // weight rows per item (MMA N)
  int nt;                      // weight tiles
  int nr;                      // raw stages
  unsigned sc_bytes;           // INT4 scale bytes of one slot (wn rows x K / 128 bf16)
};

// What the weight producer tells the epilogue and the dequantisation warps about an item
struct ItemRec {
  unsigned long long blk;      // expert block (0: the tile's assignments are invalid)
  int4 td;                     // the tile: first position, rows, expert
};

struct TShared {
  unsigned long long tfull[kMaxTiles];    // weight tile written (TMA bytes, or four dequantisation warps)
  unsigned long long tempty[kMaxTiles];   // the MMAs that read it are done
  unsigned long long rfull[kMaxRaw];      // raw codes of a stage landed
  unsigned long long rempty[kMaxRaw];     // every dequantisation unit of the stage has read them
  unsigned long long afull[kARing];       // activation tile landed
  unsigned long long aempty[kARing];      // the MMAs that read it are done
  unsigned long long cfull[kRecSlots];    // item record written
  unsigned long long cempty[kRecSlots];   // read by the epilogue and the dequantisation warps
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
// (64 bf16), 8-row groups 1024 bytes apart; the K = 16 slice j of the rows
// starts 32 * j bytes in (the swizzle applies to the resulting address)
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
// q - 8 exactly and the product with the scale is the only rounding.  Per pair
// of codes: shift, lop3, sub.bf16x2, mul.bf16x2; then byte permutes into
// element order.
__device__ __forceinline__ uint4 int4x8_bf16(uint32_t wd, uint32_t scale2) {
  uint32_t v0, v1, v2, v3;
  asm("{ .reg .b32 t, p, o;\n"
      "mov.b32 o, 0x43084308;\n"                          // bf16x2 {136, 136}
      "lop3.b32 p, %4, 0x000F000F, 0x43004300, 0xEA;\n"    // {128 + q0, 128 + q4}
      "sub.rn.bf16x2 p, p, o;\n"
      "mul.rn.bf16x2 %0, p, %5;\n"
      "shr.b32 t, %4, 4;\n"
      "lop3.b32 p, t, 0x000F000F, 0x43004300, 0xEA;\n"     // {128 + q1, 128 + q5}
      "sub.rn.bf16x2 p, p, o;\n"
      "mul.rn.bf16x2 %1, p, %5;\n"
      "shr.b32 t, %4, 8;\n"
      "lop3.b32 p, t, 0x000F000F, 0x43004300, 0xEA;\n"     // {128 + q2, 128 + q6}
      "sub.rn.bf16x2 p, p, o;\n"
      "mul.rn.bf16x2 %2, p, %5;\n"
      "shr.b32 t, %4, 12;\n"
      "lop3.b32 p, t, 0x000F000F, 0x43004300, 0xEA;\n"     // {128 + q3, 128 + q7}
      "sub.rn.bf16x2 p, p, o;\n"
      "mul.rn.bf16x2 %3, p, %5; }"
      : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
      : "r"(wd), "r"(scale2));
  return make_uint4(__byte_perm(v0, v1, 0x5410), __byte_perm(v2, v3, 0x5410), __byte_perm(v0, v1, 0x7632),
                    __byte_perm(v2, v3, 0x7632));
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
  if (tc::mbar_try(bar, parity)) return true;   // the common case, without touching the stop flag
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

// The item's expert block and where its weight rows are: region (pool,
// scratch or none: plain loads) and first row in the region's map
template <int F, int PH>
__device__ __forceinline__ void item_weights(const TArgs& g, unsigned long long blk, size_t wrb, int* reg,
                                             int* row_base) {
  const unsigned long long wblk = blk + (PH == PH_UP ? 0ull : g.off_w2);
  *reg = REG_NONE;
  for (int q = 0; q < 2; ++q)
    if (blk >= g.reg_lo[q] && blk < g.reg_hi[q] && (blk - g.reg_lo[q]) % g.reg_pitch[q] < g.reg_part[q] &&
        ((wblk - g.reg_lo[q]) % wrb) == 0ull)
      *reg = q;
  *row_base = *reg == REG_NONE ? 0 : (int)((wblk - g.reg_lo[*reg]) / wrb);
}

template <int F, int PH>
__global__ void __launch_bounds__(kTThreads, 1)
    k_moe_gemm_tma(const __grid_constant__ TmaMaps maps, TArgs g) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ TShared S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool kDq = F != MOE_BF16;
  constexpr int kRawSteps = GT<F>::kRawSteps;     // K steps per raw stage
  constexpr int kUnitsPerRaw = kRawSteps > 0 ? kRawSteps : 1;   // dequantisation units reading one raw stage
  constexpr unsigned kRecReaders = 4 + (kDq ? 4 * kDqGroups : 0);
  const int WN = g.wn, NTL = g.nt, NR = g.nr;
  const int TB = WN * kTRB;                       // bytes per weight tile
  const int RSB = WN * 64;                        // bytes per raw stage
  uint8_t* base = smem + ((1024u - (tc::smem_u32(smem) & 1023u)) & 1023u);
  uint8_t* tiles = base;                                          // [nt][WN rows x 128]
  uint8_t* raws = tiles + (size_t)NTL * TB;                       // [nr][WN rows x 64]
  uint8_t* acts = raws + (size_t)NR * RSB;                        // [kARing][64 rows x 128]
  uint8_t* scb = acts + (size_t)kARing * kATile;                  // [kScSlots][sc_bytes]
  const int K = PH == PH_UP ? g.H : g.I;
  const int nk = K / kKS;
  const int NT = PH == PH_UP ? g.I / (WN >> 1) : g.H / WN;
  const int ntiles = *g.ntiles;
  const int items = ntiles * NT;
  const size_t wrb = F == MOE_BF16 ? (size_t)K * 2 : (F == MOE_FP8_E4M3 ? (size_t)K : (size_t)K / 2);
  if (threadIdx.x == 0) {
    for (int b = 0; b < NTL; ++b) {
      tc::mbar_init(tc::smem_u32(&S.tfull[b]), kDq ? 4u : 1u);
      tc::mbar_init(tc::smem_u32(&S.tempty[b]), 1u);
    }
    for (int b = 0; b < NR; ++b) {
      tc::mbar_init(tc::smem_u32(&S.rfull[b]), 1u);
      tc::mbar_init(tc::smem_u32(&S.rempty[b]), 4u * kUnitsPerRaw);
    }
    for (int b = 0; b < kARing; ++b) {
      tc::mbar_init(tc::smem_u32(&S.afull[b]), 1u);
      tc::mbar_init(tc::smem_u32(&S.aempty[b]), 1u);
    }
    for (int b = 0; b < kRecSlots; ++b) {
      tc::mbar_init(tc::smem_u32(&S.cfull[b]), 1u);
      tc::mbar_init(tc::smem_u32(&S.cempty[b]), kRecReaders);
    }
    for (int b = 0; b < kScSlots; ++b) {
      tc::mbar_init(tc::smem_u32(&S.sfull[b]), 1u);
      tc::mbar_init(tc::smem_u32(&S.sempty[b]), 4u * kDqGroups);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(tc::smem_u32(&S.accf[b]), 1u);
      tc::mbar_init(tc::smem_u32(&S.acce[b]), 4u);
    }
    S.stop = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kWMma) tc::tmem_alloc(tc::smem_u32(&S.tmem), 2u * kMaxWN);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = S.tmem;

  if (warp == kWProdW) {
    // ------------------------------------------------------- weight producer
    unsigned gq = 0;    // weight tiles (bf16) or raw stages (INT4 / FP8) issued
    int it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < items && ok; item += gridDim.x, ++it) {
      const int tile = item / NT, mt = item - tile * NT;
      const int4 td = g.tiles[tile];
      const int asg0 = g.order[td.x];
      const unsigned long long blk = g.asg_ptr[asg0];
      int reg, row_base;
      item_weights<F, PH>(g, blk, wrb, &reg, &row_base);
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
      const int csl = it % kRecSlots;
      if (it >= kRecSlots &&
          !warp_wait(S, tc::smem_u32(&S.cempty[csl]), ((it / kRecSlots) - 1) & 1, g.err, lane, kSleepLong)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        S.rec[csl].blk = blk;
        S.rec[csl].td = td;
        mbar_arrive(tc::smem_u32(&S.cfull[csl]));
      }
      const int half = WN >> 1;
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
      // bf16: one weight tile per K step; INT4 / FP8: one raw stage per kRawSteps K steps
      const int nq = kDq ? nk / kRawSteps : nk;
      const int nslots = kDq ? NR : NTL;
      for (int kq = 0; kq < nq; ++kq, ++gq) {
        const int sl = (int)(gq % (unsigned)nslots);
        unsigned long long* fb = kDq ? &S.rfull[sl] : &S.tfull[sl];
        unsigned long long* eb = kDq ? &S.rempty[sl] : &S.tempty[sl];
        if (gq >= (unsigned)nslots &&
            !warp_wait(S, tc::smem_u32(eb), ((gq / nslots) - 1u) & 1u, g.err, lane, kSleepShort)) {
          ok = false;
          break;
        }
        uint8_t* dst = kDq ? raws + (size_t)sl * RSB : tiles + (size_t)sl * TB;
        constexpr int RB = kDq ? 64 : 128;             // bytes per row of what lands here
        const int x = kDq ? kq * 64 : kq * kKS;        // bytes of raw codes, or bf16 elements
        if (reg == REG_NONE) {
          if (blk != 0ull) {
            // weights in host memory (or not addressable through a map): plain
            // loads, stored in the layout the TMA would write
            const uint8_t* wb = reinterpret_cast<const uint8_t*>(blk + (PH == PH_UP ? 0ull : g.off_w2));
            constexpr int cpr = RB / 16;
            for (int v = lane; v < WN * cpr; v += 32) {
              const int r = v / cpr, c = v - r * cpr;
              const uint4 q = __ldcg(reinterpret_cast<const uint4*>(
                  wb + (size_t)wrow_of<PH>(r, mt, g.I, WN) * wrb + (size_t)x * (kDq ? 1 : 2) + c * 16));
              *reinterpret_cast<uint4*>(dst + (size_t)r * RB + swz_chunk(c, r, RB) * 16) = q;
            }
            if (!kDq) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic stores -> MMA reads
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(tc::smem_u32(fb));
        } else {
          if (lane == 0) {
            mbar_arrive_tx(tc::smem_u32(fb), (unsigned)(WN * RB));
            const CUtensorMap* wm = &maps.w[reg];
            const uint32_t d = tc::smem_u32(dst);
            if (PH == PH_UP) {
              // WN/2 gate rows, then WN/2 up rows of features mt * WN/2 ..
              tma_load_2d(d, wm, x, row_base + mt * half, tc::smem_u32(fb));
              tma_load_2d(d + (uint32_t)(half * RB), wm, x, row_base + g.I + mt * half, tc::smem_u32(fb));
            } else {
              tma_load_2d(d, wm, x, row_base + mt * WN, tc::smem_u32(fb));
            }
          }
          __syncwarp();
        }
      }
    }
  } else if (warp == kWProdA) {
    // --------------------------------------------------- activation producer
    unsigned ga = 0;    // activation tiles issued
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
      const int4 td = g.tiles[item / NT];
      // tile rows -> the smallest box that holds them
      const int bi = td.y <= 16 ? 0 : (td.y <= 32 ? 1 : 2);
      const unsigned abytes = (unsigned)((16 << bi) * 128);
      bool ok = true;
      for (int ks = 0; ks < nk; ++ks, ++ga) {
        const int sl = (int)(ga % kARing);
        if (ga >= (unsigned)kARing &&
            !warp_wait(S, tc::smem_u32(&S.aempty[sl]), ((ga / kARing) - 1u) & 1u, g.err, lane, kSleepShort)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t fb = tc::smem_u32(&S.afull[sl]);
          mbar_arrive_tx(fb, abytes);
          tma_load_2d(tc::smem_u32(acts + (size_t)sl * kATile), &maps.b[bi], ks * kKS, td.x, fb);
        }
        __syncwarp();
      }
      if (!ok) break;
    }
  } else if (warp == kWMma) {
    // ----------------------------------------------------------------- MMA
    const uint32_t idesc = tc::idesc_bf16(kM, (uint32_t)WN);
    unsigned ga = 0, gt = 0;   // activation tiles and weight tiles consumed
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
      for (int ks = 0; ks < nk && ok; ++ks, ++ga) {
        const int as = (int)(ga % kARing);
        // INT4 / FP8: a dequantisation warp has waited for this K step's
        // activation tile before it marked the weight tile full (below), so the
        // weight tile's barrier covers both and this warp waits once per step
        if (!kDq && lane == 0) ok = wait_or_stop(S, tc::smem_u32(&S.afull[as]), (ga / kARing) & 1u, g.err);
        const uint32_t a_u = tc::smem_u32(acts + (size_t)as * kATile);
        {
          const int tb = (int)(gt % (unsigned)NTL);
          if (lane == 0 && ok) ok = wait_or_stop(S, tc::smem_u32(&S.tfull[tb]), (gt / NTL) & 1u, g.err);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          tc::fence_after_sync();
          if (lane == 0) {
            const uint32_t b_u = tc::smem_u32(tiles + (size_t)tb * TB);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tc::mma_bf16(d_tmem, desc_sw128(a_u + (uint32_t)j * 32u), desc_sw128(b_u + (uint32_t)j * 32u), idesc,
                           (ks | j) != 0 ? 1u : 0u);
            tc::mma_commit(tc::smem_u32(&S.tempty[tb]));
          }
          __syncwarp();
          ++gt;
        }
        if (lane == 0) tc::mma_commit(tc::smem_u32(&S.aempty[as]));
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc::mma_commit(tc::smem_u32(&S.accf[buf]));
      __syncwarp();
    }
    // every MMA issued has completed before tensor memory is freed
    if (ga > 0 && lane == 0) {
      const unsigned last = ga - 1u;
      tc::mbar_wait(tc::smem_u32(&S.aempty[last % kARing]), (last / kARing) & 1u, kTWaitNs);
    }
    __syncwarp();
  } else if (warp >= kWDq) {
    // ------------------------------------------------- dequantisation warps
    // A unit is one weight tile: WN rows x one K step.  Group grp takes the
    // units u with u % kDqGroups == grp; warp w of the group converts rows
    // w * WN / 4 .., WN / 128 a thread.
    if (kDq) {
      const int grp = (warp - kWDq) >> 2;
      const int wq = (warp - kWDq) & 3;
      const int gpr = K / 128;                              // INT4 scale groups per row
      const int upi = nk;                                   // units per item
      unsigned gu = 0;                                      // units of earlier items
      int it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < items && ok; item += gridDim.x, ++it) {
        const int csl = it % kRecSlots, ssl = it % kScSlots;
        if (!warp_wait(S, tc::smem_u32(&S.cfull[csl]), (it / kRecSlots) & 1, g.err, lane, kSleepShort)) {
          ok = false;
          break;
        }
        const unsigned long long blk = S.rec[csl].blk;
        __syncwarp();
        if (lane == 0) mbar_arrive(tc::smem_u32(&S.cempty[csl]));
        if (F == MOE_INT4_G128 &&
            !warp_wait(S, tc::smem_u32(&S.sfull[ssl]), (it / kScSlots) & 1, g.err, lane, kSleepShort)) {
          ok = false;
          break;
        }
        const uint16_t* sct = reinterpret_cast<const uint16_t*>(scb + (size_t)ssl * g.sc_bytes);
        for (int v = (int)((unsigned)(grp + kDqGroups) - gu % kDqGroups) % kDqGroups; v < upi; v += kDqGroups) {
          const unsigned u = gu + (unsigned)v;               // unit; its weight tile u % nt
          const unsigned rq = u / kUnitsPerRaw;               // its raw stage
          const int part = (int)(u % kUnitsPerRaw);           // which K step of the raw row
          const int rs = (int)(rq % (unsigned)NR), tb = (int)(u % (unsigned)NTL);
          if (lane == 0) {
            ok = wait_or_stop(S, tc::smem_u32(&S.rfull[rs]), (rq / NR) & 1u, g.err, kSleepShort);
            // the tile free: the MMAs that read its previous contents are done
            if (ok && u >= (unsigned)NTL)
              ok = wait_or_stop(S, tc::smem_u32(&S.tempty[tb]), ((u / NTL) - 1u) & 1u, g.err, kSleepShort);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          __syncwarp();
          if (blk != 0ull) {
            const uint8_t* rst = raws + (size_t)rs * RSB;
            uint8_t* tile = tiles + (size_t)tb * TB;
#pragma unroll 1
            for (int h = 0; h < WN / 128; ++h) {
              const int r = wq * (WN / 4) + h * 32 + lane;   // weight row of the item (< WN)
              const uint8_t* raw = rst + (size_t)r * 64;
              uint4 o[8];
              if (F == MOE_INT4_G128) {
                // 64 codes = chunks 2 part, 2 part + 1 of the row; K step v is in scale group v / 2
                const uint32_t sb = sct[(size_t)r * gpr + (v >> 1)];
                const uint32_t s2 = sb | (sb << 16);
                const uint4 q0 = reinterpret_cast<const uint4*>(raw)[swz_chunk(2 * part, r, 64)];
                const uint4 q1 = reinterpret_cast<const uint4*>(raw)[swz_chunk(2 * part + 1, r, 64)];
                o[0] = int4x8_bf16(q0.x, s2);
                o[1] = int4x8_bf16(q0.y, s2);
                o[2] = int4x8_bf16(q0.z, s2);
                o[3] = int4x8_bf16(q0.w, s2);
                o[4] = int4x8_bf16(q1.x, s2);
                o[5] = int4x8_bf16(q1.y, s2);
                o[6] = int4x8_bf16(q1.z, s2);
                o[7] = int4x8_bf16(q1.w, s2);
              } else {
                // 64 codes = the whole row
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                  const uint4 q = reinterpret_cast<const uint4*>(raw)[swz_chunk(c, r, 64)];
                  o[2 * c] = fp8x8_bf16(q.x, q.y);
                  o[2 * c + 1] = fp8x8_bf16(q.z, q.w);
                }
              }
              uint8_t* trow = tile + (size_t)r * kTRB;
#pragma unroll
              for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(trow + swz_chunk(c, r, kTRB) * 16) = o[c];
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic stores -> MMA reads
          }
          __syncwarp();
          if (lane == 0) {
            // the first warp of the group also waits for the step's activation
            // tile: the tile barrier then completes only once both operands are
            // in place (TMA complete_tx -> this acquire -> the release of the
            // arrive -> the MMA issuer's acquire)
            if (wq == 0 && ok)
              ok = wait_or_stop(S, tc::smem_u32(&S.afull[u % kARing]), (u / kARing) & 1u, g.err, kSleepShort);
            mbar_arrive(tc::smem_u32(&S.tfull[tb]));
            mbar_arrive(tc::smem_u32(&S.rempty[rs]));
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
        }
        if (!ok) break;
        gu += (unsigned)upi;
        if (F == MOE_INT4_G128) {
          __syncwarp();
          if (lane == 0) mbar_arrive(tc::smem_u32(&S.sempty[ssl]));
        }
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ epilogue
    // with M = 64 the accumulator's row 16 q + i is in lane 32 q + i: warp q
    // reads lane quadrant q, its lanes 0-15 hold token rows 16 q .. 16 q + 15
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int half = WN >> 1;
    int it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < items && ok; item += gridDim.x, ++it) {
      const int mt = item % NT;
      const int csl = it % kRecSlots;
      if (!warp_wait(S, tc::smem_u32(&S.cfull[csl]), (it / kRecSlots) & 1, g.err, lane, kSleepLong)) {
        ok = false;
        break;
      }
      const int4 td = S.rec[csl].td;
      const unsigned long long blk = S.rec[csl].blk;
      __syncwarp();
      if (lane == 0) mbar_arrive(tc::smem_u32(&S.cempty[csl]));
      const int t = warp * 16 + lane;                  // token row of the tile (lanes 0-15)
      const bool valid = lane < 16 && t < td.y;
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
  g.wn = lu.wn;
  g.nt = lu.nt;
  g.nr = lu.nr;
  g.sc_bytes = lu.sc_bytes;
  k_moe_gemm_tma<F, PH_UP><<<sms, kTThreads, lu.bytes, s>>>(m.up, g);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  g.pending = nullptr;   // every expert has landed before the up kernel ended
  g.wn = ld.wn;
  g.nt = ld.nt;
  g.nr = ld.nr;
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
