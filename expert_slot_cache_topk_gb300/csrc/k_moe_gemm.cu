// Grouped expert MLP for steps with many tokens (batched decode, prefill) on
// the sm_103a tensor cores (tcgen05, bf16 operands, f32 accumulators in
// tensor memory).
//
// With T tokens and top-k routing there are n = T * k assignments; expert e
// serves the M_e assignments that chose it.  A per-token kernel would read
// expert e's weights M_e times; here the assignments are grouped by expert
// (k_group) and every weight tile is read once per tile of up to 128 of the
// expert's assignments, which makes each expert a dense contraction:
//   up:   [M_e x H] . [H x 2I]  -> h = w * silu(gate) * up   (bf16, [n, I])
//   down: [M_e x I] . [I x H]   -> one f32 row per assignment ([n, H])
//   combine: y[t] = sum over j of row t * k + j (+ x[t]), j in order
// (vLLM PR #37190 "Run MoE models exceeding VRAM via expert CPU offloading
// with GPU cache", "How it works": fused_experts over the remapped ids; the
// expert blocks are wherever prepare put them -- pool slot, bypass scratch, or
// mapped host memory for the cold set, "Running 125B MoE on Two 32 GB Cards",
// section 2).
//
// Each output element is one tensor-core dot product over K whose value does
// not depend on the other rows of its tile, so results do not depend on how
// assignments are grouped or where an expert's bytes live.  INT4 weights are
// dequantised to bf16 ((q - 8) * scale, rounded once) while being staged, and
// h is rounded to bf16 between the two GEMMs; both stay well inside the
// float tolerance against the float64 reference.
//
// Kernel shape: persistent CTAs of 8 warps, work item = (tile of <= 128
// assignments of one expert, N tile of 128 output columns).  For each K step
// of 64 the threads stage A (gathered activation rows) and B (weight rows) in
// shared memory as 8 x 16-byte core matrices with cp.async, three K steps
// ahead of the MMAs over five stages; one thread issues four tcgen05.mma (K = 16
// each) into a 128 x 128 f32 accumulator in tensor memory and commits them to
// the stage's mbarrier, which releases the stage for the next copies.  The
// epilogue reads the accumulator with tcgen05.ld.

#include <cuda_bf16.h>
#include <cstdint>

#include "internal.cuh"
#include "mlp_common.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace mlp;

constexpr int kGThreads = 256;                  // 8 warps
constexpr int kTileM = 128;                     // assignments per tile (MMA M)
constexpr int kTileN = 128;                     // output columns per item (MMA N)
constexpr int kTileBytes = kTileM * (int)tc::kTileK * 2;   // one 128 x 64 bf16 operand tile
constexpr int kGStageBytes = 2 * kTileBytes;               // A + B
constexpr int kGroupThreads = 1024;
constexpr unsigned long long kGWaitNs = 500000000ull;     // 0.5 s

enum { PH_UP = 0, PH_DOWN = 1 };

struct GemmArgs {
  const int32_t* order;        // [n] assignment indices grouped by expert
  const int4* tiles;           // [ntiles] {first position in order, rows, expert, 0}
  const int* ntiles;
  unsigned* work;              // [2] next item of the up / down GEMM (reset by k_group)
  const void* x;               // [T, H] bf16 activations (up)
  uint16_t* hb;                // [n, I] bf16 h (written by up, read by down)
  float* out;                  // [n, H] f32 rows, one per assignment (down)
  const unsigned long long* asg_ptr;
  const float* w;
  int k, H, I;
  unsigned long long off_w2, off_s13, off_s2;
  int* err;
  const uint8_t* pending;      // [n] or null: assignment's expert is copied in this step
  const unsigned* ready;       // [E]: ready[e] == hdr->seq once expert e has landed
  const RecHdr* hdr;
};

// ------------------------------------------------------------- grouping
// One CTA.  Counts the assignments of every expert, lays them out expert by
// expert (ascending expert; within an expert in no particular order, which
// the results do not depend on) and cuts every expert's run into tiles of at
// most `tile` assignments.
__global__ void __launch_bounds__(kGroupThreads, 1) k_group(const int32_t* __restrict__ ids, int n, int E,
                                                            int32_t* __restrict__ order, int4* __restrict__ tiles,
                                                            int* __restrict__ ntiles, unsigned* __restrict__ work,
                                                            int tile) {
  __shared__ int cnt[MOE_MAX_EXPERTS];
  __shared__ int off[MOE_MAX_EXPERTS];
  __shared__ int toff[MOE_MAX_EXPERTS];
  __shared__ int cur[MOE_MAX_EXPERTS];
  __shared__ int wsum[2][kGroupThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < 2) work[tid] = 0u;   // item counters of the up and down GEMMs
  for (int e = tid; e < E; e += blockDim.x) {
    cnt[e] = 0;
    cur[e] = 0;
  }
  __syncthreads();
  for (int i = tid; i < n; i += blockDim.x) {
    const int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  // exclusive scans of the counts and of the tile counts (E <= blockDim.x)
  const int c = tid < E ? cnt[tid] : 0;
  const int t = (c + tile - 1) / tile;
  int ic = c, it = t;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, ic, o), b = __shfl_up_sync(0xffffffffu, it, o);
    if (lane >= o) {
      ic += a;
      it += b;
    }
  }
  if (lane == 31) {
    wsum[0][warp] = ic;
    wsum[1][warp] = it;
  }
  __syncthreads();
  if (warp == 0) {
    int a = lane < kGroupThreads / 32 ? wsum[0][lane] : 0, b = lane < kGroupThreads / 32 ? wsum[1][lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int pa = __shfl_up_sync(0xffffffffu, a, o), pb = __shfl_up_sync(0xffffffffu, b, o);
      if (lane >= o) {
        a += pa;
        b += pb;
      }
    }
    if (lane < kGroupThreads / 32) {
      wsum[0][lane] = a;
      wsum[1][lane] = b;
    }
  }
  __syncthreads();
  const int base_c = warp ? wsum[0][warp - 1] : 0, base_t = warp ? wsum[1][warp - 1] : 0;
  if (tid < E) {
    off[tid] = base_c + ic - c;
    toff[tid] = base_t + it - t;
  }
  if (tid == blockDim.x - 1) *ntiles = base_t + it;
  __syncthreads();
  for (int i = tid; i < n; i += blockDim.x) {
    const int e = ids[i];
    if (e >= 0 && e < E) order[off[e] + atomicAdd(&cur[e], 1)] = i;
  }
  if (tid < E) {
    for (int q = 0; q < t; ++q) {
      const int rows = c - q * tile < tile ? c - q * tile : tile;
      tiles[toff[tid] + q] = make_int4(off[tid] + q * tile, rows, tid, 0);
    }
  }
}

// ---------------------------------------------------------------- staging
// Thread t stages row r = t % 128 of both 128 x 64 operand tiles, chunks
// 4 h .. 4 h + 3 (h = t / 128) of 8 bf16 each.  A rows and bf16 weight rows
// go straight into the core-matrix layout with cp.async (16 bytes, L2 only);
// INT4 weight rows (16 bytes = 32 codes per thread) go to a raw buffer and are
// dequantised by the same thread once they have landed.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// Eight 4-bit codes (nibble i of wd is element i) -> bf16 (q - 8) * scale, in
// element order, two elements per 32-bit word.  A code placed in the mantissa
// of a bf16 whose exponent is that of 128 is the value 128 + q exactly (seven
// mantissa bits hold q); subtracting 136 leaves q - 8 exactly, and the only
// rounding is that of the product, as when (q - 8) * scale is formed in f32
// (exactly: 4 + 8 significant bits) and rounded to bf16.  Word j below holds
// elements j and j + 4; byte permutes put the pairs back in order.
__device__ __forceinline__ uint4 int4x8_to_bf16(uint32_t wd, uint32_t scale2) {
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

// ------------------------------------------------------------------ GEMM
// PH_UP: item = (tile, N tile nt of I / 64): B rows 0..63 are gate rows
// nt*64 .., rows 64..127 the matching up rows; K = H.  Epilogue: h.
// PH_DOWN: item = (tile, N tile nt of H / 128): B rows are W2 rows nt*128 ..;
// K = I.  Epilogue: f32 output rows.
constexpr int kGStagesP = 5;                 // staged K steps
constexpr int kGAhead = 3;                   // K steps in flight ahead of the MMA
constexpr int kRawBytes = kTileM * 2 * 32;   // raw INT4 (16 B per thread) or FP8 (32 B) rows of one K step
constexpr int kMaxGroups = 64;               // scale groups per row kept in shared memory (K <= 8192)

template <int F, int PH>
__global__ void __launch_bounds__(kGThreads, 1) k_moe_gemm(GemmArgs g) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) unsigned long long mbar[kGStagesP];
  __shared__ uint32_t tmem_slot;
  __shared__ int rows_idx[kTileM];     // A row source: token (up) or assignment (down)
  __shared__ int asg_of[kTileM];       // assignment of each tile row
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = *g.ntiles;
  const int NT = PH == PH_UP ? g.I / 64 : g.H / kTileN;
  const int items = ntiles * NT;
  const int K = PH == PH_UP ? g.H : g.I;
  const int nk = K / (int)tc::kTileK;
  const size_t wrb = F == MOE_BF16 ? (size_t)K * 2 : (F == MOE_FP8_E4M3 ? (size_t)K : (size_t)K / 2);
  constexpr int kRawPer = F == MOE_FP8_E4M3 ? 32 : 16;   // raw bytes each thread stages per K step
  const int groups = K / 128;          // INT4 scale groups per weight row
  // layout: [stages x (A tile | B tile)] [stages x raw INT4] [128 x groups scales]
  uint8_t* base = smem + ((1024u - (tc::smem_u32(smem) & 1023u)) & 1023u);
  uint8_t* raw0 = base + (size_t)kGStagesP * kGStageBytes;
  uint16_t* sc = reinterpret_cast<uint16_t*>(raw0 + (size_t)kGStagesP * kRawBytes);
  if (tid == 0) {
    for (int s = 0; s < kGStagesP; ++s) tc::mbar_init(tc::smem_u32(&mbar[s]), 1u);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&tmem_slot), kTileN);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  constexpr uint32_t idesc = tc::idesc_bf16(kTileM, kTileN);
  const int r = tid & (kTileM - 1);
  const int hh = tid >> 7;             // which 32-element half of the K step this thread stages
  unsigned gs = 0;                     // K steps of this CTA so far (stage = gs % kGStagesP)
  bool dead = false;
  // items are taken from a shared counter, so a CTA that starts late (its SM
  // busy with another kernel) simply takes fewer of them
  __shared__ int next_item;
  if (tid == 0) next_item = (int)atomicAdd(g.work + PH, 1u);
  __syncthreads();
  for (int item = next_item; item < items && !dead; item = next_item) {
    const int tile = item / NT, nt = item - tile * NT;
    const int4 td = g.tiles[tile];
    const int pos0 = td.x, rows = td.y;
    if (tid < kTileM) {
      const int a = tid < rows ? g.order[pos0 + tid] : 0;
      asg_of[tid] = a;
      rows_idx[tid] = PH == PH_UP ? a / g.k : a;
    }
    __syncthreads();
    if (PH == PH_UP && g.pending != nullptr && tid == 0 && g.pending[asg_of[0]] != 0) {
      // the expert is being copied in this step: wait (bounded) until its copy is published
      const unsigned want = g.hdr->seq;
      const unsigned long long t0 = tc::global_ns();
      for (unsigned it = 0;; ++it) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(g.ready + td.z) : "memory");
        if (v == want) break;
        if ((it & 63u) == 63u && tc::global_ns() - t0 > 2000000000ull) {
          dead = true;
          break;
        }
        __nanosleep(256);
      }
    }
    if (__syncthreads_or(dead)) break;
    const unsigned long long blk = g.asg_ptr[asg_of[0]];
    const uint8_t* wb = reinterpret_cast<const uint8_t*>(blk) + (PH == PH_UP ? 0 : g.off_w2);
    const uint16_t* sbase = reinterpret_cast<const uint16_t*>(blk + (PH == PH_UP ? g.off_s13 : g.off_s2));
    const int wrow = PH == PH_UP ? (r < 64 ? nt * 64 + r : g.I + nt * 64 + (r - 64)) : nt * kTileN + r;
    const uint8_t* wrow_p = wb + (size_t)wrow * wrb;
    const bool arow_ok = r < rows;
    const uint8_t* arow_p = PH == PH_UP
                                ? reinterpret_cast<const uint8_t*>(g.x) + (size_t)rows_idx[arow_ok ? r : 0] * g.H * 2
                                : reinterpret_cast<const uint8_t*>(g.hb) + (size_t)rows_idx[arow_ok ? r : 0] * g.I * 2;
    if (F == MOE_INT4_G128) {
      // this item's scales: 128 rows x groups, two threads per row
      for (int q = hh; q < groups; q += 2) sc[r * kMaxGroups + q] = sbase[(size_t)wrow * groups + q];
    }
    float fsg = 1.f, fsu = 1.f, fsd = 1.f;   // FP8: the expert's gate, up and down tensor scales
    if (F == MOE_FP8_E4M3 && PH == PH_UP && blk != 0ull) {
      const float* f13 = reinterpret_cast<const float*>(blk + g.off_s13);
      fsg = __ldcg(f13);
      fsu = __ldcg(f13 + 1);
      fsd = __ldcg(reinterpret_cast<const float*>(blk + g.off_s2));
    }
    // stage the operands of K step ks (global step gq) into stage gq % kGStagesP
    auto issue = [&](int ks, unsigned gq) {
      const int s = (int)(gq % kGStagesP);
      uint8_t* sa = base + (size_t)s * kGStageBytes;
      const uint32_t sa_u = tc::smem_u32(sa), sb_u = sa_u + kTileBytes;
      const int k0 = ks * (int)tc::kTileK;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t kk = (uint32_t)((hh * 4 + i) * 8);
        cp_async16(sa_u + tc::tile_offset((uint32_t)r, kk), arow_p + (size_t)(k0 + kk) * 2, arow_ok);
      }
      if (F == MOE_BF16) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t kk = (uint32_t)((hh * 4 + i) * 8);
          cp_async16(sb_u + tc::tile_offset((uint32_t)r, kk), wrow_p + (size_t)(k0 + kk) * 2, true);
        }
      } else if (F == MOE_FP8_E4M3) {
        const uint32_t d0 = tc::smem_u32(raw0 + (size_t)s * kRawBytes + (size_t)tid * kRawPer);
        cp_async16(d0, wrow_p + (size_t)(k0 + 32 * hh), true);
        cp_async16(d0 + 16u, wrow_p + (size_t)(k0 + 32 * hh) + 16, true);
      } else {
        cp_async16(tc::smem_u32(raw0 + (size_t)s * kRawBytes + (size_t)tid * kRawPer),
                   wrow_p + (size_t)(k0 + 32 * hh) / 2, true);
      }
    };
    for (int q = 0; q < kGAhead; ++q) {
      if (q < nk) {
        const unsigned gq = gs + q;
        if (gq >= (unsigned)kGStagesP &&
            !tc::mbar_wait(tc::smem_u32(&mbar[gq % kGStagesP]), ((gq / kGStagesP) - 1u) & 1u, kGWaitNs))
          dead = true;
        issue(q, gq);
      }
      cp_async_commit();
    }
    __syncthreads();   // scales in shared memory
    for (int ks = 0; ks < nk; ++ks, ++gs) {
      const int s = (int)(gs % kGStagesP);
      // prefetch K step ks + kGAhead once the MMA that last used its stage is done
      {
        const int kp = ks + kGAhead;
        if (kp < nk) {
          const unsigned gq = gs + kGAhead;
          if (gq >= (unsigned)kGStagesP &&
              !tc::mbar_wait(tc::smem_u32(&mbar[gq % kGStagesP]), ((gq / kGStagesP) - 1u) & 1u, kGWaitNs))
            dead = true;
          issue(kp, gq);
        }
        cp_async_commit();
      }
      cp_async_wait<kGAhead>();          // this thread's copies of step ks have landed
      uint8_t* sa = base + (size_t)s * kGStageBytes;
      uint8_t* sbt = sa + kTileBytes;
      if (F == MOE_FP8_E4M3) {
        // 32 E4M3 codes -> bf16 (exact); the tensor scales apply in the epilogue
        const uint4* rq = reinterpret_cast<const uint4*>(raw0 + (size_t)s * kRawBytes + (size_t)tid * kRawPer);
        const uint4 q0 = rq[0], q1 = rq[1];
        const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t o[4];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const uint32_t wd = words[2 * i + h2];   // elements 8 i + 4 h2 .. + 3
            const float2 a = e4m3x2_to_f2(wd), b = e4m3x2_to_f2(wd >> 16);
            o[2 * h2] = pack_bf16x2(a.x, a.y);
            o[2 * h2 + 1] = pack_bf16x2(b.x, b.y);
          }
          *reinterpret_cast<uint4*>(sbt + tc::tile_offset((uint32_t)r, (uint32_t)((hh * 4 + i) * 8))) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      if (F == MOE_INT4_G128) {
        const uint4 qv = *reinterpret_cast<const uint4*>(raw0 + (size_t)s * kRawBytes + (size_t)tid * kRawPer);
        const uint32_t sb = sc[r * kMaxGroups + ((ks * (int)tc::kTileK) >> 7)];
        const uint32_t words[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)   // elements 8 i .. 8 i + 7 of this thread's 32
          *reinterpret_cast<uint4*>(sbt + tc::tile_offset((uint32_t)r, (uint32_t)((hh * 4 + i) * 8))) =
              int4x8_to_bf16(words[i], sb | (sb << 16));
      }
      tc::fence_async_smem();
      if (__syncthreads_or(dead)) {
        dead = true;
        break;
      }
      if (tid == 0) {
        tc::fence_after_sync();
        const uint32_t a0 = tc::smem_u32(sa), b0 = tc::smem_u32(sbt);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          tc::mma_bf16(tmem, tc::smem_desc(a0 + 256u * j), tc::smem_desc(b0 + 256u * j), idesc,
                       (ks | j) != 0 ? 1u : 0u);
        tc::mma_commit(tc::smem_u32(&mbar[s]));
      }
    }
    cp_async_wait<0>();
    if (dead) break;
    // accumulator complete: the last commit covers every MMA issued before it
    {
      const unsigned last = gs - 1u;
      if (!tc::mbar_wait(tc::smem_u32(&mbar[last % kGStagesP]), (last / kGStagesP) & 1u, kGWaitNs)) dead = true;
    }
    if (__syncthreads_or(dead)) break;
    tc::fence_after_sync();
    const int m = (warp & 3) * 32 + lane;            // accumulator row of this thread
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int ch = warp >> 2;                        // column half
    if (PH == PH_UP) {
      uint32_t gv[32], uv[32];
      tc::tmem_ld32(lane_base + (uint32_t)(ch * 32), gv);
      tc::tmem_ld32(lane_base + (uint32_t)(64 + ch * 32), uv);
      if (m < rows) {
        const int a = asg_of[m];
        const float wa = g.w[a];
        uint4* dst = reinterpret_cast<uint4*>(g.hb + (size_t)a * g.I + nt * 64 + ch * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float hv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float gg = __uint_as_float(gv[8 * q + e]) * fsg, uu = __uint_as_float(uv[8 * q + e]) * fsu;
            hv[e] = wa * (gg / (1.0f + expf(-gg)) * uu) * fsd;
          }
          uint4 o;
          o.x = pack_bf16x2(hv[0], hv[1]);
          o.y = pack_bf16x2(hv[2], hv[3]);
          o.z = pack_bf16x2(hv[4], hv[5]);
          o.w = pack_bf16x2(hv[6], hv[7]);
          dst[q] = o;
        }
      }
    } else {
      uint32_t v0[32], v1[32];
      tc::tmem_ld32(lane_base + (uint32_t)(ch * 64), v0);
      tc::tmem_ld32(lane_base + (uint32_t)(ch * 64 + 32), v1);
      if (m < rows) {
        float4* dst = reinterpret_cast<float4*>(g.out + (size_t)asg_of[m] * g.H + nt * kTileN + ch * 64);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[q] = make_float4(__uint_as_float(v0[4 * q]), __uint_as_float(v0[4 * q + 1]),
                               __uint_as_float(v0[4 * q + 2]), __uint_as_float(v0[4 * q + 3]));
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[8 + q] = make_float4(__uint_as_float(v1[4 * q]), __uint_as_float(v1[4 * q + 1]),
                                   __uint_as_float(v1[4 * q + 2]), __uint_as_float(v1[4 * q + 3]));
      }
    }
    if (tid == 0) next_item = (int)atomicAdd(g.work + PH, 1u);
    tc::fence_before_sync();
    __syncthreads();    // accumulator, tile tables and scales free for the next item
  }
  cp_async_wait<0>();
  if (dead && tid == 0) atomicExch(g.err, DEVERR_RING);
  // every MMA this CTA issued has completed before tensor memory is freed
  if (gs > 0 && tid == 0) {
    const unsigned last = gs - 1u;
    tc::mbar_wait(tc::smem_u32(&mbar[last % kGStagesP]), (last / kGStagesP) & 1u, kGWaitNs);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_free(tmem, kTileN);
}

// y[t] = sum over j of out[t * k + j] (+ x[t]), j in order
template <int F>
__global__ void __launch_bounds__(256) k_combine(const float* __restrict__ out, const void* __restrict__ x,
                                                 void* __restrict__ y, int T, int k, int H, int residual) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;   // group of 4 columns
  const int H4 = H / 4;
  if (i >= (long long)T * H4) return;
  const int t = (int)(i / H4), c4 = (int)(i - (long long)t * H4);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const float4 v = reinterpret_cast<const float4*>(out + ((size_t)t * k + j) * H)[c4];
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  const size_t o = (size_t)t * H + 4 * c4;
  if (residual) {
    const uint16_t* xb = reinterpret_cast<const uint16_t*>(x) + o;
    acc.x += bf16_bits(xb[0]);
    acc.y += bf16_bits(xb[1]);
    acc.z += bf16_bits(xb[2]);
    acc.w += bf16_bits(xb[3]);
  }
  uint2 pk;
  pk.x = pack_bf16x2(acc.x, acc.y);
  pk.y = pack_bf16x2(acc.z, acc.w);
  *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(y) + o) = pk;
}

// ------------------------------------------------------------------ host
constexpr size_t kGemmSmem = (size_t)kGStagesP * (kGStageBytes + kRawBytes) +
                             (size_t)kTileM * kMaxGroups * 2 + 1024;   // + alignment slack

// Whether the attributes are set and the occupancy, per weight format and
// device (guarded by launch_state_mutex()).
struct GemmLaunchState {
  bool configured = false;
  int blocks_per_sm = 0;
};
GemmLaunchState g_gemm_state[4][kMaxDevices];

template <int F>
cudaError_t gemm_configure_impl() {
  device_sm_count();   // cache the SM count outside any capture
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(launch_state_mutex());
  GemmLaunchState& st = g_gemm_state[F][dev];
  if (st.configured) return cudaSuccess;
  const void* kernels[] = {(const void*)k_moe_gemm<F, PH_UP>, (const void*)k_moe_gemm<F, PH_DOWN>};
  for (const void* kf : kernels) {
    cudaError_t e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kf, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  int nb = 0;
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k_moe_gemm<F, PH_UP>, kGThreads, kGemmSmem);
  if (e != cudaSuccess) return e;
  st.blocks_per_sm = nb;
  st.configured = true;
  return cudaSuccess;
}

template <int F>
cudaError_t gemm_impl(const MlpArgs& a, const GemmBuffers& b, cudaStream_t s) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorNotSupported;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(launch_state_mutex());
    const GemmLaunchState& st = g_gemm_state[F][dev];
    if (!st.configured || st.blocks_per_sm < 1) return cudaErrorNotSupported;
    per_sm = st.blocks_per_sm;
  }
  const int n = a.T * a.k;
  k_group<<<1, kGroupThreads, 0, s>>>(b.ids, n, b.E, b.order, b.tiles, b.ntiles, b.work, kTileM);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  GemmArgs g{};
  g.order = b.order;
  g.tiles = b.tiles;
  g.ntiles = b.ntiles;
  g.work = b.work;
  g.x = a.x;
  g.hb = b.hb;
  g.out = b.out;
  g.asg_ptr = a.asg_ptr;
  g.w = a.w;
  g.k = a.k;
  g.H = a.H;
  g.I = a.I;
  g.off_w2 = a.off_w2;
  g.off_s13 = a.off_s13;
  g.off_s2 = a.off_s2;
  g.err = b.err;
  g.pending = b.pending;
  g.ready = b.ready;
  g.hdr = b.hdr;
  const int grid = per_sm * device_sm_count();
  k_moe_gemm<F, PH_UP><<<grid, kGThreads, kGemmSmem, s>>>(g);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_moe_gemm<F, PH_DOWN><<<grid, kGThreads, kGemmSmem, s>>>(g);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long groups = (long long)a.T * (a.H / 4);
  k_combine<F><<<(unsigned)((groups + 255) / 256), 256, 0, s>>>(b.out, a.x, a.y, a.T, a.k, a.H, a.residual);
  return cudaGetLastError();
}

}  // namespace

bool moe_gemm_supported(int wdtype, int H, int I, int k) {
  if (wdtype != MOE_BF16 && wdtype != MOE_INT4_G128 && wdtype != MOE_FP8_E4M3) return false;
  if (k < 1 || k > MOE_MAX_TOPK) return false;
  if (H % kTileN || I % 64) return false;          // N tiles of the two GEMMs, K tiles of 64
  if (H > 128 * kMaxGroups || I > 128 * kMaxGroups) return false;   // scales of an item in shared memory
  if (wdtype == MOE_INT4_G128 && (H % 128 || I % 128)) return false;
  return true;
}

cudaError_t moe_gemm_configure(int wdtype) {
  switch (wdtype) {
    case MOE_BF16: return gemm_configure_impl<MOE_BF16>();
    case MOE_INT4_G128: return gemm_configure_impl<MOE_INT4_G128>();
    case MOE_FP8_E4M3: return gemm_configure_impl<MOE_FP8_E4M3>();
  }
  return cudaErrorNotSupported;
}

cudaError_t launch_group(const int32_t* ids, int n, int E, int32_t* order, int4* tiles, int* ntiles, unsigned* work,
                         int tile, cudaStream_t s) {
  k_group<<<1, kGroupThreads, 0, s>>>(ids, n, E, order, tiles, ntiles, work, tile);
  return cudaGetLastError();
}

cudaError_t launch_combine(int wdtype, const float* out, const void* x, void* y, int T, int k, int H, int residual,
                           cudaStream_t s) {
  const long long groups = (long long)T * (H / 4);
  const unsigned grid = (unsigned)((groups + 255) / 256);
  if (wdtype == MOE_BF16) k_combine<MOE_BF16><<<grid, 256, 0, s>>>(out, x, y, T, k, H, residual);
  else if (wdtype == MOE_INT4_G128) k_combine<MOE_INT4_G128><<<grid, 256, 0, s>>>(out, x, y, T, k, H, residual);
  else if (wdtype == MOE_FP8_E4M3) k_combine<MOE_FP8_E4M3><<<grid, 256, 0, s>>>(out, x, y, T, k, H, residual);
  else return cudaErrorNotSupported;
  return cudaGetLastError();
}

cudaError_t launch_moe_gemm(int wdtype, const MlpArgs& a, const GemmBuffers& b, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (!moe_gemm_supported(wdtype, a.H, a.I, a.k) || a.x == nullptr) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(a.x) | reinterpret_cast<uintptr_t>(a.y)) & 15) return cudaErrorNotSupported;
  switch (wdtype) {
    case MOE_BF16: return gemm_impl<MOE_BF16>(a, b, s);
    case MOE_INT4_G128: return gemm_impl<MOE_INT4_G128>(a, b, s);
    case MOE_FP8_E4M3: return gemm_impl<MOE_FP8_E4M3>(a, b, s);
  }
  return cudaErrorNotSupported;
}

}  // namespace moe
