// Internal declarations shared by the libmoecache translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <string>
#include <vector>

#include "moe_cache.h"

namespace moe {

constexpr int kPrepThreads = 1024;   // one CTA does the whole per-layer bookkeeping
constexpr int kMlpThreads = 512;     // 16 warps per CTA, one CTA per SM, in the expert MLP kernels
constexpr int kCopyThreads = 256;
constexpr int kCopyVecPerThread = 8; // 8 x 16 B in flight per thread
constexpr int kCopyChunkVec = kCopyThreads * kCopyVecPerThread;  // 32 KiB per CTA step

// Per-layer counters and LRU clock, device resident.
enum {
  ST_STEPS = 0, ST_HITS, ST_MISSES, ST_EVICT, ST_BYPASS, ST_COLD,
  ST_B_MISS, ST_B_BYPASS, ST_B_COLD, ST_MOVES, ST_COUNT
};

struct LayerState {
  unsigned long long clock;   // next recency stamp
  int nfree;                  // free slots: free_stack[0 .. nfree), the next miss takes the last
  unsigned counted;           // steps counted for run-time moves
  unsigned long long stats[ST_COUNT];
};

// Header of the last prepare of a layer; the lists follow in a separate
// [LST_COUNT][E] int32 block per layer.
struct RecHdr {
  int n_ids, bypass, n_distinct, n_cold, n_noncold, n_hits, n_misses, n_evictions;
  unsigned seq;   // unique number of this prepare call (per handle)
};
enum { LST_HITS = 0, LST_MISS_E, LST_MISS_SLOT, LST_MISS_EV, LST_COLD, LST_NONCOLD, LST_COUNT };

// Device error flag values (sticky until reset)
enum { DEVERR_NONE = 0, DEVERR_BAD_ID = 1, DEVERR_BARRIER = 2, DEVERR_RING = 3 };

// Grid-wide barrier state.  The cooperative MLP kernel uses count / gen
// (count returns to 0 after every barrier; gen counts completed barriers);
// the staged kernel uses arrivals, which only grows: every barrier adds one
// per CTA, so a CTA whose arrival returned a waits until arrivals reaches the
// next multiple of the grid size.
struct GridBar {
  unsigned count;
  unsigned gen;
  unsigned long long arrivals;
};

struct PrepArgs {
  // fused router (do_route != 0): logits [T, E] -> ids / w
  const float* logits;
  float* w_out;
  int do_route;
  int renorm;
  // ids [T*k] (read; written first when do_route)
  int32_t* ids;
  int T, k, E, N;
  uint8_t* cold;                     // [E] of this layer, may be null (updated by run-time moves)
  int32_t* free_stack;               // [N] of this layer
  float* counts;                     // [E] of this layer: use counts for run-time moves
  int move_interval;                 // 0 = no run-time moves
  int move_count_tokens;
  float move_decay, move_threshold;
  int32_t* slot_map;                 // [E]
  int32_t* slot_expert;              // [N]
  long long* slot_stamp;             // [N]
  int32_t* slot_aux;                 // [N]: LFU steps used, SLRU segment (1 = protected)
  unsigned* ring_cnt;                // [3 * MOE_MAX_TOPK] or null: zeroed (copy and h counts of the next MLP)
  int policy;                        // moe_evict_policy
  LayerState* st;
  RecHdr* hdr;
  int32_t* lists;                    // [LST_COUNT * E]
  int32_t* slot_ids_out;             // [T*k] or null
  unsigned long long* asg_ptr;       // [T*k] or null: expert block pointer per assignment
  unsigned long long* src_ptr;       // [T*k] or null: the expert's pinned host block
  uint8_t* pending;                  // [T*k] or null: 1 if the assignment's expert is copied this step
  unsigned long long pool_base;      // this layer's pool
  unsigned long long scratch_base;   // bypass scratch
  unsigned long long host_base;      // device-usable address of this layer's backing store
  unsigned long long stride;         // bytes between experts / slots
  unsigned long long expert_bytes;
  int* err;
  unsigned* seq_ctr;                 // per-handle prepare counter (stamps RecHdr.seq)
};

struct CopyArgs {
  const RecHdr* hdr;
  const int32_t* lists;
  int E;
  const uint8_t* host_base;          // this layer's backing store (device-usable)
  uint8_t* pool_base;                // this layer's pool
  uint8_t* scratch_base;
  unsigned long long stride;
  unsigned long long nvec;           // 16-byte vectors per expert
  unsigned* ready;                   // [E] or null: ready[e] = RecHdr.seq once expert e is copied
};

struct MlpArgs {
  const void* x;                     // [T, H] bf16 or f32
  const unsigned long long* asg_ptr; // [T*k] expert block pointers (0 = skip)
  const float* w;                    // [T*k]
  float* h;                          // [T*k, I] scratch
  void* y;                           // [T, H]
  int T, k, H, I;
  int residual;
  unsigned long long off_w2, off_s13, off_s2;
  // Optional split of the up (w13) pass: with `pending` set and phase >= 0,
  // only assignments whose pending flag equals `phase` are processed (0 =
  // expert already in HBM, 1 = expert copied in this step); otherwise all.
  const uint8_t* pending;
  int phase;
  // Read-through (fused kernel only): assignments whose expert is pending are
  // read from src_ptr (pinned host block) and written into asg_ptr (their
  // slot) while computing; bytes [tail_off, tail_off + tail_bytes) of each
  // pending block (w2 and scales) are copied by extra tasks.
  const unsigned long long* src_ptr;
  int readthrough;
  unsigned long long tail_off, tail_bytes;
  // Staged decode kernel with read-through: a copier warp per CTA moves the
  // pending blocks (blk_bytes each) from src_ptr into their slots in chunks,
  // counting landed chunks per assignment in copy_cnt[j] (w13 + gate/up
  // scales) and copy_cnt[MOE_MAX_TOPK + j] (all); prepare zeroes the counts.
  unsigned* copy_cnt;
  unsigned long long blk_bytes;
  // Device addresses [host_lo, host_hi) are the mapped pinned backing store:
  // the staged decode kernel reads blocks there with plain loads, never with
  // bulk copies (0, 0 = no host blocks).
  unsigned long long host_lo, host_hi;
  // Timing only (null otherwise): the staged kernel's copier writes, every
  // launch and without atomics, copy_span[0] = blocks copied, copy_span[1] =
  // grid size, and per CTA b copy_span[2 + 2b] / [3 + 2b] = global time its
  // copier warp issued its first chunk / had landed its last one (0, 0 when it
  // copied nothing).  Launches with more than kSpanMaxCtas CTAs record nothing.
  unsigned long long* copy_span;
  // Staged decode kernel: h_cnt[j] counts the gate/up pairs of assignment j
  // whose h is written (zeroed by prepare); null = the kernel is not used.
  unsigned* h_cnt;
};
constexpr int kSpanMaxCtas = 256;
constexpr int kSpanRecWords = 2 + 2 * kSpanMaxCtas;   // u64 words of one launch's copy-span record

// ---- launchers (k_route_prepare.cu) ----
cudaError_t launch_router(const float* logits, int T, int E, int k, int renorm,
                          int32_t* ids, float* w, cudaStream_t s);
cudaError_t launch_prepare(const PrepArgs& a, cudaStream_t s);
cudaError_t prepare_configure();   // kernel attributes, call outside capture
cudaError_t launch_copy(const CopyArgs& a, int grid, cudaStream_t s);
// Whole experts per CTA, each announced in a.ready once its bytes are written
// (consumers poll the flag instead of waiting for the whole copy).
cudaError_t launch_copy_flagged(const CopyArgs& a, int grid, cudaStream_t s);
cudaError_t launch_copy_raw(const void* src, void* dst, unsigned long long nvec, int grid,
                            cudaStream_t s);
cudaError_t launch_verify(const int32_t* slot_expert, int N, const uint8_t* pool_base,
                          const uint8_t* host_base, unsigned long long stride,
                          unsigned long long nvec, int* mismatches, cudaStream_t s);

// ---- moe_cache.cu: set the message moe_cache_last_error(NULL) returns ----
moe_status set_global_error(moe_status st, const char* msg);

// ---- moe_cache.cu: the canonical expert block, shared by every entry point ----
// Byte sizes of the block's parts [w13 | w2 | s13 | s2] for a weight format and
// shape; false if the format is unknown or the shape does not suit it.
bool block_layout(int wdtype, int H, int I, size_t* w13, size_t* w2, size_t* s13, size_t* s2);
// Elements per 16-byte chunk of a weight row (H and I must be multiples of it).
int chunk_elems(int wdtype);
// Kernel arguments for one grouped expert-MLP call, block offsets from block_layout.
MlpArgs mlp_args(int wdtype, int H, int I, int k, const void* x, const unsigned long long* asg,
                 const float* w, float* h, void* y, int T, int flags);

// ---- moe_cache.cu: per-device launch state ----
// Kernel attributes (the dynamic shared-memory opt-in, the carve-out) are set
// per device, so every record of "already configured" is kept per device and
// guarded by one mutex.
constexpr int kMaxDevices = 64;
int current_device();              // the current device, or -1 (none / index >= kMaxDevices)
std::mutex& launch_state_mutex();
int device_sm_count();             // multiprocessors of the current device (cached per device)

// ---- launchers (k_mlp.cu) ----
cudaError_t mlp_configure(int wdtype, int H, int I, int k);  // smem opt-in, call outside capture
cudaError_t launch_mlp_up(int wdtype, const MlpArgs& a, cudaStream_t s);
cudaError_t launch_mlp_down(int wdtype, const MlpArgs& a, cudaStream_t s);
// Up + down in one cooperative launch; cudaErrorNotSupported = use up/down.
cudaError_t launch_mlp_fused(int wdtype, const MlpArgs& a, GridBar* bar, int* err, cudaStream_t s);
size_t mlp_down_smem_bytes(int k, int I);
size_t mlp_up_smem_bytes(int H);

// ---- launchers (k_mlp_ring.cu): one-token expert MLP with weights staged in
// shared memory by bulk copies; cudaErrorNotSupported = use launch_mlp_fused.
// `bar` is not used by this kernel (its CTAs wait on per-expert h counts).
cudaError_t mlp_ring_configure(int wdtype, int H, int I, int k);  // call outside capture
cudaError_t launch_mlp_ring(int wdtype, const MlpArgs& a, GridBar* bar, int* err, cudaStream_t s);
// floats the staged kernel's h scratch needs (it keeps several copies of h)
size_t mlp_ring_h_floats(int k, int I);

// ---- one VMM table per layer: device rows (pool), then host rows (backing store) (table_vmm.cu)
struct VmmTable {
  unsigned long long va = 0;       // CUdeviceptr of the reserved range
  size_t bytes = 0;                // layers * pitch
  size_t pitch = 0;                // bytes per layer: pool_part + host_part
  size_t pool_part = 0, host_part = 0;
  // per layer: allocation handles (CUmemGenericAllocationHandle, 0 = none) and
  // whether each part is mapped (cuMemMap maps whole allocations only)
  std::vector<unsigned long long> hdev, hhost;
  std::vector<char> dev_mapped, host_mapped;
};
bool vmm_table_create(int device, int host_numa, int layers, size_t pool_bytes, size_t host_bytes, VmmTable* t,
                      std::string* err);
void vmm_table_destroy(VmmTable* t);

// ---- launchers (k_moe_gemm.cu): grouped expert MLP on the tensor cores for
// steps with several tokens (group by expert, tcgen05 up and down GEMMs,
// combine).  cudaErrorNotSupported = use the per-token kernels.
struct GemmBuffers {
  const int32_t* ids;      // [T*k] routed expert ids
  int E;
  int32_t* order;          // [T*k]
  int4* tiles;             // [T*k]
  int* ntiles;             // [1]
  unsigned* work;          // [2] item counters of the up / down GEMMs
  uint16_t* hb;            // [T*k, I] bf16
  float* out;              // [T*k, H] f32
  int* err;
  // experts still being copied in this step: the up GEMM waits for
  // ready[e] == hdr->seq before it reads an expert whose assignments are
  // pending (null = everything is in place before the launch)
  const uint8_t* pending;  // [T*k]
  const unsigned* ready;   // [E]
  const RecHdr* hdr;
};
bool moe_gemm_supported(int wdtype, int H, int I, int k);
cudaError_t moe_gemm_configure(int wdtype);   // call outside capture
cudaError_t launch_moe_gemm(int wdtype, const MlpArgs& a, const GemmBuffers& b, cudaStream_t s);
// the grouping (assignments expert by expert, tiles of <= `tile`) and the
// combine (y[t] = sum over j of the f32 rows, j in order, + x) of both GEMMs
cudaError_t launch_group(const int32_t* ids, int n, int E, int32_t* order, int4* tiles, int* ntiles, unsigned* work,
                         int tile, cudaStream_t s);
cudaError_t launch_combine(int wdtype, const float* out, const void* x, void* y, int T, int k, int H, int residual,
                           cudaStream_t s);

// ---- launchers (k_moe_gemm_tma.cu): the grouped expert MLP with the weights
// on the MMA's M side, operands staged by TMA from tensor maps over the pool
// and the scratch.  cudaErrorNotSupported = use launch_moe_gemm.
struct MoeTmaMaps;                // host copies of the tensor maps (opaque)
struct TmaRegions {
  unsigned long long pool_lo, pool_hi;         // device addresses the pool maps cover
  unsigned long long pool_pitch, pool_part;    // per layer: pitch, and the device rows at its start
  unsigned long long scratch_lo, scratch_hi;   // ... and the scratch maps
  void* xg;                                    // [rows, H] bf16: the activation rows in tile order
};
bool moe_gemm_tma_supported(int wdtype, int H, int I, int k);
// maps over pool [pool, pool + pool_bytes), scratch, xg [n_rows, H] and the
// bf16 h rows [n_rows, I] at hb; null when the driver gives no encoder
MoeTmaMaps* moe_gemm_tma_maps(int wdtype, int H, int I, const void* pool, size_t pool_bytes, const void* scratch,
                              size_t scratch_bytes, const void* xg, const void* hb, size_t n_rows);
void moe_gemm_tma_maps_free(MoeTmaMaps* m);
bool moe_gemm_tma_maps_ok(const MoeTmaMaps* m);
cudaError_t moe_gemm_tma_configure(int wdtype);   // call outside capture
cudaError_t launch_moe_gemm_tma(int wdtype, const MlpArgs& a, const GemmBuffers& b, const MoeTmaMaps* m,
                                const TmaRegions& r, cudaStream_t s);

}  // namespace moe
