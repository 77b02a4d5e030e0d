/*
 * moe_cache.h -- C ABI of libmoecache.so
 *
 * One MoE layer forward through a persistent per-layer GPU expert-slot cache,
 * on one NVIDIA GB300 (sm_103a).  Routed expert weights live in a pinned host
 * backing store owned by the library; each layer has a fixed-address pool of
 * N expert slots in HBM.  A step runs router top-k, the LRU hit/miss/evict
 * bookkeeping with the id->slot remap, the host-to-device copy of missed
 * experts into their victim slots, and the grouped expert MLP (gate/up w13,
 * SiLU-mul, down w2, top-k weighted combine) indexed by slot.
 *
 * Sources (web pages this library restates; cited by title and section):
 *  [vLLM #37190]  "[MoE][Offload] Run MoE models exceeding VRAM via expert CPU
 *                 offloading with GPU cache (--moe-expert-cache-size)"
 *  [llama.cpp #28248] "RFC: Persistent expert slot pool for MoE CPU offload
 *                 (--moe-expert-cache)"
 *  [Flash-Next 2x32GB] "Running 125B MoE on Two 32 GB Cards - vLLM
 *                 Optimization Edition"
 *  [vLLM #51710 article] czykbl.com article on vLLM PR #51710 (layer prefetch)
 *
 * Conventions for every entry point
 *  - Return a moe_status; on failure moe_cache_last_error() holds a message.
 *    Invalid arguments are rejected before any GPU work (MOE_EINVAL).
 *  - Pointers suffixed _d are device pointers (or pointers the device can
 *    dereference), _h are host pointers.  The caller owns every buffer it
 *    passes; the library owns the backing store, pools, scratch, device
 *    state, its copy stream and its events.
 *  - Work is stream-ordered on the caller's stream (a cudaStream_t passed as
 *    void*; NULL = legacy default stream).  Work the library issues on its
 *    internal copy stream is joined back to the caller's stream before the
 *    call returns, so later work on that stream sees the filled slots.
 *  - A handle is single-threaded and single-stream: calls on one handle must
 *    not overlap (the pages make the same single-threaded assumption,
 *    [vLLM #37190] review point 1 "Thread safety").
 *  - Device-side input errors (an expert id outside [0, E) reaching prepare)
 *    do not fault: that whole step is skipped (pool state untouched, slot ids
 *    written as -1, every assignment contributes zero to y), a sticky device
 *    error flag is set, and the next synchronising call (moe_cache_check,
 *    moe_cache_stats, moe_cache_last_prepare, moe_cache_get_state) returns
 *    MOE_ESTATE.  moe_cache_reset clears it.
 */
#ifndef MOE_CACHE_H
#define MOE_CACHE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_cache moe_cache_t;   /* opaque, library-owned */
typedef void* moe_stream_t;             /* cudaStream_t */

/* Weight formats.  Canonical expert block layout, every part row-major:
 *   [ w13 [2I, H] | w2 [H, I] | s13 [2I, H/128] | s2 [H, I/128] ]
 * w13 rows [0, I) are the gate projection, rows [I, 2I) the up projection.
 *  MOE_F32       f32 weights, no scales.
 *  MOE_BF16      bf16 weights, no scales.
 *  MOE_INT4_G128 two 4-bit codes per byte along the row, low nibble = even
 *                column; weight = (code - 8) * scale, one bf16 scale per 128
 *                consecutive columns of a row; no zero point.  H and I must be
 *                multiples of 128.  At w13 [1280, 2560] + w2 [2560, 640] this
 *                is 2,534,400 bytes = 2.417 MiB ([Flash-Next 2x32GB] section 1
 *                "What does not fit").
 *  MOE_FP8_E4M3  one OCP E4M3 byte per weight (sign, 4 exponent bits with bias
 *                7, 3 mantissa bits, exponent 0 = subnormal, no infinities,
 *                S.1111.111 = NaN); per-tensor scales ([vLLM #37190] "BF16 +
 *                FP8 per-tensor", scale buffers copied with the weights):
 *                s13 = float32 [gate scale, up scale] and s2 = float32 [down
 *                scale], each part zero-padded to 16 bytes; weight = decoded
 *                byte * its tensor's scale.  H and I must be multiples of 16.
 * Hidden states x / y are f32 for MOE_F32 and bf16 otherwise. */
typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_INT4_G128 = 2, MOE_FP8_E4M3 = 3 } moe_wdtype;

/* How missed experts reach their slot.
 *  MOE_COPY_MEMCPY  prepare reads the miss list back to the host (one small
 *                   read-back per layer step, as in [llama.cpp #28248]
 *                   "Design" item 3) and issues one cudaMemcpyAsync per miss
 *                   on the copy stream.  Not capturable in a CUDA graph.
 *  MOE_COPY_UVA     an SM copy kernel on the copy stream reads the device-side
 *                   miss list and copies from the mapped pinned host store with
 *                   16-byte loads.  No host round trip; graph-capturable.
 *  MOE_COPY_FUSED   single-token steps (decode): no separate copy launch.  A
 *                   copier warp in every CTA of the expert-MLP kernel moves the
 *                   missed experts' blocks from the pinned host store into
 *                   their slots (the host link on GB300 is coherent
 *                   NVLink-C2C) while the other warps compute with the experts
 *                   already in HBM; a missed expert's rows are used once they
 *                   have landed, so host-link traffic overlaps HBM streaming.
 *                   When the staged kernel cannot take the shape, the
 *                   cooperative kernel reads missed rows through instead.
 *                   Steps with T > 1 use the flagged copy kernel overlapped
 *                   with the grouped GEMM; moe_cache_prepare uses the UVA copy
 *                   kernel.  Graph-capturable.
 *  MOE_COPY_AUTO    at create, time cudaMemcpyAsync and the SM copy kernel on
 *                   the backing store; MEMCPY if it is more than 15% faster,
 *                   else FUSED (no host round trip per layer, so host-side
 *                   stalls cannot idle the copy engine).  moe_cache_info
 *                   reports both bandwidths and the mode chosen. */
typedef enum { MOE_COPY_AUTO = 0, MOE_COPY_MEMCPY = 1, MOE_COPY_UVA = 2, MOE_COPY_FUSED = 3 } moe_copy_mode;

/* Expert-MLP kernel of moe_forward.  AUTO: one-token steps stage the weight
 * rows that sit in HBM through shared memory with bulk copies (one persistent
 * CTA per SM, a producer warp and eight consumer warps), when the shape allows
 * it (inter a multiple of 8, two stages fit in shared memory); every other step
 * uses the cooperative up/down kernel.  PLAIN: always the cooperative kernel.
 * Each kernel's output does not depend on where an expert's bytes live (pool,
 * scratch, host); the two kernels sum in different orders and agree to
 * rounding. */
typedef enum { MOE_MLP_AUTO = 0, MOE_MLP_PLAIN = 1 } moe_mlp_kernel;

/* Which resident expert a miss evicts when no slot is free ([vLLM #37190],
 * the review thread that added a cache-policy option).  Under every policy an
 * expert used in the current step is never evicted, hits are booked before
 * misses and both go in ascending expert id.
 *   LRU   least recently used (a hit refreshes).
 *   LFU   fewest steps used since it was inserted; ties to the earliest inserted.
 *   FIFO  earliest inserted (a hit does not refresh).
 *   SLRU  two segments: misses enter the probationary one; a hit there moves
 *         the expert to the protected one's most recent end, which holds at
 *         most floor(4N/5) experts (overflow moves the protected least recent
 *         one to the probationary most recent end); a hit in the protected one
 *         refreshes it.  The victim is the probationary least recent expert,
 *         else the protected least recent one. */
typedef enum { MOE_EVICT_LRU = 0, MOE_EVICT_LFU = 1, MOE_EVICT_FIFO = 2, MOE_EVICT_SLRU = 3 } moe_evict_policy;

/* Where the pool slots and the backing store live.
 *  MOE_TABLE_SPLIT  slots in device memory (cudaMalloc), backing store in pinned,
 *                   device-mapped host memory (cudaHostAlloc): two allocations.
 *  MOE_TABLE_VMM    one virtual-address table per layer ([Flash-Next 2x32GB]
 *                   section 4.2): cuMemAddressReserve, cuMemCreate of device rows
 *                   and of host rows on the device's host NUMA node, cuMemMap of
 *                   the two side by side, so row r < N of layer l's table is pool
 *                   slot r and row N + e is expert e's backing copy (each part
 *                   rounded up to the allocation granularity).  The CPU writes the
 *                   backing store through the same addresses.  moe_cache_create
 *                   fails with MOE_ECUDA (message from the driver) if the driver
 *                   refuses any step; nothing falls back silently. */
typedef enum { MOE_TABLE_SPLIT = 0, MOE_TABLE_VMM = 1 } moe_table_layout;

typedef enum {
  MOE_OK = 0,
  MOE_EINVAL = -1,    /* bad argument, nothing done */
  MOE_ENOMEM = -2,    /* host/device allocation failed or over the HBM budget */
  MOE_ECUDA = -3,     /* a CUDA call failed; message holds cudaGetErrorString */
  MOE_ETIMEOUT = -4,  /* a bounded host wait on the GPU gave up */
  MOE_ESTATE = -5     /* call not valid in the current state, or device error flag set */
} moe_status;

/* Slot-id encoding written by prepare (one per routed id):
 *   kind << 29 | index
 *   MOE_SLOT_POOL    index = pool slot in [0, N)
 *   MOE_SLOT_SCRATCH index = bypass scratch position = rank of the expert among
 *                    the step's distinct non-cold experts (ascending id)
 *   MOE_SLOT_COLD    index = expert id; read in place from pinned host memory */
#define MOE_SLOT_KIND_SHIFT 29
#define MOE_SLOT_POOL (0u << MOE_SLOT_KIND_SHIFT)
#define MOE_SLOT_SCRATCH (1u << MOE_SLOT_KIND_SHIFT)
#define MOE_SLOT_COLD (2u << MOE_SLOT_KIND_SHIFT)
#define MOE_SLOT_INDEX_MASK ((1u << MOE_SLOT_KIND_SHIFT) - 1u)

/* moe_forward flags */
#define MOE_FWD_RESIDUAL 1   /* y = x + MoE(x) instead of y = MoE(x) */

/* Limits checked at create */
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOPK 32

typedef struct {
  int num_layers;        /* L >= 1 */
  int num_experts;       /* E, 1..MOE_MAX_EXPERTS */
  int top_k;             /* k, 1..min(E, MOE_MAX_TOPK) */
  int hidden;            /* H */
  int inter;             /* I, expert intermediate size */
  int wdtype;            /* moe_wdtype */
  int slots_per_layer;   /* N, 0..E; 0 = every step bypasses the pool */
  int max_tokens;        /* largest T per call; sizes scratch and id buffers */
  int renormalize;       /* 0: weights = softmax probs of the chosen; 1: divided by their sum */
  const uint8_t* cold_mask_h; /* [L*E] nonzero = cold (never pooled, read via UVA); NULL = none. Copied. */
  int copy_mode;         /* moe_copy_mode */
  int device;            /* CUDA device ordinal */
  size_t hbm_budget_bytes; /* cap on pool + scratch bytes; 0 = half of free device memory */
  int mlp_kernel;        /* moe_mlp_kernel */
  /* Run-time moves between the cold set and the pool ([Flash-Next 2x32GB]
   * sections 4.3-4.4).  Steps with at most move_count_tokens tokens add each
   * expert's number of assignments to a per-layer float32 use count; every
   * move_interval such steps the counts are multiplied by move_decay, and if
   * (largest count of a cold expert) - (smallest count of a non-cold expert)
   * > move_threshold, the two trade places (ties to the lower id): the cold
   * one is copied into a slot at its next use, the other is read in place from
   * then on and its slot, if it held one, is freed.  move_interval = 0: off
   * (the cold set never changes).  The pages' values: interval 8, decay
   * 2^(-1/64) (half-life 512 steps), threshold 2, count tokens 1. */
  int move_interval;
  float move_decay;      /* (0, 1] */
  float move_threshold;  /* >= 0 */
  int move_count_tokens; /* >= 1 */
  int evict_policy;      /* moe_evict_policy */
  int table_layout;      /* moe_table_layout */
  int gemm_kernel;       /* steps of several tokens: 0 = automatic (MOE_GEMM_TMA where the driver
                            and the shape allow it, else MOE_GEMM_TC); MOE_GEMM_TC = the cp.async
                            kernel even where the TMA kernel would run; MOE_GEMM_TMA = automatic */
} moe_cache_config;

/* Cumulative per-layer counters (moe_cache_stats with layer = -1 sums layers).
 * hits/misses count once per distinct expert per pool-path step
 * ([vLLM #37190] "How it works"); bypass steps count neither. */
typedef struct {
  uint64_t steps;            /* prepare calls with T > 0 */
  uint64_t hits;
  uint64_t misses;
  uint64_t evictions;
  uint64_t bypass_steps;     /* steps with distinct non-cold experts > N */
  uint64_t cold_reads;       /* distinct cold experts read in place */
  uint64_t bytes_h2d_miss;   /* misses * expert bytes */
  uint64_t bytes_h2d_bypass; /* sum over bypass steps of D * expert bytes */
  uint64_t bytes_uva_cold;   /* cold_reads * expert bytes */
  uint64_t moves;            /* run-time moves between the cold set and the pool */
} moe_cache_counters;

/* Result of the last prepare of one layer (moe_cache_last_prepare).
 * Array pointers are caller-owned host buffers of at least E entries each, or
 * NULL to skip that list. */
typedef struct {
  int n_ids;         /* T*k of that step */
  int bypass;        /* 1 if the step took the bypass path */
  int n_distinct, n_cold, n_noncold;
  int n_hits, n_misses, n_evictions;
  int32_t* hits_h;           /* [n_hits] ascending */
  int32_t* miss_expert_h;    /* [n_misses] ascending expert id */
  int32_t* miss_slot_h;      /* [n_misses] slot it was copied into */
  int32_t* miss_evicted_h;   /* [n_misses] expert evicted from that slot, -1 if free */
  int32_t* cold_h;           /* [n_cold] ascending */
  int32_t* noncold_h;        /* [n_noncold] ascending; on bypass, scratch position = index */
} moe_prepare_info;

typedef struct {
  size_t expert_bytes;       /* B_e, canonical block size */
  size_t slot_stride;        /* bytes between slots / backing experts (B_e rounded up to 256) */
  size_t pool_bytes;         /* L*N*slot_stride in HBM */
  size_t scratch_bytes;      /* bypass scratch in HBM */
  size_t backing_bytes;      /* L*E*slot_stride pinned host */
  int copy_mode;             /* the mode in use (AUTO resolved) */
  double memcpy_gbs;         /* measured at create (AUTO only, else 0) */
  double uva_gbs;            /* measured at create (AUTO only, else 0) */
  uint64_t kernel_launches;  /* kernels launched by this handle so far */
  int scratch_experts;       /* bypass scratch capacity in experts */
  int table_layout;          /* moe_table_layout in use */
  int gemm_kernel;           /* grouped expert MLP of multi-token steps: MOE_GEMM_* */
} moe_cache_info;

/* moe_cache_info.gemm_kernel: which kernel runs steps of several tokens.
 *  MOE_GEMM_NONE  the per-token kernels (max_tokens 1, f32 weights, or a shape
 *                 the tensor-core kernels do not take)
 *  MOE_GEMM_TC    tcgen05, tokens on M, operands staged with cp.async
 *  MOE_GEMM_TMA   tcgen05, weight rows on N (256 per instruction) and the tile's
 *                 tokens on M = 64, operands staged by TMA from tensor maps,
 *                 warp-specialised with dequantisation warps (the default when
 *                 the CUDA driver provides tensor-map encoding) */
#define MOE_GEMM_NONE 0
#define MOE_GEMM_TC 1
#define MOE_GEMM_TMA 2

/* Per-phase GPU time accumulated while timing is on (CUDA events on the
 * stream each kernel is launched on).  Works under stream capture too: the
 * events become graph nodes and are read after the graph has run. */
typedef struct {
  double route_ms, copy_ms, up_ms, down_ms;   /* router+prepare, miss/bypass copy, w13, w2 */
  uint64_t route_n, copy_n, up_n, down_n;     /* launches timed */
  /* moe_forward normally runs w13 and w2 in one fused kernel, timed under
   * up_ms / up_n (down_n then stays 0); separate up/down launches are timed
   * under their own fields. */
} moe_cache_timing;

/* ---------------------------------------------------------------- lifecycle */

/* Allocate the pinned backing store (L*E experts), the per-layer pools
 * (fixed addresses for the handle's life, [vLLM #37190] "torch.compile
 * compatibility"), the bypass scratch (min(E, max_tokens*k) experts), device
 * state (all slots free), the copy stream and events.  Fails with MOE_ENOMEM
 * when pools + scratch exceed the budget (default: half of free device memory,
 * [llama.cpp #28248] "Design" item 4) -- never a silent downgrade
 * ([vLLM #37190] "Changes": errors instead of silent downgrades).
 * On failure *out is NULL and moe_cache_last_error(NULL) has the reason. */
moe_status moe_cache_create(const moe_cache_config* cfg, moe_cache_t** out);

/* Free everything.  NULL is ignored.  Synchronises the device first. */
void moe_cache_destroy(moe_cache_t* c);

/* Message of the last failure on c, or of the last failed create when c is NULL. */
const char* moe_cache_last_error(const moe_cache_t* c);

/* Bytes of one canonical expert block for a format and shape. */
moe_status moe_cache_expert_bytes(int wdtype, int hidden, int inter, size_t* bytes);

moe_status moe_cache_get_info(moe_cache_t* c, moe_cache_info* out);

/* -------------------------------------------------------------- weights in */

/* Host address (pinned, device-mapped) where expert (layer, expert)'s block
 * lives, so a caller can write it in place; *stride_bytes = slot stride. */
moe_status moe_cache_backing_ptr(moe_cache_t* c, int layer, int expert,
                                 void** block_h, size_t* stride_bytes);

/* Copy one canonical block (bytes must equal expert_bytes) into the backing
 * store.  Host-synchronous.  If the expert currently sits in a pool slot the
 * slot is refreshed too, so pool and backing never disagree. */
moe_status moe_cache_load_expert(moe_cache_t* c, int layer, int expert,
                                 const void* block_h, size_t bytes);

/* ------------------------------------------------------------- hot path */

/* Router top-k: logits_d f32 [T, E] -> ids_d int32 [T, k], w_d f32 [T, k].
 * ids are the k largest logits in descending order, lower id first on equal
 * logits ([Flash-Next 2x32GB] section 4.2, "the lower id wins"); NaN ranks
 * below every number.  w = softmax over all E of the chosen (divided by their
 * sum when renormalize).  One warp per token. */
moe_status moe_cache_router(moe_cache_t* c, const float* logits_d, int T,
                            int32_t* ids_d, float* w_d, moe_stream_t stream);

/* Pool bookkeeping + remap + copies for one layer step.
 * ids_d int32 [T, k] (device).  Distinct ids are taken in ascending order
 * ([vLLM #37190] "How it works": topk_ids.unique()).  Cold experts are read
 * in place.  If the distinct non-cold count D exceeds N the step bypasses the
 * pool: all D experts are copied to scratch in ascending id order and the
 * LRU state is untouched ([llama.cpp #28248] "Why not the other approaches on
 * the table").  Otherwise hits are touched first (ascending), then each miss
 * (ascending) takes the highest free slot or evicts the least recently used
 * slot not used this step ([vLLM #37190] "Architecture", OrderedDict LRU), and
 * is copied host-to-device into that slot.  slot_ids_d int32 [T, k] receives
 * the encoded slot ids (NULL = don't write).  On return the copies are
 * ordered before later work on `stream`. */
moe_status moe_cache_prepare(moe_cache_t* c, int layer, const int32_t* ids_d, int T,
                             int32_t* slot_ids_d, moe_stream_t stream);

/* Read back the last prepare of `layer` (synchronises the device). */
moe_status moe_cache_last_prepare(moe_cache_t* c, int layer, moe_prepare_info* out);

/* The whole layer: router + prepare + copies + grouped expert MLP.
 * x_d [T, H] and y_d [T, H] (bf16, or f32 for MOE_F32) are caller-owned and
 * may not alias; logits_d f32 [T, E].  y[t] = sum_j w[t,j] * W2_e silu(Wg_e x)
 * * (Wu_e x) summed in j order, with weights read from the slot / scratch /
 * cold host copy of expert e ([vLLM #37190] "How it works": fused_experts on
 * slot buffers with remapped ids).  flags: MOE_FWD_RESIDUAL adds x. */
moe_status moe_forward(moe_cache_t* c, int layer, const void* x_d, const float* logits_d,
                       int T, void* y_d, int flags, moe_stream_t stream);

/* Grouped expert MLP alone, no cache: for each assignment a = t*k + j,
 * block_ptrs_d[a] is a device-readable, 16-byte aligned pointer to expert e's
 * canonical block (HBM or mapped pinned host; 0 = skip, contributes zero) and
 * w_d[a] its weight.  h_scratch_d is caller-provided scratch of T*k*I floats.  Same
 * arithmetic and summation order as moe_forward. */
moe_status moe_expert_mlp(int wdtype, int hidden, int inter, int top_k,
                          const void* x_d, const uint64_t* block_ptrs_d, const float* w_d,
                          int T, float* h_scratch_d, void* y_d, int flags,
                          moe_stream_t stream);

/* Allocation-free variant of moe_expert_mlp (the pages have no counterpart;
 * this entry point exists for callers of this library that cannot allocate
 * device memory where they call it: plugins whose host framework's caching
 * allocator owns all device memory, and latency-critical loops that must not
 * hit cudaMalloc's implicit device synchronisation).  Same arguments, shape
 * rules, block layout, arithmetic and results as moe_expert_mlp, minus
 * h_scratch_d: the intermediate h lives in a 2 MiB array compiled into the
 * library, which every GPU that loads the library holds until the process
 * exits.  The call allocates nothing.
 *  - Rejects T * top_k * inter > MOE_NOALLOC_MAX_SCRATCH_FLOATS (MOE_EINVAL).
 *  - All calls on a device share the array and it keeps the last call's
 *    contents (nothing in it needs to start at zero); calls whose kernels
 *    overlap on the GPU race on it -- order them on one stream.
 *  - The first call on each device looks up the array's device address
 *    (one-time set-up, with that device current); make it before any stream
 *    capture. */
#define MOE_NOALLOC_MAX_SCRATCH_FLOATS (1 << 19)
moe_status moe_expert_mlp_noalloc(int wdtype, int hidden, int inter, int top_k,
                                  const void* x_d, const uint64_t* block_ptrs_d, const float* w_d,
                                  int T, void* y_d, int flags, moe_stream_t stream);

/* End-to-end step from host buffers: copies x_h [T, H] and logits_h
 * [L, T, E] (pinned host recommended) to the device, runs every layer as
 * x <- x + MoE_l(x), copies the final x back to y_h [T, H] and waits for it
 * (bounded wait, MOE_ETIMEOUT after timeout_ms). */
moe_status moe_model_step_host(moe_cache_t* c, const void* x_h, const float* logits_h, int T,
                               void* y_h, int timeout_ms, moe_stream_t stream);

/* ------------------------------------------------------------ inspection */

/* Cumulative counters of one layer, or the sum over layers (layer = -1).
 * Synchronises the device. */
moe_status moe_cache_stats(moe_cache_t* c, int layer, moe_cache_counters* out);

/* Device state of one layer (synchronises): slot_map_h int32[E] (-1 absent),
 * slot_expert_h int32[N] (-1 free), slot_stamp_h int64[N] (recency stamp,
 * larger = more recent).  Any pointer may be NULL.  *n_free_h (may be NULL)
 * receives the free-slot count. */
moe_status moe_cache_get_state(moe_cache_t* c, int layer, int32_t* slot_map_h,
                               int32_t* slot_expert_h, int64_t* slot_stamp_h, int32_t* n_free_h);

/* Compare every occupied slot of `layer` with its expert's backing block on
 * the GPU; *mismatched_slots receives the number of slots whose bytes differ
 * ([vLLM #37190] "Test results": test_gpu_buffer_matches_source_weights).
 * Synchronises the device. */
moe_status moe_cache_verify_slots(moe_cache_t* c, int layer, int* mismatched_slots);

/* Current cold set of one layer (it changes only with run-time moves):
 * cold_h[E] host buffer, 1 = cold.  Synchronises the device. */
moe_status moe_cache_get_cold(moe_cache_t* c, int layer, uint8_t* cold_h);

/* Device pointers of a layer's pool and of the bypass scratch. */
moe_status moe_cache_pool_ptrs(moe_cache_t* c, int layer, void** pool_d, void** scratch_d);

/* Synchronise and report the sticky device error flag (MOE_ESTATE if set). */
moe_status moe_cache_check(moe_cache_t* c);

/* Empty every pool, zero the counters and the device error flag. */
moe_status moe_cache_reset(moe_cache_t* c);

/* Per-phase event timing: on != 0 starts (and clears) accumulation; capacity
 * = launches per phase to reserve events for (0 = 4096).  Reserve enough
 * before a stream capture: no events are created while capturing, and
 * launches past the reserve go untimed. */
moe_status moe_cache_set_timing(moe_cache_t* c, int on, int capacity);
/* Synchronises the device and returns the accumulated per-phase times. */
moe_status moe_cache_read_timing(moe_cache_t* c, moe_cache_timing* out);
/* Per-launch record of the expert-MLP phase (synchronises): ms_h[i] = GPU
 * time of the i-th timed MLP launch, misses_h[i] = misses of that layer step
 * (copied on the device, so it is right under graph replay too).  Up to `cap`
 * records; *n receives the number available. */
moe_status moe_cache_read_timing_launches(moe_cache_t* c, float* ms_h, int32_t* misses_h, int cap,
                                          int* n);

/* Copy span of each timed expert-MLP launch (synchronises): for launch i,
 * rec_h[3i] / rec_h[3i + 1] = %globaltimer ns when the staged kernel's copier
 * warps issued their first chunk of missed (or bypassed) expert bytes / when
 * their last chunk had landed in its slot, rec_h[3i + 2] = experts copied in
 * that launch.  (rec_h[3i + 1] - rec_h[3i]) is the host-link transfer time of
 * the launch's copies ([Flash-Next 2x32GB] section 3.2, "the cost of one host
 * read"); records of launches that copied nothing, or that ran another kernel
 * or copy mode, hold (~0, 0, 0).  Indexed like moe_cache_read_timing_launches.
 * Up to `cap` records; *n receives the number available. */
moe_status moe_cache_read_copy_spans(moe_cache_t* c, uint64_t* rec_h, int cap, int* n);

#ifdef __cplusplus
}
#endif
#endif /* MOE_CACHE_H */
