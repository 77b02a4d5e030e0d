// Host side of libmoecache.so: the C ABI declared in include/moe_cache.h.
//
// Owns the pinned backing store (all experts of all layers, device-mapped),
// the fixed-address HBM slot pools (vLLM PR #37190 "Run MoE models exceeding
// VRAM via expert CPU offloading with GPU cache", "Architecture":
// GPUSlotManager + CPUBackingStore), the bypass scratch, the per-layer device
// state, one copy stream and the events that join it to the caller's stream
// (czykbl.com article on vLLM PR #51710, "为什么还要处理 CUDA Graph": copies on
// a side stream must be joined back by an event).

#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cstdio>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

#include "internal.cuh"

using namespace moe;

namespace {

std::string g_create_error;

enum { TM_ROUTE = 0, TM_COPY, TM_UP, TM_DOWN, TM_COUNT };

struct TimingPool {
  std::vector<cudaEvent_t> beg, end;
  size_t used = 0;
};

constexpr int kDefaultTimingCap = 4096;

size_t round_up(size_t v, size_t m) { return (v + m - 1) / m * m; }

size_t act_bytes(int wd) { return wd == MOE_F32 ? 4 : 2; }

}  // namespace

bool moe::block_layout(int wd, int H, int I, size_t* w13, size_t* w2, size_t* s13, size_t* s2) {
  const size_t h = (size_t)H, i = (size_t)I;
  switch (wd) {
    case MOE_F32: *w13 = 2 * i * h * 4; *w2 = h * i * 4; *s13 = *s2 = 0; return true;
    case MOE_BF16: *w13 = 2 * i * h * 2; *w2 = h * i * 2; *s13 = *s2 = 0; return true;
    case MOE_INT4_G128:
      if (H % 128 || I % 128) return false;
      *w13 = 2 * i * h / 2; *w2 = h * i / 2;
      *s13 = 2 * i * (h / 128) * 2; *s2 = h * (i / 128) * 2;
      return true;
    case MOE_FP8_E4M3:
      if (H % 16 || I % 16) return false;
      *w13 = 2 * i * h; *w2 = h * i; *s13 = 16; *s2 = 16;
      return true;
  }
  return false;
}

int moe::chunk_elems(int wd) {
  return wd == MOE_F32 ? 4 : (wd == MOE_BF16 ? 8 : (wd == MOE_FP8_E4M3 ? 16 : 32));
}

MlpArgs moe::mlp_args(int wd, int H, int I, int k, const void* x, const unsigned long long* asg,
                      const float* w, float* h, void* y, int T, int flags) {
  size_t w13 = 0, w2 = 0, s13 = 0, s2 = 0;
  block_layout(wd, H, I, &w13, &w2, &s13, &s2);
  MlpArgs a{};
  a.x = x;
  a.asg_ptr = asg;
  a.w = w;
  a.h = h;
  a.y = y;
  a.T = T;
  a.k = k;
  a.H = H;
  a.I = I;
  a.residual = (flags & MOE_FWD_RESIDUAL) ? 1 : 0;
  a.off_w2 = w13;
  a.off_s13 = w13 + w2;
  a.off_s2 = w13 + w2 + s13;
  return a;
}

namespace {
std::mutex g_launch_state_mu;
int g_device_sms[moe::kMaxDevices];
}  // namespace

int moe::current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

std::mutex& moe::launch_state_mutex() { return g_launch_state_mu; }

int moe::device_sm_count() {
  const int dev = current_device();
  if (dev < 0) return 1;
  std::lock_guard<std::mutex> lock(g_launch_state_mu);
  if (g_device_sms[dev] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    g_device_sms[dev] = v > 0 ? v : 1;
  }
  return g_device_sms[dev];
}

struct moe_cache {
  moe_cache_config cfg{};
  int L = 0, E = 0, K = 0, H = 0, I = 0, N = 0, maxT = 0, wd = 0;
  size_t Be = 0, stride = 0, nvec = 0, off_w2 = 0, off_s13 = 0, off_s2 = 0;
  int scratch_n = 0;
  uint8_t* backing_h = nullptr;   // pinned, device-mapped (or the host rows of the VMM table)
  uint8_t* backing_dv = nullptr;  // its device-usable address
  size_t pool_pitch = 0;          // bytes from one layer's pool to the next
  size_t back_pitch = 0;          // bytes from one layer's backing store to the next
  VmmTable vmm;                   // MOE_TABLE_VMM: the reserved table of all layers
  bool staged_mlp = false;        // one-token steps may use the staged-weight kernel
  bool gemm_mlp = false;          // multi-token steps may use the tensor-core grouped GEMM
  int32_t* order_d = nullptr;     // grouped GEMM: assignments grouped by expert
  int4* tiles_d = nullptr;        //               tiles of up to 128 assignments
  int* ntiles_d = nullptr;
  float* gout_d = nullptr;        //               [T*k, H] f32 per-assignment outputs
  uint8_t* xg_d = nullptr;        //               [T*k, H] bf16 activation rows in tile order (TMA GEMM)
  MoeTmaMaps* tma = nullptr;      //               tensor maps of the TMA GEMM (null: the cp.async GEMM)
  size_t scratch_bytes = 0;
  unsigned* seq_d = nullptr;      // prepare counter (RecHdr.seq)
  unsigned* ready_d = nullptr;    // [E] expert e copied in the step with that seq
  std::vector<uint8_t> cold_h;
  bool any_cold = false;
  uint8_t* pool_d = nullptr;
  uint8_t* scratch_d = nullptr;
  uint8_t* cold_d = nullptr;
  int32_t* fstack_d = nullptr;    // [L][N] free-slot stacks
  float* counts_d = nullptr;      // [L][E] use counts for run-time moves (null when off)
  int32_t* slot_map_d = nullptr;
  int32_t* slot_expert_d = nullptr;
  long long* slot_stamp_d = nullptr;
  int32_t* slot_aux_d = nullptr;  // [L][N] per-slot policy state
  LayerState* state_d = nullptr;
  RecHdr* hdr_d = nullptr;
  int32_t* lists_d = nullptr;
  unsigned long long* asg_d = nullptr;
  unsigned long long* src_d = nullptr;   // host block of each assignment's expert
  uint8_t* pend_d = nullptr;
  int32_t* ids_d = nullptr;
  float* w_d = nullptr;
  float* h_d = nullptr;
  int* err_d = nullptr;
  int* verify_d = nullptr;
  GridBar* bar_d = nullptr;       // grid barrier of the fused MLP kernel
  unsigned* ring_cnt_d = nullptr; // [3 * MOE_MAX_TOPK] staged kernel: copier's landed-chunk counts, h counts
  RecHdr* hdr_h = nullptr;        // pinned mirror for MEMCPY mode
  int32_t* lists_h = nullptr;
  uint8_t* xs_d[2] = {nullptr, nullptr};
  float* logits_stage_d = nullptr;
  cudaStream_t copy_stream = nullptr;
  cudaStream_t cap_stream = nullptr;            // capture stream of the host-buffer model step
  std::vector<cudaGraphExec_t> step_graph;      // [maxT + 1]: all layers of a T-token step, captured once
  std::vector<unsigned long long> step_graph_launches;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_sync = nullptr;
  int copy_mode = MOE_COPY_UVA;
  int copy_grid = 0;
  int flag_grid = 0;              // CTAs of the flagged (overlapped) copy: enough to fill the host link
  double memcpy_gbs = 0, uva_gbs = 0;
  unsigned long long launches = 0;
  bool timing_on = false;
  TimingPool tp[TM_COUNT];
  int32_t* tm_miss_d = nullptr;   // per timed MLP launch: misses of that layer step
  unsigned long long* tm_span_d = nullptr;   // per timed MLP launch: copier span record [3] (staged kernel)
  size_t tm_miss_cap = 0;
  std::string err;
};

namespace {

// layer l's pool slots, and its backing store as the host and the device see it
uint8_t* pool_of(const moe_cache* c, int l) { return c->pool_d + (size_t)l * c->pool_pitch; }
uint8_t* back_h_of(const moe_cache* c, int l) { return c->backing_h + (size_t)l * c->back_pitch; }
uint8_t* back_d_of(const moe_cache* c, int l) { return c->backing_dv + (size_t)l * c->back_pitch; }

moe_status fail(moe_cache* c, moe_status st, const std::string& msg) {
  if (c) c->err = msg;
  else g_create_error = msg;
  return st;
}

moe_status cuda_fail(moe_cache* c, cudaError_t e, const char* what) {
  std::string m = std::string(what) + ": " + cudaGetErrorString(e);
  return fail(c, MOE_ECUDA, m);
}

#define CK(c, call)                                   \
  do {                                                \
    cudaError_t _e = (call);                          \
    if (_e != cudaSuccess) return cuda_fail(c, _e, #call); \
  } while (0)

bool capturing(cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) != cudaSuccess) return false;
  return st == cudaStreamCaptureStatusActive;
}

// ---- per-phase event timing ------------------------------------------------
int tm_begin(moe_cache* c, int cat, cudaStream_t s) {
  if (!c->timing_on) return -1;
  TimingPool& p = c->tp[cat];
  const bool cap = capturing(s);
  if (p.used == p.beg.size()) {
    if (cap) return -1;   // cannot create events mid-capture safely; skip this sample
    for (int i = 0; i < 256; ++i) {
      cudaEvent_t a, b;
      if (cudaEventCreate(&a) != cudaSuccess) return -1;
      if (cudaEventCreate(&b) != cudaSuccess) { cudaEventDestroy(a); return -1; }
      p.beg.push_back(a);
      p.end.push_back(b);
    }
  }
  const int idx = (int)p.used++;
  if (cap) cudaEventRecordWithFlags(p.beg[idx], s, cudaEventRecordExternal);
  else cudaEventRecord(p.beg[idx], s);
  return idx;
}

void tm_end(moe_cache* c, int cat, int idx, cudaStream_t s) {
  if (idx < 0) return;
  if (capturing(s)) cudaEventRecordWithFlags(c->tp[cat].end[idx], s, cudaEventRecordExternal);
  else cudaEventRecord(c->tp[cat].end[idx], s);
}

// After a timed MLP launch: copy that layer step's miss count next to its
// events (a device-to-device copy, so graph replays refresh it too).
void tm_note_misses(moe_cache* c, int idx, int layer, cudaStream_t s) {
  if (idx < 0 || c->tm_miss_d == nullptr || (size_t)idx >= c->tm_miss_cap) return;
  cudaMemcpyAsync(c->tm_miss_d + idx, &c->hdr_d[layer].n_misses, sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
}

// The copier span record of a timed staged-MLP launch (null when timing is
// off or the record does not fit); the kernel rewrites all of it every launch.
unsigned long long* tm_span_slot(moe_cache* c, int idx) {
  if (idx < 0 || c->tm_span_d == nullptr || (size_t)idx >= c->tm_miss_cap) return nullptr;
  return c->tm_span_d + (size_t)kSpanRecWords * idx;
}

moe_status wait_event_bounded(moe_cache* c, cudaEvent_t ev, int timeout_ms) {
  const auto t0 = std::chrono::steady_clock::now();
  int spins = 0;
  for (;;) {
    const cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return MOE_OK;
    if (e != cudaErrorNotReady) return cuda_fail(c, e, "cudaEventQuery");
    const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                        std::chrono::steady_clock::now() - t0).count();
    if (ms > timeout_ms) return fail(c, MOE_ETIMEOUT, "timed out waiting for the GPU");
    if (++spins > 2000) std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
}

moe_status check_layer(moe_cache* c, int layer) {
  if (!c) return fail(nullptr, MOE_EINVAL, "null handle");
  if (layer < 0 || layer >= c->L) return fail(c, MOE_EINVAL, "layer out of range");
  return MOE_OK;
}

moe_status device_error(moe_cache* c) {
  int e = 0;
  CK(c, cudaMemcpy(&e, c->err_d, sizeof(int), cudaMemcpyDeviceToHost));
  if (e == DEVERR_BAD_ID)
    return fail(c, MOE_ESTATE, "device error: an expert id outside [0, E) reached prepare; that step was skipped");
  if (e == DEVERR_BARRIER)
    return fail(c, MOE_ESTATE, "device error: the fused MLP kernel's grid barrier timed out; outputs are invalid, call moe_cache_reset");
  if (e == DEVERR_RING)
    return fail(c, MOE_ESTATE, "device error: a staged-weight wait in the decode MLP kernel timed out; outputs are invalid, call moe_cache_reset");
  if (e != DEVERR_NONE) return fail(c, MOE_ESTATE, "device error flag set");
  return MOE_OK;
}

// ---- the three stages of a layer step ------------------------------------
moe_status run_prepare(moe_cache* c, int layer, const float* logits, const int32_t* ids_in,
                       int T, int32_t* slot_ids_out, cudaStream_t s) {
  PrepArgs a{};
  a.T = T;
  a.k = c->K;
  a.E = c->E;
  a.N = c->N;
  a.renorm = c->cfg.renormalize;
  a.cold = c->any_cold ? c->cold_d + (size_t)layer * c->E : nullptr;
  a.free_stack = c->fstack_d + (size_t)layer * c->N;
  if (c->counts_d != nullptr && c->any_cold) {
    a.counts = c->counts_d + (size_t)layer * c->E;
    a.move_interval = c->cfg.move_interval;
    a.move_count_tokens = c->cfg.move_count_tokens;
    a.move_decay = c->cfg.move_decay;
    a.move_threshold = c->cfg.move_threshold;
  }
  a.slot_map = c->slot_map_d + (size_t)layer * c->E;
  a.slot_expert = c->slot_expert_d + (size_t)layer * c->N;
  a.slot_stamp = c->slot_stamp_d + (size_t)layer * c->N;
  a.slot_aux = c->slot_aux_d + (size_t)layer * c->N;
  a.ring_cnt = c->ring_cnt_d;
  a.policy = c->cfg.evict_policy;
  a.st = c->state_d + layer;
  a.hdr = c->hdr_d + layer;
  a.lists = c->lists_d + (size_t)layer * LST_COUNT * c->E;
  a.slot_ids_out = slot_ids_out;
  a.asg_ptr = c->asg_d;
  a.src_ptr = c->src_d;
  a.pending = c->pend_d;
  a.pool_base = (unsigned long long)pool_of(c, layer);
  a.scratch_base = (unsigned long long)c->scratch_d;
  a.host_base = (unsigned long long)back_d_of(c, layer);
  a.stride = c->stride;
  a.expert_bytes = c->Be;
  a.err = c->err_d;
  a.seq_ctr = c->seq_d;
  const int ti = tm_begin(c, TM_ROUTE, s);
  if (logits) {
    a.w_out = c->w_d;
    a.ids = c->ids_d;
    if (T <= 64) {
      a.logits = logits;
      a.do_route = 1;
    } else {
      CK(c, launch_router(logits, T, c->E, c->K, c->cfg.renormalize, c->ids_d, c->w_d, s));
      c->launches++;
    }
  } else {
    a.ids = const_cast<int32_t*>(ids_in);
  }
  CK(c, launch_prepare(a, s));
  c->launches++;
  tm_end(c, TM_ROUTE, ti, s);
  return MOE_OK;
}

// The expert MLP of one layer step: the staged-weight kernel for one-token
// steps and the tensor-core grouped GEMM for multi-token steps, where the
// shape allows it; else the cooperative up/down kernel.  `*launches` = the
// kernels launched.  cudaErrorNotSupported (or a too-large cooperative grid)
// = none fits; the caller then runs the separate up and down kernels.
cudaError_t launch_layer_mlp(moe_cache* c, const MlpArgs& m, cudaStream_t s, int* launches,
                             int overlap_layer = -1) {
  *launches = 1;
  if (c->staged_mlp && m.T == 1) {
    const cudaError_t e = launch_mlp_ring(c->wd, m, c->bar_d, c->err_d, s);
    if (e != cudaErrorNotSupported) return e;
  }
  if (c->gemm_mlp && m.T > 1) {
    GemmBuffers b{};
    b.ids = c->ids_d;
    b.E = c->E;
    b.order = c->order_d;
    b.tiles = c->tiles_d;
    b.ntiles = c->ntiles_d;
    b.work = reinterpret_cast<unsigned*>(c->ntiles_d + 2);
    b.hb = reinterpret_cast<uint16_t*>(c->h_d);
    b.out = c->gout_d;
    b.err = c->err_d;
    if (overlap_layer >= 0) {
      b.pending = c->pend_d;
      b.ready = c->ready_d;
      b.hdr = c->hdr_d + overlap_layer;
    }
    if (c->tma != nullptr) {
      TmaRegions r{};
      r.pool_lo = (unsigned long long)c->pool_d;
      r.pool_hi = r.pool_lo + (unsigned long long)c->L * c->pool_pitch;
      r.pool_pitch = c->pool_pitch;
      r.pool_part = c->vmm.va ? c->vmm.pool_part : c->pool_pitch;
      r.scratch_lo = (unsigned long long)c->scratch_d;
      r.scratch_hi = r.scratch_lo + c->scratch_bytes;
      r.xg = c->xg_d;
      const cudaError_t e = launch_moe_gemm_tma(c->wd, m, b, c->tma, r, s);
      if (e != cudaErrorNotSupported) {
        *launches = 5;
        return e;
      }
    }
    const cudaError_t e = launch_moe_gemm(c->wd, m, b, s);
    if (e != cudaErrorNotSupported) {
      *launches = 4;
      return e;
    }
  }
  return launch_mlp_fused(c->wd, m, c->bar_d, c->err_d, s);
}

// After the prepare kernel of a layer step: the missed (or, on bypass, all
// non-cold) experts are copied on the copy stream, forked from the caller's
// stream right after prepare and joined back before the expert MLP runs.  (An
// up pass over the experts already in HBM could overlap the copy, but the
// one-CTA-per-SM up kernel cannot share SMs with the copy kernel, so the
// overlap was measured slower; the kernels keep the pass filter for callers
// that want it.)  `mlp` null = prepare only.
moe_status run_copies_and_mlp(moe_cache* c, int layer, cudaStream_t s, const MlpArgs* mlp) {
  uint8_t* pool = pool_of(c, layer);
  if (c->copy_mode == MOE_COPY_FUSED && mlp != nullptr && mlp->T == 1) {
    // read-through: the fused expert-MLP kernel fills the slots itself
    MlpArgs m = *mlp;
    m.readthrough = 1;
    m.pending = c->pend_d;
    m.src_ptr = c->src_d;
    m.phase = -1;
    m.tail_off = c->off_w2;
    m.tail_bytes = c->Be - c->off_w2;
    m.copy_cnt = c->ring_cnt_d;
    m.blk_bytes = c->Be;
    const int ti = tm_begin(c, TM_UP, s);
    m.copy_span = tm_span_slot(c, ti);
    int nl = 1;
    const cudaError_t fe = launch_layer_mlp(c, m, s, &nl);
    if (fe == cudaSuccess) {
      c->launches += nl;
      tm_end(c, TM_UP, ti, s);
      tm_note_misses(c, ti, layer, s);
      return MOE_OK;
    }
    if (fe != cudaErrorNotSupported && fe != cudaErrorCooperativeLaunchTooLarge)
      return cuda_fail(c, fe, "fused expert MLP launch");
    cudaGetLastError();
    tm_end(c, TM_UP, ti, s);
    // no co-resident grid for this shape: copy kernel, then the MLP
  }
  const bool memcpy_mode = c->copy_mode == MOE_COPY_MEMCPY;
  if (mlp != nullptr && mlp->T > 1 && c->gemm_mlp && !memcpy_mode) {
    // Multi-token step on the tensor cores: the copy kernel publishes every
    // expert as it lands and the grouped GEMM starts on the first ones while
    // later ones are still crossing the host link; the caller's stream joins
    // the copy stream after the MLP.
    CK(c, cudaEventRecord(c->ev_fork, s));
    CK(c, cudaStreamWaitEvent(c->copy_stream, c->ev_fork, 0));
    int ti = tm_begin(c, TM_COPY, c->copy_stream);
    CopyArgs a{};
    a.hdr = c->hdr_d + layer;
    a.lists = c->lists_d + (size_t)layer * LST_COUNT * c->E;
    a.E = c->E;
    a.host_base = back_d_of(c, layer);
    a.pool_base = pool;
    a.scratch_base = c->scratch_d;
    a.stride = c->stride;
    a.nvec = c->nvec;
    a.ready = c->ready_d;
    CK(c, launch_copy_flagged(a, c->flag_grid, c->copy_stream));
    c->launches++;
    tm_end(c, TM_COPY, ti, c->copy_stream);
    CK(c, cudaEventRecord(c->ev_join, c->copy_stream));
    ti = tm_begin(c, TM_UP, s);
    int nl = 1;
    const cudaError_t fe = launch_layer_mlp(c, *mlp, s, &nl, layer);
    if (fe == cudaSuccess) {
      c->launches += nl;
      tm_end(c, TM_UP, ti, s);
      CK(c, cudaStreamWaitEvent(s, c->ev_join, 0));
      return MOE_OK;
    }
    if (fe != cudaErrorNotSupported && fe != cudaErrorCooperativeLaunchTooLarge)
      return cuda_fail(c, fe, "grouped expert MLP launch");
    cudaGetLastError();
    tm_end(c, TM_UP, ti, s);
    // the grouped GEMM could not be launched: join, then the per-token kernels
    CK(c, cudaStreamWaitEvent(s, c->ev_join, 0));
    ti = tm_begin(c, TM_UP, s);
    CK(c, launch_mlp_up(c->wd, *mlp, s));
    c->launches++;
    tm_end(c, TM_UP, ti, s);
    ti = tm_begin(c, TM_DOWN, s);
    CK(c, launch_mlp_down(c->wd, *mlp, s));
    c->launches++;
    tm_end(c, TM_DOWN, ti, s);
    return MOE_OK;
  }
  if (memcpy_mode && capturing(s))
    return fail(c, MOE_ESTATE, "MOE_COPY_MEMCPY needs a host decision per step and cannot be captured; use MOE_COPY_UVA");
  CK(c, cudaEventRecord(c->ev_fork, s));
  bool joined = true;
  if (memcpy_mode) {
    // read the copy list back (one small read-back per layer step)
    CK(c, cudaMemcpyAsync(c->hdr_h, c->hdr_d + layer, sizeof(RecHdr), cudaMemcpyDeviceToHost, s));
    CK(c, cudaMemcpyAsync(c->lists_h, c->lists_d + (size_t)layer * LST_COUNT * c->E,
                          sizeof(int32_t) * LST_COUNT * c->E, cudaMemcpyDeviceToHost, s));
    CK(c, cudaEventRecord(c->ev_sync, s));
  } else {
    CK(c, cudaStreamWaitEvent(c->copy_stream, c->ev_fork, 0));
    const int ti = tm_begin(c, TM_COPY, c->copy_stream);
    CopyArgs a{};
    a.hdr = c->hdr_d + layer;
    a.lists = c->lists_d + (size_t)layer * LST_COUNT * c->E;
    a.E = c->E;
    a.host_base = back_d_of(c, layer);
    a.pool_base = pool;
    a.scratch_base = c->scratch_d;
    a.stride = c->stride;
    a.nvec = c->nvec;
    CK(c, launch_copy(a, c->copy_grid, c->copy_stream));
    c->launches++;
    tm_end(c, TM_COPY, ti, c->copy_stream);
    CK(c, cudaEventRecord(c->ev_join, c->copy_stream));
  }
  if (memcpy_mode) {
    moe_status st = wait_event_bounded(c, c->ev_sync, 30000);
    if (st != MOE_OK) return st;
    const RecHdr h = *c->hdr_h;
    const int n = h.bypass ? h.n_noncold : h.n_misses;
    joined = n > 0;
    if (n > 0) {
      // one cudaMemcpyAsync per expert on the copy stream
      CK(c, cudaStreamWaitEvent(c->copy_stream, c->ev_fork, 0));
      const int ti = tm_begin(c, TM_COPY, c->copy_stream);
      const int32_t* src = c->lists_h + (h.bypass ? LST_NONCOLD : LST_MISS_E) * c->E;
      const int32_t* slot = c->lists_h + LST_MISS_SLOT * c->E;
      const uint8_t* host = back_h_of(c, layer);
      for (int i = 0; i < n; ++i) {
        uint8_t* dst = h.bypass ? c->scratch_d + (size_t)i * c->stride : pool + (size_t)slot[i] * c->stride;
        CK(c, cudaMemcpyAsync(dst, host + (size_t)src[i] * c->stride, c->Be, cudaMemcpyDefault,
                              c->copy_stream));
      }
      tm_end(c, TM_COPY, ti, c->copy_stream);
      CK(c, cudaEventRecord(c->ev_join, c->copy_stream));
    }
  }
  if (joined) CK(c, cudaStreamWaitEvent(s, c->ev_join, 0));
  if (mlp) {
    // one cooperative launch (up, grid barrier, down); up + down if it cannot fit
    int ti = tm_begin(c, TM_UP, s);
    int nl = 1;
    const cudaError_t fe = launch_layer_mlp(c, *mlp, s, &nl);
    if (fe == cudaSuccess) {
      c->launches += nl;
      tm_end(c, TM_UP, ti, s);
      tm_note_misses(c, ti, layer, s);
      return MOE_OK;
    }
    if (fe != cudaErrorNotSupported && fe != cudaErrorCooperativeLaunchTooLarge)
      return cuda_fail(c, fe, "fused expert MLP launch");
    cudaGetLastError();
    CK(c, launch_mlp_up(c->wd, *mlp, s));
    c->launches++;
    tm_end(c, TM_UP, ti, s);
    tm_note_misses(c, ti, layer, s);
    ti = tm_begin(c, TM_DOWN, s);
    CK(c, launch_mlp_down(c->wd, *mlp, s));
    c->launches++;
    tm_end(c, TM_DOWN, ti, s);
  }
  return MOE_OK;
}

moe_status measure_copy_modes(moe_cache* c) {
  // Time a pinned-host -> HBM copy both ways on the handle's own buffers.
  // (layer 0's pool or the scratch, from layer 0's backing store: contiguous in either table layout)
  size_t dev_bytes = (size_t)c->N * c->stride;
  uint8_t* dst = c->pool_d;
  if (dev_bytes < (size_t)c->scratch_n * c->stride) {
    dev_bytes = (size_t)c->scratch_n * c->stride;
    dst = c->scratch_d;
  }
  size_t bytes = std::min(std::min(dev_bytes, (size_t)c->E * c->stride), (size_t)256 << 20);
  bytes &= ~(size_t)15;
  if (bytes == 0) return MOE_OK;
  cudaStream_t s = c->copy_stream;
  cudaEvent_t a, b;
  CK(c, cudaEventCreate(&a));
  CK(c, cudaEventCreate(&b));
  float best_m = 1e30f, best_u = 1e30f, ms = 0;
  for (int rep = 0; rep < 3; ++rep) {
    CK(c, cudaEventRecord(a, s));
    CK(c, cudaMemcpyAsync(dst, c->backing_h, bytes, cudaMemcpyDefault, s));
    CK(c, cudaEventRecord(b, s));
    CK(c, cudaEventSynchronize(b));
    CK(c, cudaEventElapsedTime(&ms, a, b));
    best_m = std::min(best_m, ms);
    CK(c, cudaEventRecord(a, s));
    CK(c, launch_copy_raw(c->backing_dv, dst, bytes / 16, c->copy_grid, s));
    CK(c, cudaEventRecord(b, s));
    CK(c, cudaEventSynchronize(b));
    CK(c, cudaEventElapsedTime(&ms, a, b));
    best_u = std::min(best_u, ms);
  }
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  c->memcpy_gbs = bytes / (best_m * 1e-3) / 1e9;
  c->uva_gbs = bytes / (best_u * 1e-3) / 1e9;
  c->copy_mode = c->memcpy_gbs > 1.15 * c->uva_gbs ? MOE_COPY_MEMCPY : MOE_COPY_FUSED;
  return MOE_OK;
}

void free_all(moe_cache* c) {
  if (!c) return;
  cudaDeviceSynchronize();
  for (auto& p : c->tp) {
    for (auto e : p.beg) cudaEventDestroy(e);
    for (auto e : p.end) cudaEventDestroy(e);
  }
  for (cudaGraphExec_t g : c->step_graph)
    if (g) cudaGraphExecDestroy(g);
  if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
  if (c->ev_fork) cudaEventDestroy(c->ev_fork);
  if (c->ev_join) cudaEventDestroy(c->ev_join);
  if (c->ev_sync) cudaEventDestroy(c->ev_sync);
  if (c->copy_stream) cudaStreamDestroy(c->copy_stream);
  if (c->vmm.va) {
    vmm_table_destroy(&c->vmm);
    c->pool_d = nullptr;
    c->backing_h = nullptr;
  }
  void* dev[] = {c->pool_d, c->scratch_d, c->cold_d, c->fstack_d, c->counts_d, c->slot_map_d, c->slot_expert_d,
                 c->slot_stamp_d, c->slot_aux_d, c->state_d, c->hdr_d, c->lists_d, c->asg_d, c->pend_d, c->src_d, c->ids_d,
                 c->w_d, c->h_d, c->err_d, c->verify_d, c->bar_d, c->ring_cnt_d, c->tm_miss_d, c->tm_span_d, c->xs_d[0], c->xs_d[1],
                 c->logits_stage_d, c->order_d, c->tiles_d, c->ntiles_d, c->gout_d, c->seq_d, c->ready_d, c->xg_d};
  for (void* p : dev)
    if (p) cudaFree(p);
  moe_gemm_tma_maps_free(c->tma);
  if (c->backing_h) cudaFreeHost(c->backing_h);
  if (c->hdr_h) cudaFreeHost(c->hdr_h);
  if (c->lists_h) cudaFreeHost(c->lists_h);
  delete c;
}

moe_status init_state(moe_cache* c) {
  const size_t L = c->L, E = c->E, N = c->N;
  CK(c, cudaMemset(c->slot_map_d, 0xFF, L * E * sizeof(int32_t)));
  if (N) {
    CK(c, cudaMemset(c->slot_expert_d, 0xFF, L * N * sizeof(int32_t)));
    CK(c, cudaMemset(c->slot_stamp_d, 0, L * N * sizeof(long long)));
    CK(c, cudaMemset(c->slot_aux_d, 0, L * N * sizeof(int32_t)));
  }
  if (N) {
    std::vector<int32_t> fs(L * N);
    for (size_t l = 0; l < L; ++l)
      for (size_t i = 0; i < N; ++i) fs[l * N + i] = (int32_t)i;   // the first miss takes slot N - 1
    CK(c, cudaMemcpy(c->fstack_d, fs.data(), fs.size() * sizeof(int32_t), cudaMemcpyHostToDevice));
  }
  // the cold set given at create (run-time moves change it) and zero use counts
  CK(c, cudaMemcpy(c->cold_d, c->cold_h.data(), L * E, cudaMemcpyHostToDevice));
  if (c->counts_d) CK(c, cudaMemset(c->counts_d, 0, L * E * sizeof(float)));
  std::vector<LayerState> st(L);
  for (auto& s : st) {
    memset(&s, 0, sizeof(s));
    s.nfree = c->N;
  }
  CK(c, cudaMemcpy(c->state_d, st.data(), L * sizeof(LayerState), cudaMemcpyHostToDevice));
  CK(c, cudaMemset(c->hdr_d, 0, L * sizeof(RecHdr)));
  CK(c, cudaMemset(c->lists_d, 0, L * LST_COUNT * E * sizeof(int32_t)));
  CK(c, cudaMemset(c->err_d, 0, sizeof(int)));
  CK(c, cudaMemset(c->bar_d, 0, sizeof(GridBar)));
  return MOE_OK;
}

}  // namespace

moe_status moe::set_global_error(moe_status st, const char* msg) {
  g_create_error = msg ? msg : "";
  return st;
}

// ============================================================== C ABI

extern "C" {

const char* moe_cache_last_error(const moe_cache_t* c) {
  return c ? c->err.c_str() : g_create_error.c_str();
}

moe_status moe_cache_expert_bytes(int wdtype, int hidden, int inter, size_t* bytes) {
  size_t a, b, s1, s2;
  if (!bytes || hidden <= 0 || inter <= 0 || !block_layout(wdtype, hidden, inter, &a, &b, &s1, &s2))
    return fail(nullptr, MOE_EINVAL, "bad weight format or shape");
  *bytes = a + b + s1 + s2;
  return MOE_OK;
}

moe_status moe_cache_create(const moe_cache_config* cfg, moe_cache_t** out) {
  if (!out) return fail(nullptr, MOE_EINVAL, "out is NULL");
  *out = nullptr;
  if (!cfg) return fail(nullptr, MOE_EINVAL, "cfg is NULL");
  const moe_cache_config& g = *cfg;
  if (g.num_layers < 1 || g.num_experts < 1 || g.num_experts > MOE_MAX_EXPERTS)
    return fail(nullptr, MOE_EINVAL, "need num_layers >= 1 and 1 <= num_experts <= 1024");
  if (g.top_k < 1 || g.top_k > g.num_experts || g.top_k > MOE_MAX_TOPK)
    return fail(nullptr, MOE_EINVAL, "need 1 <= top_k <= min(num_experts, 32)");
  if (g.slots_per_layer < 0 || g.slots_per_layer > g.num_experts)
    return fail(nullptr, MOE_EINVAL, "need 0 <= slots_per_layer <= num_experts");
  if (g.max_tokens < 1 || (long long)g.max_tokens * g.top_k > 65535)
    return fail(nullptr, MOE_EINVAL, "need max_tokens >= 1 and max_tokens * top_k <= 65535");
  size_t w13, w2, s13, s2;
  if (g.hidden <= 0 || g.inter <= 0 || !block_layout(g.wdtype, g.hidden, g.inter, &w13, &w2, &s13, &s2))
    return fail(nullptr, MOE_EINVAL, "bad wdtype or shape (int4 needs hidden, inter multiples of 128; fp8 of 16)");
  if (g.hidden % chunk_elems(g.wdtype) || g.inter % chunk_elems(g.wdtype))
    return fail(nullptr, MOE_EINVAL, "hidden and inter must be multiples of 4 (f32), 8 (bf16) or 16 (fp8)");
  if (g.mlp_kernel != MOE_MLP_AUTO && g.mlp_kernel != MOE_MLP_PLAIN)
    return fail(nullptr, MOE_EINVAL, "mlp_kernel must be MOE_MLP_AUTO or MOE_MLP_PLAIN");
  if (g.copy_mode < MOE_COPY_AUTO || g.copy_mode > MOE_COPY_FUSED)
    return fail(nullptr, MOE_EINVAL, "bad copy_mode");
  if (g.renormalize != 0 && g.renormalize != 1) return fail(nullptr, MOE_EINVAL, "renormalize must be 0 or 1");
  if (g.table_layout != MOE_TABLE_SPLIT && g.table_layout != MOE_TABLE_VMM)
    return fail(nullptr, MOE_EINVAL, "table_layout must be MOE_TABLE_SPLIT or MOE_TABLE_VMM");
  if (g.gemm_kernel < 0 || g.gemm_kernel > MOE_GEMM_TMA)
    return fail(nullptr, MOE_EINVAL, "gemm_kernel must be 0, MOE_GEMM_TC or MOE_GEMM_TMA");
  if (g.evict_policy < MOE_EVICT_LRU || g.evict_policy > MOE_EVICT_SLRU)
    return fail(nullptr, MOE_EINVAL, "evict_policy must be MOE_EVICT_LRU, _LFU, _FIFO or _SLRU");
  if (g.move_interval < 0) return fail(nullptr, MOE_EINVAL, "move_interval must be >= 0");
  if (g.move_interval > 0 && (!(g.move_decay > 0.f && g.move_decay <= 1.f) || !(g.move_threshold >= 0.f) ||
                              !(g.move_threshold < 3.0e38f) || g.move_count_tokens < 1))
    return fail(nullptr, MOE_EINVAL, "moves need 0 < move_decay <= 1, finite move_threshold >= 0, move_count_tokens >= 1");
  if (mlp_up_smem_bytes(g.hidden) > 200 * 1024 || mlp_down_smem_bytes(g.top_k, g.inter) > 200 * 1024)
    return fail(nullptr, MOE_EINVAL, "hidden*4 and top_k*inter*4 must each fit in 200 KiB of shared memory");
  int ndev = 0;
  cudaError_t ce = cudaGetDeviceCount(&ndev);
  if (ce != cudaSuccess) return cuda_fail(nullptr, ce, "cudaGetDeviceCount");
  if (g.device < 0 || g.device >= ndev) return fail(nullptr, MOE_EINVAL, "device out of range");

  moe_cache* c = new moe_cache();
  c->cfg = g;
  c->cfg.cold_mask_h = nullptr;
  c->L = g.num_layers;
  c->E = g.num_experts;
  c->K = g.top_k;
  c->H = g.hidden;
  c->I = g.inter;
  c->N = g.slots_per_layer;
  c->maxT = g.max_tokens;
  c->step_graph.assign((size_t)c->maxT + 1, nullptr);
  c->step_graph_launches.assign((size_t)c->maxT + 1, 0ull);
  c->wd = g.wdtype;
  c->Be = w13 + w2 + s13 + s2;
  c->off_w2 = w13;
  c->off_s13 = w13 + w2;
  c->off_s2 = w13 + w2 + s13;
  c->stride = round_up(c->Be, 256);
  c->nvec = c->Be / 16;
  c->scratch_n = std::min(c->E, c->maxT * c->K);
  c->cold_h.assign((size_t)c->L * c->E, 0);
  if (g.cold_mask_h) {
    for (size_t i = 0; i < c->cold_h.size(); ++i) c->cold_h[i] = g.cold_mask_h[i] ? 1 : 0;
    c->any_cold = std::any_of(c->cold_h.begin(), c->cold_h.end(), [](uint8_t v) { return v != 0; });
  }

  auto bail = [&](moe_status st) {
    g_create_error = c->err;
    free_all(c);
    return st;
  };
#define CKC(call)                                                       \
  do {                                                                  \
    cudaError_t _e = (call);                                            \
    if (_e != cudaSuccess) return bail(cuda_fail(c, _e, #call));        \
  } while (0)

  CKC(cudaSetDevice(g.device));
  CKC(cudaFree(nullptr));
  const size_t pool_bytes = (size_t)c->L * c->N * c->stride;
  const size_t scratch_bytes = (size_t)c->scratch_n * c->stride;
  size_t free_b = 0, total_b = 0;
  CKC(cudaMemGetInfo(&free_b, &total_b));
  const size_t budget = g.hbm_budget_bytes ? g.hbm_budget_bytes : free_b / 2;
  if (pool_bytes + scratch_bytes > budget) {
    char msg[256];
    snprintf(msg, sizeof msg, "pools + scratch need %zu bytes, over the HBM budget of %zu bytes",
             pool_bytes + scratch_bytes, budget);
    fail(c, MOE_ENOMEM, msg);
    return bail(MOE_ENOMEM);
  }
  const size_t backing_bytes = (size_t)c->L * c->E * c->stride;
  auto dmalloc = [&](void** p, size_t n) { return cudaMalloc(p, n ? n : 16); };
  if (g.table_layout == MOE_TABLE_VMM) {
    int numa = -1;
    if (cudaDeviceGetAttribute(&numa, cudaDevAttrHostNumaId, g.device) != cudaSuccess) {
      cudaGetLastError();
      numa = 0;
    }
    std::string why;
    if (!vmm_table_create(g.device, numa, c->L, (size_t)c->N * c->stride, (size_t)c->E * c->stride, &c->vmm,
                          &why)) {
      fail(c, MOE_ECUDA, "one VMM table per layer: " + why);
      return bail(MOE_ECUDA);
    }
    c->pool_d = reinterpret_cast<uint8_t*>(c->vmm.va);
    c->backing_h = c->backing_dv = reinterpret_cast<uint8_t*>(c->vmm.va + c->vmm.pool_part);
    c->pool_pitch = c->back_pitch = c->vmm.pitch;
  } else {
    if (cudaHostAlloc((void**)&c->backing_h, backing_bytes, cudaHostAllocMapped | cudaHostAllocPortable) !=
        cudaSuccess) {
      cudaGetLastError();
      c->backing_h = nullptr;
      fail(c, MOE_ENOMEM, "cudaHostAlloc of the pinned backing store failed");
      return bail(MOE_ENOMEM);
    }
    CKC(cudaHostGetDevicePointer((void**)&c->backing_dv, c->backing_h, 0));
    c->pool_pitch = (size_t)c->N * c->stride;
    c->back_pitch = (size_t)c->E * c->stride;
  }
  c->scratch_bytes = scratch_bytes;
  if ((g.table_layout != MOE_TABLE_VMM && dmalloc((void**)&c->pool_d, pool_bytes) != cudaSuccess) ||
      dmalloc((void**)&c->scratch_d, scratch_bytes) != cudaSuccess) {
    cudaGetLastError();
    fail(c, MOE_ENOMEM, "cudaMalloc of the slot pools failed");
    return bail(MOE_ENOMEM);
  }
  const size_t L = c->L, E = c->E, N = c->N, TK = (size_t)c->maxT * c->K;
  CKC(dmalloc((void**)&c->cold_d, L * E));
  CKC(dmalloc((void**)&c->slot_map_d, L * E * sizeof(int32_t)));
  CKC(dmalloc((void**)&c->slot_expert_d, L * N * sizeof(int32_t)));
  CKC(dmalloc((void**)&c->slot_stamp_d, L * N * sizeof(long long)));
  CKC(dmalloc((void**)&c->slot_aux_d, L * N * sizeof(int32_t)));
  CKC(dmalloc((void**)&c->fstack_d, (L * N > 0 ? L * N : 1) * sizeof(int32_t)));
  if (g.move_interval > 0) CKC(dmalloc((void**)&c->counts_d, L * E * sizeof(float)));
  CKC(dmalloc((void**)&c->state_d, L * sizeof(LayerState)));
  CKC(dmalloc((void**)&c->hdr_d, L * sizeof(RecHdr)));
  CKC(dmalloc((void**)&c->lists_d, L * LST_COUNT * E * sizeof(int32_t)));
  CKC(dmalloc((void**)&c->asg_d, TK * sizeof(unsigned long long)));
  CKC(dmalloc((void**)&c->pend_d, TK));
  CKC(dmalloc((void**)&c->src_d, TK * sizeof(unsigned long long)));
  CKC(dmalloc((void**)&c->ids_d, TK * sizeof(int32_t)));
  CKC(dmalloc((void**)&c->w_d, TK * sizeof(float)));
  // h: [T*k, I] f32 (per-token kernels), the staged kernel's copies, or (TMA
  // GEMM) at least 128 rows of bf16 so that every activation box lies inside it
  size_t h_floats = TK * c->I > mlp_ring_h_floats(c->K, c->I) ? TK * c->I : mlp_ring_h_floats(c->K, c->I);
  if (h_floats < (size_t)64 * c->I) h_floats = (size_t)64 * c->I;
  CKC(dmalloc((void**)&c->h_d, h_floats * sizeof(float)));
  CKC(dmalloc((void**)&c->err_d, sizeof(int)));
  CKC(dmalloc((void**)&c->bar_d, sizeof(GridBar)));
  CKC(dmalloc((void**)&c->ring_cnt_d, 3 * MOE_MAX_TOPK * sizeof(unsigned)));
  CKC(cudaMemset(c->ring_cnt_d, 0, 3 * MOE_MAX_TOPK * sizeof(unsigned)));
  CKC(dmalloc((void**)&c->seq_d, sizeof(unsigned)));
  CKC(dmalloc((void**)&c->ready_d, (size_t)E * sizeof(unsigned)));
  // zeroed once: the prepare counter never goes back (not even on reset), so
  // a ready flag left by an earlier step can never match a later step
  CKC(cudaMemset(c->seq_d, 0, sizeof(unsigned)));
  CKC(cudaMemset(c->ready_d, 0, (size_t)E * sizeof(unsigned)));
  CKC(dmalloc((void**)&c->verify_d, sizeof(int)));
  CKC(dmalloc((void**)&c->xs_d[0], (size_t)c->maxT * c->H * act_bytes(c->wd)));
  CKC(dmalloc((void**)&c->xs_d[1], (size_t)c->maxT * c->H * act_bytes(c->wd)));
  CKC(dmalloc((void**)&c->logits_stage_d, L * c->maxT * E * sizeof(float)));
  CKC(cudaHostAlloc((void**)&c->hdr_h, sizeof(RecHdr), cudaHostAllocDefault));
  CKC(cudaHostAlloc((void**)&c->lists_h, LST_COUNT * E * sizeof(int32_t), cudaHostAllocDefault));
  CKC(cudaMemcpy(c->cold_d, c->cold_h.data(), L * E, cudaMemcpyHostToDevice));
  if (init_state(c) != MOE_OK) return bail(MOE_ECUDA);
  CKC(cudaStreamCreateWithFlags(&c->copy_stream, cudaStreamNonBlocking));
  CKC(cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming));
  CKC(cudaEventCreateWithFlags(&c->ev_join, cudaEventDisableTiming));
  CKC(cudaEventCreateWithFlags(&c->ev_sync, cudaEventDisableTiming));
  CKC(prepare_configure());
  CKC(mlp_configure(c->wd, c->H, c->I, c->K));
  c->staged_mlp = g.mlp_kernel != MOE_MLP_PLAIN;
  if (c->staged_mlp) CKC(mlp_ring_configure(c->wd, c->H, c->I, c->K));
  if (c->staged_mlp && c->maxT > 1 && moe_gemm_supported(c->wd, c->H, c->I, c->K)) {
    CKC(dmalloc((void**)&c->order_d, TK * sizeof(int32_t)));
    CKC(dmalloc((void**)&c->tiles_d, TK * sizeof(int4)));
    CKC(dmalloc((void**)&c->ntiles_d, 4 * sizeof(int)));   // tile count + two item counters
    CKC(dmalloc((void**)&c->gout_d, TK * c->H * sizeof(float)));
    CKC(moe_gemm_configure(c->wd));
    c->gemm_mlp = true;
    if (g.gemm_kernel != MOE_GEMM_TC && moe_gemm_tma_supported(c->wd, c->H, c->I, c->K)) {
      // the TMA GEMM: activation rows gathered in tile order, tensor maps over
      // the pool (device rows of every layer), the scratch and the h rows
      const size_t rows = TK > 128 ? TK : 128;   // every activation box (<= 128 rows) inside the buffers
      CKC(dmalloc((void**)&c->xg_d, rows * c->H * 2));
      CKC(cudaMemset(c->xg_d, 0, rows * c->H * 2));
      c->tma = moe_gemm_tma_maps(c->wd, c->H, c->I, c->pool_d, (size_t)c->L * c->pool_pitch, c->scratch_d,
                                 c->scratch_bytes, c->xg_d, c->h_d, rows);
      if (!moe_gemm_tma_maps_ok(c->tma) || moe_gemm_tma_configure(c->wd) != cudaSuccess) {
        cudaGetLastError();
        moe_gemm_tma_maps_free(c->tma);
        c->tma = nullptr;
      }
    }
  }
  int sms = 0;
  CKC(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, g.device));
  c->copy_grid = std::max(1, sms) * 4;
  c->flag_grid = std::max(1, std::min(64, sms / 2));
  c->copy_mode = g.copy_mode;
  if (g.copy_mode == MOE_COPY_AUTO) {
    if (measure_copy_modes(c) != MOE_OK) return bail(MOE_ECUDA);
  }
  CKC(cudaDeviceSynchronize());
#undef CKC
  *out = c;
  return MOE_OK;
}

void moe_cache_destroy(moe_cache_t* c) {
  if (!c) return;
  cudaSetDevice(c->cfg.device);
  free_all(c);
}

moe_status moe_cache_get_info(moe_cache_t* c, moe_cache_info* out) {
  if (!c || !out) return fail(c, MOE_EINVAL, "null argument");
  out->expert_bytes = c->Be;
  out->slot_stride = c->stride;
  out->pool_bytes = (size_t)c->L * c->N * c->stride;
  out->scratch_bytes = (size_t)c->scratch_n * c->stride;
  out->backing_bytes = (size_t)c->L * c->E * c->stride;
  out->copy_mode = c->copy_mode;
  out->memcpy_gbs = c->memcpy_gbs;
  out->uva_gbs = c->uva_gbs;
  out->kernel_launches = c->launches;
  out->scratch_experts = c->scratch_n;
  out->table_layout = c->cfg.table_layout;
  out->gemm_kernel = !c->gemm_mlp ? MOE_GEMM_NONE : (c->tma != nullptr ? MOE_GEMM_TMA : MOE_GEMM_TC);
  return MOE_OK;
}

moe_status moe_cache_backing_ptr(moe_cache_t* c, int layer, int expert, void** block_h,
                                 size_t* stride_bytes) {
  moe_status st = check_layer(c, layer);
  if (st != MOE_OK) return st;
  if (expert < 0 || expert >= c->E || !block_h) return fail(c, MOE_EINVAL, "expert out of range or null out");
  *block_h = back_h_of(c, layer) + (size_t)expert * c->stride;
  if (stride_bytes) *stride_bytes = c->stride;
  return MOE_OK;
}

moe_status moe_cache_load_expert(moe_cache_t* c, int layer, int expert, const void* block_h,
                                 size_t bytes) {
  moe_status st = check_layer(c, layer);
  if (st != MOE_OK) return st;
  if (expert < 0 || expert >= c->E || !block_h || bytes != c->Be)
    return fail(c, MOE_EINVAL, "expert out of range, null block or wrong byte count");
  CK(c, cudaSetDevice(c->cfg.device));
  CK(c, cudaDeviceSynchronize());
  uint8_t* dst = back_h_of(c, layer) + (size_t)expert * c->stride;
  memcpy(dst, block_h, bytes);
  int32_t s = -1;
  CK(c, cudaMemcpy(&s, c->slot_map_d + (size_t)layer * c->E + expert, sizeof s, cudaMemcpyDeviceToHost));
  if (s >= 0)
    CK(c, cudaMemcpy(pool_of(c, layer) + (size_t)s * c->stride, dst, bytes, cudaMemcpyDefault));
  return MOE_OK;
}

moe_status moe_cache_router(moe_cache_t* c, const float* logits_d, int T, int32_t* ids_d,
                            float* w_d, moe_stream_t stream) {
  if (!c) return fail(nullptr, MOE_EINVAL, "null handle");
  if (T < 0 || T > c->maxT) return fail(c, MOE_EINVAL, "T out of range [0, max_tokens]");
  if (T == 0) return MOE_OK;
  if (!logits_d || !ids_d || !w_d) return fail(c, MOE_EINVAL, "null buffer");
  CK(c, cudaSetDevice(c->cfg.device));
  CK(c, launch_router(logits_d, T, c->E, c->K, c->cfg.renormalize, ids_d, w_d, (cudaStream_t)stream));
  c->launches++;
  return MOE_OK;
}

moe_status moe_cache_prepare(moe_cache_t* c, int layer, const int32_t* ids_d, int T,
                             int32_t* slot_ids_d, moe_stream_t stream) {
  moe_status st = check_layer(c, layer);
  if (st != MOE_OK) return st;
  if (T < 0 || T > c->maxT) return fail(c, MOE_EINVAL, "T out of range [0, max_tokens]");
  if (T == 0) return MOE_OK;
  if (!ids_d) return fail(c, MOE_EINVAL, "null ids");
  CK(c, cudaSetDevice(c->cfg.device));
  cudaStream_t s = (cudaStream_t)stream;
  st = run_prepare(c, layer, nullptr, ids_d, T, slot_ids_d, s);
  if (st != MOE_OK) return st;
  return run_copies_and_mlp(c, layer, s, nullptr);
}

moe_status moe_cache_last_prepare(moe_cache_t* c, int layer, moe_prepare_info* out) {
  moe_status st = check_layer(c, layer);
  if (st != MOE_OK) return st;
  if (!out) return fail(c, MOE_EINVAL, "null out");
  CK(c, cudaSetDevice(c->cfg.device));
  CK(c, cudaDeviceSynchronize());
  RecHdr h;
  CK(c, cudaMemcpy(&h, c->hdr_d + layer, sizeof h, cudaMemcpyDeviceToHost));
  std::vector<int32_t> lists((size_t)LST_COUNT * c->E);
  CK(c, cudaMemcpy(lists.data(), c->lists_d + (size_t)layer * LST_COUNT * c->E,
                   lists.size() * sizeof(int32_t), cudaMemcpyDeviceToHost));
  out->n_ids = h.n_ids;
  out->bypass = h.bypass;
  out->n_distinct = h.n_distinct;
  out->n_cold = h.n_cold;
  out->n_noncold = h.n_noncold;
  out->n_hits = h.n_hits;
  out->n_misses = h.n_misses;
  out->n_evictions = h.n_evictions;
  auto put = [&](int32_t* dst, int lst, int n) {
    if (dst && n > 0) memcpy(dst, lists.data() + (size_t)lst * c->E, sizeof(int32_t) * n);
  };
  put(out->hits_h, LST_HITS, h.n_hits);
  put(out->miss_expert_h, LST_MISS_E, h.n_misses);
  put(out->miss_slot_h, LST_MISS_SLOT, h.n_misses);
  put(out->miss_evicted_h, LST_MISS_EV, h.n_misses);
  put(out->cold_h, LST_COLD, h.n_cold);
  put(out->noncold_h, LST_NONCOLD, h.n_noncold);
  return device_error(c);
}

moe_status moe_forward(moe_cache_t* c, int layer, const void* x_d, const float* logits_d, int T,
                       void* y_d, int flags, moe_stream_t stream) {
  moe_status st = check_layer(c, layer);
  if (st != MOE_OK) return st;
  if (T < 0 || T > c->maxT) return fail(c, MOE_EINVAL, "T out of range [0, max_tokens]");
  if (T == 0) return MOE_OK;
  if (!x_d || !logits_d || !y_d) return fail(c, MOE_EINVAL, "null buffer");
  if (x_d == y_d) return fail(c, MOE_EINVAL, "x and y may not alias");
  if (flags & ~MOE_FWD_RESIDUAL) return fail(c, MOE_EINVAL, "unknown flags");
  CK(c, cudaSetDevice(c->cfg.device));
  cudaStream_t s = (cudaStream_t)stream;
  st = run_prepare(c, layer, logits_d, nullptr, T, nullptr, s);
  if (st != MOE_OK) return st;
  MlpArgs a = mlp_args(c->wd, c->H, c->I, c->K, x_d, c->asg_d, c->w_d, c->h_d, y_d, T, flags);
  // this layer's host rows (in the VMM layout they sit between two layers' pools)
  a.host_lo = (unsigned long long)back_d_of(c, layer);
  a.host_hi = a.host_lo + (unsigned long long)c->E * c->stride;
  a.h_cnt = c->ring_cnt_d + 2 * MOE_MAX_TOPK;   // zeroed by this step's prepare
  return run_copies_and_mlp(c, layer, s, &a);
}

moe_status moe_expert_mlp(int wdtype, int hidden, int inter, int top_k, const void* x_d,
                          const uint64_t* block_ptrs_d, const float* w_d, int T,
                          float* h_scratch_d, void* y_d, int flags, moe_stream_t stream) {
  size_t a1, a2, a3, a4;
  if (!block_layout(wdtype, hidden, inter, &a1, &a2, &a3, &a4) || hidden % chunk_elems(wdtype) ||
      inter % chunk_elems(wdtype))
    return fail(nullptr, MOE_EINVAL, "bad weight format or shape");
  if (top_k < 1 || top_k > MOE_MAX_TOPK || T < 0 || (long long)T * top_k > 65535)
    return fail(nullptr, MOE_EINVAL, "bad top_k or T");
  if (mlp_up_smem_bytes(hidden) > 200 * 1024 || mlp_down_smem_bytes(top_k, inter) > 200 * 1024)
    return fail(nullptr, MOE_EINVAL, "shape exceeds shared-memory staging limits");
  if (flags & ~MOE_FWD_RESIDUAL) return fail(nullptr, MOE_EINVAL, "unknown flags");
  if (T == 0) return MOE_OK;
  if (!x_d || !block_ptrs_d || !w_d || !h_scratch_d || !y_d || x_d == y_d)
    return fail(nullptr, MOE_EINVAL, "null or aliased buffer");
  cudaStream_t s = (cudaStream_t)stream;
  if (!capturing(s)) {
    const cudaError_t ce = mlp_configure(wdtype, hidden, inter, top_k);
    if (ce != cudaSuccess) return cuda_fail(nullptr, ce, "mlp_configure");
  }
  const MlpArgs a = mlp_args(wdtype, hidden, inter, top_k, x_d,
                             reinterpret_cast<const unsigned long long*>(block_ptrs_d), w_d,
                             h_scratch_d, y_d, T, flags);
  cudaError_t e = launch_mlp_up(wdtype, a, s);
  if (e == cudaSuccess) e = launch_mlp_down(wdtype, a, s);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "moe_expert_mlp launch");
  return MOE_OK;
}

namespace {

// Every layer of a T-token step, from xs_d[0] and logits_stage_d; the result
// lands in xs_d[L & 1].
moe_status run_layers(moe_cache* c, int T, moe_stream_t stream) {
  int cur = 0;
  for (int l = 0; l < c->L; ++l) {
    moe_status st = moe_forward(c, l, c->xs_d[cur], c->logits_stage_d + (size_t)l * T * c->E, T,
                                c->xs_d[cur ^ 1], MOE_FWD_RESIDUAL, stream);
    if (st != MOE_OK) return st;
    cur ^= 1;
  }
  return MOE_OK;
}

moe_status capture_step_graph(moe_cache* c, int T) {
  if (!c->cap_stream) CK(c, cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking));
  const unsigned long long l0 = c->launches;
  CK(c, cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal));
  const moe_status st = run_layers(c, T, (moe_stream_t)c->cap_stream);
  cudaGraph_t g = nullptr;
  const cudaError_t ce = cudaStreamEndCapture(c->cap_stream, &g);
  c->step_graph_launches[T] = c->launches - l0;
  c->launches = l0;
  if (st != MOE_OK) {
    if (g) cudaGraphDestroy(g);
    return st;
  }
  if (ce != cudaSuccess) return cuda_fail(c, ce, "capturing the model step");
  const cudaError_t ie = cudaGraphInstantiate(&c->step_graph[T], g, 0);
  cudaGraphDestroy(g);
  if (ie != cudaSuccess) {
    c->step_graph[T] = nullptr;
    return cuda_fail(c, ie, "instantiating the model step graph");
  }
  return MOE_OK;
}

}  // namespace

moe_status moe_model_step_host(moe_cache_t* c, const void* x_h, const float* logits_h, int T,
                               void* y_h, int timeout_ms, moe_stream_t stream) {
  if (!c) return fail(nullptr, MOE_EINVAL, "null handle");
  if (T < 0 || T > c->maxT) return fail(c, MOE_EINVAL, "T out of range [0, max_tokens]");
  if (T == 0) return MOE_OK;
  if (!x_h || !logits_h || !y_h) return fail(c, MOE_EINVAL, "null buffer");
  CK(c, cudaSetDevice(c->cfg.device));
  cudaStream_t s = (cudaStream_t)stream;
  const size_t xb = (size_t)T * c->H * act_bytes(c->wd);
  CK(c, cudaMemcpyAsync(c->xs_d[0], x_h, xb, cudaMemcpyHostToDevice, s));
  CK(c, cudaMemcpyAsync(c->logits_stage_d, logits_h, (size_t)c->L * T * c->E * sizeof(float),
                        cudaMemcpyHostToDevice, s));
  // the layers run from the staged x / logits: replayed from a graph captured
  // at the first call with this T (MEMCPY mode takes a host decision per
  // layer and per-launch timing records host-side events, so both run eagerly)
  const int cur = c->L & 1;
  if (c->copy_mode != MOE_COPY_MEMCPY && !c->timing_on) {
    if (!c->step_graph[T]) {
      moe_status st = capture_step_graph(c, T);
      if (st != MOE_OK) return st;
    }
    CK(c, cudaGraphLaunch(c->step_graph[T], s));
    c->launches += c->step_graph_launches[T];
  } else {
    moe_status st = run_layers(c, T, (moe_stream_t)s);
    if (st != MOE_OK) return st;
  }
  CK(c, cudaMemcpyAsync(y_h, c->xs_d[cur], xb, cudaMemcpyDeviceToHost, s));
  CK(c, cudaEventRecord(c->ev_sync, s));
  return wait_event_bounded(c, c->ev_sync, timeout_ms > 0 ? timeout_ms : 60000);
}

moe_status moe_cache_stats(moe_cache_t* c, int layer, moe_cache_counters* out) {
  if (!c || !out) return fail(c, MOE_EINVAL, "null argument");
  if (layer < -1 || layer >= c->L) return fail(c, MOE_EINVAL, "layer out of range");
  CK(c, cudaSetDevice(c->cfg.device));
  CK(c, cudaDeviceSynchronize());
  std::vector<LayerState> st(c->L);
  CK(c, cudaMemcpy(st.data(), c->state_d, st.size() * sizeof(LayerState), cudaMemcpyDeviceToHost));
  unsigned long long acc[ST_COUNT] = {0};
  for (int l = 0; l < c->L; ++l)
    if (layer == -1 || layer == l)
      for (int i = 0; i < ST_COUNT; ++i) acc[i] += st[l].stats[i];
  out->steps = acc[ST_STEPS];
  out->hits = acc[ST_HITS];
  out->misses = acc[ST_MISSES];
  out->evictions = acc[ST_EVICT];
  out->bypass_steps = acc[ST_BYPASS];
  out->cold_reads = acc[ST_COLD];
  out->bytes_h2d_miss = acc[ST_B_MISS];
  out->bytes_h2d_bypass = acc[ST_B_BYPASS];
  out->bytes_uva_cold = acc[ST_B_COLD];
  out->moves = acc[ST_MOVES];
  return device_error(c);
}

moe_status moe_cache_get_state(moe_cache_t* c, int layer, int32_t* slot_map_h, int32_t* slot_expert_h,
                               int64_t* slot_stamp_h, int32_t* n_free_h) {
  moe_status st = check_layer(c, layer);
  if (st != MOE_OK) return st;
  CK(c, cudaSetDevice(c->cfg.device));
  CK(c, cudaDeviceSynchronize());
  if (slot_map_h)
    CK(c, cudaMemcpy(slot_map_h, c->slot_map_d + (size_t)layer * c->E, c->E * sizeof(int32_t),
                     cudaMemcpyDeviceToHost));
  if (slot_expert_h && c->N)
    CK(c, cudaMemcpy(slot_expert_h, c->slot_expert_d + (size_t)layer * c->N, c->N * sizeof(int32_t),
                     cudaMemcpyDeviceToHost));
  if (slot_stamp_h && c->N)
    CK(c, cudaMemcpy(slot_stamp_h, c->slot_stamp_d + (size_t)layer * c->N, c->N * sizeof(int64_t),
                     cudaMemcpyDeviceToHost));
  if (n_free_h) {
    LayerState ls;
    CK(c, cudaMemcpy(&ls, c->state_d + layer, sizeof ls, cudaMemcpyDeviceToHost));
    *n_free_h = ls.nfree;
  }
  return device_error(c);
}

moe_status moe_cache_verify_slots(moe_cache_t* c, int layer, int* mismatched_slots) {
  moe_status st = check_layer(c, layer);
  if (st != MOE_OK) return st;
  if (!mismatched_slots) return fail(c, MOE_EINVAL, "null out");
  CK(c, cudaSetDevice(c->cfg.device));
  CK(c, cudaDeviceSynchronize());
  CK(c, cudaMemset(c->verify_d, 0, sizeof(int)));
  CK(c, launch_verify(c->slot_expert_d + (size_t)layer * c->N, c->N,
                      pool_of(c, layer), back_d_of(c, layer), c->stride, c->nvec,
                      c->verify_d, 0));
  c->launches++;
  CK(c, cudaDeviceSynchronize());
  CK(c, cudaMemcpy(mismatched_slots, c->verify_d, sizeof(int), cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status moe_cache_get_cold(moe_cache_t* c, int layer, uint8_t* cold_h) {
  moe_status st = check_layer(c, layer);
  if (st != MOE_OK) return st;
  if (!cold_h) return fail(c, MOE_EINVAL, "null buffer");
  CK(c, cudaSetDevice(c->cfg.device));
  CK(c, cudaDeviceSynchronize());
  CK(c, cudaMemcpy(cold_h, c->cold_d + (size_t)layer * c->E, c->E, cudaMemcpyDeviceToHost));
  return device_error(c);
}

moe_status moe_cache_pool_ptrs(moe_cache_t* c, int layer, void** pool_d, void** scratch_d) {
  moe_status st = check_layer(c, layer);
  if (st != MOE_OK) return st;
  if (pool_d) *pool_d = pool_of(c, layer);
  if (scratch_d) *scratch_d = c->scratch_d;
  return MOE_OK;
}

moe_status moe_cache_check(moe_cache_t* c) {
  if (!c) return fail(nullptr, MOE_EINVAL, "null handle");
  CK(c, cudaSetDevice(c->cfg.device));
  CK(c, cudaDeviceSynchronize());
  return device_error(c);
}

moe_status moe_cache_reset(moe_cache_t* c) {
  if (!c) return fail(nullptr, MOE_EINVAL, "null handle");
  CK(c, cudaSetDevice(c->cfg.device));
  CK(c, cudaDeviceSynchronize());
  moe_status st = init_state(c);
  if (st != MOE_OK) return st;
  CK(c, cudaDeviceSynchronize());
  return MOE_OK;
}

moe_status moe_cache_set_timing(moe_cache_t* c, int on, int capacity) {
  if (!c) return fail(nullptr, MOE_EINVAL, "null handle");
  if (capacity < 0 || capacity > (1 << 22)) return fail(c, MOE_EINVAL, "timing capacity out of range");
  CK(c, cudaSetDevice(c->cfg.device));
  const size_t cap = capacity ? (size_t)capacity : (size_t)kDefaultTimingCap;
  for (auto& p : c->tp) {
    p.used = 0;
    if (on) {
      while (p.beg.size() < cap) {
        cudaEvent_t a, b;
        CK(c, cudaEventCreate(&a));
        CK(c, cudaEventCreate(&b));
        p.beg.push_back(a);
        p.end.push_back(b);
      }
    }
  }
  if (on && c->tm_miss_cap < cap) {
    if (c->tm_miss_d) CK(c, cudaFree(c->tm_miss_d));
    if (c->tm_span_d) CK(c, cudaFree(c->tm_span_d));
    c->tm_miss_d = nullptr;
    c->tm_span_d = nullptr;
    c->tm_miss_cap = 0;
    CK(c, cudaMalloc((void**)&c->tm_miss_d, cap * sizeof(int32_t)));
    CK(c, cudaMalloc((void**)&c->tm_span_d, (size_t)kSpanRecWords * cap * sizeof(unsigned long long)));
    c->tm_miss_cap = cap;
  }
  if (on) CK(c, cudaMemset(c->tm_span_d, 0, (size_t)kSpanRecWords * c->tm_miss_cap * sizeof(unsigned long long)));
  c->timing_on = on != 0;
  return MOE_OK;
}

moe_status moe_cache_read_timing_launches(moe_cache_t* c, float* ms_h, int32_t* misses_h, int cap,
                                          int* n) {
  if (!c || !n || cap < 0) return fail(c, MOE_EINVAL, "null argument");
  CK(c, cudaSetDevice(c->cfg.device));
  CK(c, cudaDeviceSynchronize());
  const TimingPool& p = c->tp[TM_UP];
  const int avail = (int)p.used;
  const int m = avail < cap ? avail : cap;
  std::vector<int32_t> mi(m > 0 ? m : 1, 0);
  const int mc = m < (int)c->tm_miss_cap ? m : (int)c->tm_miss_cap;
  if (mc > 0 && c->tm_miss_d)
    CK(c, cudaMemcpy(mi.data(), c->tm_miss_d, (size_t)mc * sizeof(int32_t), cudaMemcpyDeviceToHost));
  for (int i = 0; i < m; ++i) {
    float v = -1.f;
    if (cudaEventElapsedTime(&v, p.beg[i], p.end[i]) != cudaSuccess) {
      cudaGetLastError();
      v = -1.f;
    }
    if (ms_h) ms_h[i] = v;
    if (misses_h) misses_h[i] = mi[i];
  }
  *n = m;
  return MOE_OK;
}

moe_status moe_cache_read_copy_spans(moe_cache_t* c, uint64_t* rec_h, int cap, int* n) {
  if (!c || !n || cap < 0 || (cap > 0 && !rec_h)) return fail(c, MOE_EINVAL, "null argument");
  CK(c, cudaSetDevice(c->cfg.device));
  CK(c, cudaDeviceSynchronize());
  const int avail = (int)c->tp[TM_UP].used;
  int m = avail < cap ? avail : cap;
  if (m > (int)c->tm_miss_cap) m = (int)c->tm_miss_cap;
  if (m <= 0 || c->tm_span_d == nullptr) {
    *n = 0;
    return MOE_OK;
  }
  std::vector<unsigned long long> raw((size_t)m * kSpanRecWords);
  CK(c, cudaMemcpy(raw.data(), c->tm_span_d, raw.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost));
  for (int i = 0; i < m; ++i) {
    const unsigned long long* r = raw.data() + (size_t)i * kSpanRecWords;
    const unsigned long long grid = r[1] <= (unsigned long long)kSpanMaxCtas ? r[1] : 0ull;
    unsigned long long first = ~0ull, last = 0ull;
    for (unsigned long long b = 0; b < grid; ++b) {
      if (r[2 + 2 * b] != 0ull && r[2 + 2 * b] < first) first = r[2 + 2 * b];
      if (r[3 + 2 * b] > last) last = r[3 + 2 * b];
    }
    rec_h[3 * (size_t)i] = first;
    rec_h[3 * (size_t)i + 1] = last;
    rec_h[3 * (size_t)i + 2] = grid ? r[0] : 0ull;
  }
  *n = m;
  return MOE_OK;
}

moe_status moe_cache_read_timing(moe_cache_t* c, moe_cache_timing* out) {
  if (!c || !out) return fail(c, MOE_EINVAL, "null argument");
  CK(c, cudaSetDevice(c->cfg.device));
  CK(c, cudaDeviceSynchronize());
  double ms[TM_COUNT] = {0};
  uint64_t n[TM_COUNT] = {0};
  for (int k = 0; k < TM_COUNT; ++k) {
    TimingPool& p = c->tp[k];
    for (size_t i = 0; i < p.used; ++i) {
      float v = 0;
      if (cudaEventElapsedTime(&v, p.beg[i], p.end[i]) == cudaSuccess) {
        ms[k] += v;
        n[k]++;
      } else {
        cudaGetLastError();
      }
    }
  }
  out->route_ms = ms[TM_ROUTE];
  out->copy_ms = ms[TM_COPY];
  out->up_ms = ms[TM_UP];
  out->down_ms = ms[TM_DOWN];
  out->route_n = n[TM_ROUTE];
  out->copy_n = n[TM_COPY];
  out->up_n = n[TM_UP];
  out->down_n = n[TM_DOWN];
  return MOE_OK;
}

}  // extern "C"
