// C ABI of the fused MoE-FFN layer: argument checks, workspace carve-up, kernel sequence.
//
// Forward (RFC "HyperParallel Multicore HyperMegaMoE fused forward/backward operator", §2.1):
//   status clear -> route count -> route scan -> route rank -> gather x rows ->
//   [shared expert GEMM1 + GEMM2] -> GEMM1 + SwiGLU -> GEMM2 -> weighted combine into y
//   (GEMM1 and GEMM2 in one launch with MM_FLAG_FUSED_FORWARD_GEMMS; the combine inside GEMM2
//   with MM_FLAG_FUSED_COMBINE).
// Backward (§2.2): gather dy rows -> act_grad + SwiGLU backward -> d_topk_weights ->
//   W2Grad (-> sum of split experts' partial slices) -> input_grad ->
//   [shared expert act_grad, W2Grad, input_grad] ->
//   combine dx (side stream) || W1Grad (-> sum of partial slices) -> [shared expert W1Grad].
// The host never waits on the device here (except the optional id pre-check); the caller's
// stream orders everything (the side stream is forked from it and joined back within the
// call). The two-phase size query / execute split mirrors §2.3.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "mm_kernels.h"
#include "mm_layout.h"

namespace mm {

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // bounded device waits: 2 s
constexpr uint64_t kTestTimeoutNs = 50000000ull;       // with MM_FLAG_TEST_STALL: 50 ms

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool dims_ok(const mm_dims& d) {
  if (d.T < 0 || d.H < 8 || d.I < 8 || d.E < 1 || d.K < 1) return false;
  if (d.H % 8 || d.I % 8) return false;
  if (d.E > 1024 || d.K > 16) return false;
  if (d.T > (int64_t)1 << 31 || d.H > ((int64_t)1 << 20) || d.I > ((int64_t)1 << 20)) return false;
  const int64_t S = d.T * d.K;
  if (S + d.E * (BM - 1) + BM >= ((int64_t)1 << 31)) return false;
  return true;
}

// ---- optional per-stage timer (process-global, not thread-safe)
struct TimerRecord {
  int stage;
  cudaEvent_t start, stop;
};
struct Timer {
  bool on = false;
  uint32_t mask = 0xFFFFFFFFu;  // stages that are bracketed while on
  std::vector<TimerRecord> pending;
  std::vector<cudaEvent_t> pool;
  cudaEvent_t get() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
  }
};
Timer g_timer;

// ---- optional trace (process-global, not thread-safe): the caller's buffer and the sequence
// number of the next traced launch
struct TraceState {
  uint32_t* buf = nullptr;
  uint32_t cap = 0;
  uint32_t next_launch = 0;
};
TraceState g_trace;
// the trace context of the launch this thread is enqueueing (read by the launchers)
thread_local TraceCtx t_trace_cur = {nullptr, 0, 0, 0};

template <typename F>
cudaError_t timed_launch(int stage, cudaStream_t st, F&& launch) {
  if (!g_timer.on || !((g_timer.mask >> stage) & 1u)) return launch();
  cudaEvent_t a = g_timer.get(), b = g_timer.get();
  if (a) cudaEventRecord(a, st);
  cudaError_t e = launch();
  if (b) cudaEventRecord(b, st);
  if (a && b)
    g_timer.pending.push_back({stage, a, b});
  else {
    if (a) g_timer.pool.push_back(a);
    if (b) g_timer.pool.push_back(b);
  }
  return e;
}

// Every launch of a forward or backward goes through here: the stage timer's events, and the
// trace context the launcher passes to its kernel.
template <typename F>
cudaError_t timed(int stage, cudaStream_t st, F&& launch) {
  if (g_trace.buf != nullptr)
    t_trace_cur = {g_trace.buf, g_trace.cap, (uint32_t)stage, g_trace.next_launch++};
  const cudaError_t e = timed_launch(stage, st, launch);
  t_trace_cur = {nullptr, 0, 0, 0};
  return e;
}

const char* kStageNames[ST_COUNT] = {
    "route_count", "route_scan",  "route_rank", "gather_x",   "gemm1_swiglu",
    "gemm2",       "combine_y",   "gather_dy",  "act_grad",   "d_topk",
    "w2_grad",     "input_grad",  "combine_dx", "w1_grad",    "shared_expert",
    "gemm1_gemm2", "wgrad_reduce"};

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Text of the last CUDA failure seen by a call of this thread (see mm_last_error_detail).
thread_local char g_err[256] = "";

mm_status cuda_fail(cudaError_t e, const char* what) {
  // the previous detail (a note from a lower layer) is kept after this one, shortened to fit
  char inner[160];
  memcpy(inner, g_err, sizeof(inner) - 1);
  inner[sizeof(inner) - 1] = 0;
  snprintf(g_err, sizeof(g_err), "%.80s: %.60s (%.40s)%s%.60s", what, cudaGetErrorString(e),
           cudaGetErrorName(e), inner[0] ? "; " : "", inner);
  return MM_ERR_CUDA;
}

#define MM_TRY(expr)                                    \
  do {                                                  \
    cudaError_t _e = (expr);                            \
    if (_e != cudaSuccess) return cuda_fail(_e, #expr); \
  } while (0)

// A second stream per device and host thread, for work that may overlap the caller's stream
// inside one call, with the two events that fork it from and join it back to the caller's
// stream. Created once per device and thread (non-blocking, highest priority, so its small grids
// are scheduled ahead of a persistent GEMM's CTAs as soon as an SM has room). One per thread, so
// that calls from two host threads can never interleave their records of, and waits on, the same
// events; a thread's own calls are sequential.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

cudaError_t side_stream(SideStream** out) {
  thread_local SideStream per_dev[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  SideStream& ss = per_dev[dev];
  if (ss.s == nullptr) {
    int lo = 0, hi = 0;
    if ((e = cudaDeviceGetStreamPriorityRange(&lo, &hi)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithPriority(&ss.s, cudaStreamNonBlocking, hi)) != cudaSuccess)
      return e;
  }
  *out = &ss;
  return cudaSuccess;
}

// Makes the current device's primary context current on this thread. Tensor-map encoding is a
// driver call that needs one, and a thread that has not launched anything yet (an autograd
// worker thread, say) may not have it bound.
cudaError_t bind_context() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return cudaSetDevice(dev);
}

}  // namespace

TraceCtx trace_ctx() { return t_trace_cur; }
static_assert(sizeof(mm_trace_record) == 32 && offsetof(mm_trace_record, unit) == 8 &&
                  offsetof(mm_trace_record, launch) == 12 && offsetof(mm_trace_record, t0) == 16,
              "trace record layout (written by trace_end as two 16-byte words)");

void note_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

bool plan_workspace(const mm_dims& d, Workspace* w, bool direct_rows) {
  if (!dims_ok(d)) return false;
  Workspace p{};
  p.T = d.T;
  p.H = d.H;
  p.I = d.I;
  p.E = d.E;
  p.K = d.K;
  p.S = d.T * d.K;
  const int64_t nonempty = std::min<int64_t>(d.E, p.S);
  p.S_pad = (p.S + nonempty * (BM - 1) + BM - 1) / BM * BM;
  p.n_chunks = (p.S + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
  p.n_act_tiles = 2 * ((d.I + BN - 1) / BN);  // two column halves per act_grad tile
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  p.off_hdr = take(HDR_WORDS * sizeof(int32_t));
  p.off_counts = take(d.E * sizeof(int32_t));
  p.off_offsets = take((d.E + 1) * sizeof(int32_t));
  p.off_poff = take((d.E + 1) * sizeof(int32_t));
  p.off_chunk = take((size_t)p.n_chunks * d.E * sizeof(int32_t));
  p.off_tile_expert = take((size_t)(p.S_pad / BM) * sizeof(int32_t));
  p.off_ready = take((size_t)(p.S_pad / BM) * sizeof(int32_t));
  p.off_cnt = take((size_t)d.T * ((d.H + 127) / 128) * sizeof(int32_t));
  p.off_pair_tile = take((size_t)(p.S_pad / BM) * sizeof(int32_t));
  p.off_row_of_slot = take((size_t)p.S * sizeof(int32_t));
  p.off_slot_of_row = take((size_t)p.S_pad * sizeof(int32_t));
  p.off_w_row = take((size_t)p.S_pad * sizeof(float));
  p.off_x_slot = take(direct_rows ? 0 : (size_t)p.S_pad * d.H * 2);
  p.off_gu = take((size_t)p.S_pad * 2 * d.I * 4);
  p.off_h = take((size_t)p.S_pad * d.I * 2);
  p.off_hw_lo = take((size_t)p.S_pad * d.I * 2);
  p.off_o = take((size_t)p.S_pad * d.H * 2);
  p.off_dy_slot = take(direct_rows ? 0 : (size_t)p.S_pad * d.H * 2);
  p.off_dgu = take((size_t)p.S_pad * 2 * d.I * 2);
  p.off_dgu_lo = take((size_t)p.S_pad * 2 * d.I * 2);
  p.off_p_part = take((size_t)p.n_act_tiles * p.S_pad * sizeof(float));
  p.off_o_lo = take(direct_rows ? (size_t)p.S_pad * d.H * 2 : 0);
  if (!direct_rows) {  // the partial slices reuse the o / dx and dy row buffers
    p.wg_slices[WG_W2] = std::min<int64_t>(1024, (p.S_pad * d.H * 2) / (d.I * d.H * 4));
    p.wg_slices[WG_W1] = std::min<int64_t>(1024, (p.S_pad * d.H * 2) / (2 * d.I * d.H * 4));
  }
  p.wg_slices_max = std::max(p.wg_slices[WG_W2], p.wg_slices[WG_W1]);
  p.off_wg_plan = take((size_t)2 * (d.E + p.wg_slices_max) * 16);
  p.off_wg_red = take((size_t)2 * d.E * 16);
  p.total = off;
  *w = p;
  return true;
}

}  // namespace mm

using namespace mm;

extern "C" {

int mm_abi_version(void) { return 3; }

const char* mm_last_error_detail(void) { return g_err; }

const char* mm_status_string(mm_status s) {
  switch (s) {
    case MM_OK: return "ok";
    case MM_ERR_INVALID_ARG: return "invalid argument";
    case MM_ERR_UNSUPPORTED: return "unsupported sizes";
    case MM_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MM_ERR_CUDA: return "CUDA runtime error";
    case MM_ERR_BAD_EXPERT_ID: return "expert id out of range";
    case MM_ERR_TIMEOUT: return "device-side wait timed out";
    case MM_ERR_TOKENS_PER_EXPERT: return "tokens_per_expert does not match topk_ids";
  }
  return "unknown status";
}

size_t mm_workspace_size(mm_dims d, uint32_t flags) {
  (void)flags;
  Workspace w;
  if (!plan_workspace(d, &w)) return 0;
  return w.total;
}

// The main layout, and with a shared expert its sub-workspace (sizes T, H, I_s, E = 1, K = 1,
// no dispatched-row buffers) placed after it.
struct Plan {
  Workspace w;
  bool shared = false;
  Workspace ws_s;
  size_t base_s = 0;
  size_t total = 0;
};

static bool plan_all(const mm_dims& d, int64_t shared_I, Plan* p) {
  if (!plan_workspace(d, &p->w)) return false;
  p->total = p->w.total;
  p->shared = shared_I > 0;
  if (!p->shared) return true;
  const mm_dims ds{d.T, d.H, shared_I, 1, 1};
  if (!plan_workspace(ds, &p->ws_s, true)) return false;
  p->base_s = align_up(p->w.total, 256);
  p->total = p->base_s + p->ws_s.total;
  return true;
}

static mm_status check_common(const mm_dims& d, const mm_shared_expert* se, const void* ws,
                              size_t ws_bytes, Plan* p) {
  if (d.T < 0 || d.H < 1 || d.I < 1 || d.E < 1 || d.K < 1) return MM_ERR_INVALID_ARG;
  if (se != nullptr && se->I < 1) return MM_ERR_INVALID_ARG;
  if (!plan_all(d, se ? se->I : 0, p)) return MM_ERR_UNSUPPORTED;
  if (ws == nullptr || !aligned(ws, 256) || ws_bytes < p->total) return MM_ERR_WORKSPACE;
  return MM_OK;
}

// CTA-pair form of the row-grouped GEMMs: 0 one CTA per tile, 2 (default) pairs sharing one
// M = 256 MMA.
static int pair_mode(uint32_t flags) { return (flags & MM_FLAG_SINGLE_CTA_TILES) ? 0 : 2; }

// GEMM1 -> GEMM2 as one counter-released launch: when asked for, or, unless the caller asked for
// two launches, where it measured faster (include/mm.h, MM_FLAG_FUSED_FORWARD_GEMMS): CTA-pair
// launches of 1 to 16 waves, estimated as ceil(S / 256) row-tile pairs x (ceil(I / 128) GEMM1 +
// ceil(H / 256) GEMM2 column tiles) over the SM pairs. Measured on a GB300 (H = 2048, I = 768,
// 1024 rows per expert): forward 4-7 % faster at 8k and 16k slots (3 and 12 waves), 1-3 % slower
// from 32k slots (24 waves) up; skew and tail workloads 4 and 3 % faster steps.
static bool fused_forward(const Workspace& w, uint32_t flags) {
  if (flags & MM_FLAG_FUSED_FORWARD_GEMMS) return true;
  if (flags & (MM_FLAG_SEPARATE_FORWARD_GEMMS | MM_FLAG_SINGLE_CTA_TILES | MM_FLAG_FUSED_COMBINE |
               MM_FLAG_TEST_STALL))
    return false;
  const int64_t pairs = std::max(1, device_sm_count() / 2);
  const int64_t units = (w.S + 255) / 256 * ((w.I + 127) / 128 + (w.H + 255) / 256);
  return units >= pairs && units <= 16 * pairs;
}

// An empty batch (T = 0): no slot to route or compute. The header and the routing tables are
// written as empty (zero counts and offsets), and a caller's tokens_per_expert is still compared
// with them by the scan kernel, which reads no chunk histogram when there is none.
static mm_status forward_empty(const Plan& p, const mm_shared_expert* se, const int32_t* tpe,
                               const void* up_proj_weight, const void* down_proj_weight,
                               void* workspace, void* stream, uint32_t flags) {
  const Workspace& w = p.w;
  if (!up_proj_weight || !down_proj_weight || !aligned(up_proj_weight, 16) ||
      !aligned(down_proj_weight, 16))
    return MM_ERR_INVALID_ARG;
  if (se && (!se->up_proj_weight || !se->down_proj_weight || !aligned(se->up_proj_weight, 16) ||
             !aligned(se->down_proj_weight, 16)))
    return MM_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = reinterpret_cast<char*>(workspace);
  g_err[0] = 0;
  MM_TRY(bind_context());
  MM_TRY(cudaMemsetAsync(ws + w.off_hdr, 0, HDR_WORDS * sizeof(int32_t), st));
  if (flags & MM_FLAG_FORWARD_ONLY)
    MM_TRY(cudaMemsetAsync(ws + w.off_hdr + HDR_NO_BACKWARD * sizeof(int32_t), 1,
                           sizeof(int32_t), st));
  MM_TRY(timed(ST_ROUTE_SCAN, st, [&] { return launch_route_scan(w, ws, tpe, st); }));
  if (flags & MM_FLAG_VALIDATE_IDS) {
    int32_t status = 0;
    MM_TRY(cudaMemcpyAsync(&status, ws + w.off_hdr, sizeof(status), cudaMemcpyDeviceToHost, st));
    MM_TRY(cudaStreamSynchronize(st));
    if (status != 0) return static_cast<mm_status>(status);
  }
  return MM_OK;
}

// The backward of an empty batch: every weight gradient is zero (written as zeros, or left as it
// is when accumulating); dx and d_topk_weights have no element. A workspace whose forward was
// forward-only is refused through the status word, as for T > 0.
static mm_status backward_empty(const Plan& p, const mm_shared_expert* se,
                                const void* up_proj_weight, const void* down_proj_weight,
                                void* d_up_proj_weight, void* d_down_proj_weight, void* workspace,
                                void* stream, uint32_t flags) {
  const Workspace& w = p.w;
  if (!up_proj_weight || !down_proj_weight || !d_up_proj_weight || !d_down_proj_weight ||
      !aligned(up_proj_weight, 16) || !aligned(down_proj_weight, 16) ||
      !aligned(d_up_proj_weight, 16) || !aligned(d_down_proj_weight, 16))
    return MM_ERR_INVALID_ARG;
  if (se && (!se->up_proj_weight || !se->down_proj_weight || !se->d_up_proj_weight ||
             !se->d_down_proj_weight || !aligned(se->up_proj_weight, 16) ||
             !aligned(se->down_proj_weight, 16) || !aligned(se->d_up_proj_weight, 16) ||
             !aligned(se->d_down_proj_weight, 16)))
    return MM_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  g_err[0] = 0;
  MM_TRY(bind_context());
  MM_TRY(launch_backward_check(w, reinterpret_cast<char*>(workspace), st));
  if (flags & MM_FLAG_ACCUMULATE_WEIGHT_GRADS) return MM_OK;  // adding zero changes nothing
  const size_t es = (flags & MM_FLAG_FP32_WEIGHT_GRADS) ? 4 : 2;
  const size_t n_up = (size_t)w.E * w.H * 2 * w.I, n_down = (size_t)w.E * w.I * w.H;
  MM_TRY(cudaMemsetAsync(d_up_proj_weight, 0, n_up * es, st));
  MM_TRY(cudaMemsetAsync(d_down_proj_weight, 0, n_down * es, st));
  if (se) {
    MM_TRY(cudaMemsetAsync(se->d_up_proj_weight, 0, (size_t)w.H * 2 * se->I * es, st));
    MM_TRY(cudaMemsetAsync(se->d_down_proj_weight, 0, (size_t)se->I * w.H * es, st));
  }
  return MM_OK;
}

static mm_status forward_impl(mm_dims d, const mm_shared_expert* se, const int32_t* tpe,
                              const void* x,
                              const int32_t* topk_ids, const float* topk_weights,
                              const void* up_proj_weight, const void* down_proj_weight, void* y,
                              void* workspace, size_t workspace_bytes, void* stream,
                              uint32_t flags) {
  Plan p;
  mm_status s = check_common(d, se, workspace, workspace_bytes, &p);
  if (s != MM_OK) return s;
  const Workspace& w = p.w;
  if ((flags & MM_FLAG_FUSED_FORWARD_GEMMS) && (flags & MM_FLAG_SEPARATE_FORWARD_GEMMS))
    return MM_ERR_INVALID_ARG;
  if (d.T == 0) return forward_empty(p, se, tpe, up_proj_weight, down_proj_weight, workspace,
                                     stream, flags);
  if (!x || !topk_ids || !topk_weights || !up_proj_weight || !down_proj_weight || !y)
    return MM_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(up_proj_weight, 16) || !aligned(down_proj_weight, 16) ||
      !aligned(y, 16) || !aligned(topk_ids, 4) || !aligned(topk_weights, 4))
    return MM_ERR_INVALID_ARG;
  if (se && (!se->up_proj_weight || !se->down_proj_weight || !aligned(se->up_proj_weight, 16) ||
             !aligned(se->down_proj_weight, 16)))
    return MM_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = reinterpret_cast<char*>(workspace);
  g_err[0] = 0;
  MM_TRY(bind_context());

  MM_TRY(cudaMemsetAsync(ws + w.off_hdr, 0, HDR_WORDS * sizeof(int32_t), st));
  MM_TRY(timed(ST_ROUTE_COUNT, st, [&] { return launch_route_count(w, ws, topk_ids, st); }));
  MM_TRY(timed(ST_ROUTE_SCAN, st, [&] { return launch_route_scan(w, ws, tpe, st); }));
  if (flags & MM_FLAG_VALIDATE_IDS) {
    int32_t status = 0;
    MM_TRY(cudaMemcpyAsync(&status, ws + w.off_hdr, sizeof(status), cudaMemcpyDeviceToHost, st));
    MM_TRY(cudaStreamSynchronize(st));
    if (status != 0) return static_cast<mm_status>(status);
  }
  MM_TRY(timed(ST_ROUTE_RANK, st,
               [&] { return launch_route_rank(w, ws, topk_ids, topk_weights, st); }));
  MM_TRY(timed(ST_GATHER_X, st,
               [&] { return launch_gather_rows(w, ws, x, ws + w.off_x_slot, st); }));
  const bool stall = (flags & MM_FLAG_TEST_STALL) != 0;
  GemmCall c{GK_GEMM1_SWIGLU, up_proj_weight, down_proj_weight, nullptr,
             stall ? kTestTimeoutNs : kDefaultTimeoutNs, stall ? 1 : 0, 0, nullptr, nullptr};
  c.paired = pair_mode(flags);
  if (flags & MM_FLAG_FORWARD_ONLY) {  // no gate|up kept; a backward from here is refused
    c.skip_gu = 1;
    MM_TRY(cudaMemsetAsync(ws + w.off_hdr + HDR_NO_BACKWARD * sizeof(int32_t), 1,
                           sizeof(int32_t), st));
  }
  // the shared expert first: its output rows must exist before a combine reads them
  const void* extra = nullptr;
  const void* extra_lo = nullptr;
  if (p.shared) {  // the shared expert: identity routing over all tokens, weight 1
    char* wss = ws + p.base_s;
    GemmCall cs{GK_GEMM1_SWIGLU, se->up_proj_weight, se->down_proj_weight, nullptr,
                c.timeout_ns, 0, 0, x, reinterpret_cast<int*>(ws + w.off_hdr) + HDR_STATUS,
                1};  // its output is added with weight 1: kept as a bf16 hi + lo pair
    cs.skip_gu = c.skip_gu;
    cs.paired = c.paired;  // row tiles of its T rows pair like an expert's
    MM_TRY(timed(ST_SHARED, st, [&] { return launch_shared_tables(p.ws_s, wss, st); }));
    MM_TRY(timed(ST_SHARED, st, [&] { return launch_gemm(p.ws_s, wss, cs, st); }));
    cs.kind = GK_GEMM2;
    MM_TRY(timed(ST_SHARED, st, [&] { return launch_gemm(p.ws_s, wss, cs, st); }));
    extra = wss + p.ws_s.off_o;
    extra_lo = wss + p.ws_s.off_o_lo;
  }
  const bool fuse_combine = (flags & MM_FLAG_FUSED_COMBINE) != 0;
  if (fuse_combine) {  // GEMM2's epilogue sums y; its per-(token, chunk) counters start at zero
    MM_TRY(cudaMemsetAsync(ws + w.off_cnt, 0,
                           (size_t)w.T * ((w.H + 127) / 128) * sizeof(int32_t), st));
    c.comb_y = y;
    c.comb_w = nullptr;  // GEMM2's rows already carry the routing weight
    c.comb_extra = extra;
    c.comb_extra_lo = extra_lo;
  }
  if (fused_forward(w, flags)) {
    // one launch: GEMM2 row blocks start as soon as their GEMM1 tiles are stored (the routing
    // scan zeroed the ready counters of the row tiles in use)
    c.kind = GK_FWD_FUSED;
    MM_TRY(timed(ST_FWD_GEMMS, st, [&] { return launch_gemm(w, ws, c, st); }));
    c.inject_stall = 0;
  } else {
    MM_TRY(timed(ST_GEMM1_SWIGLU, st, [&] { return launch_gemm(w, ws, c, st); }));
    c.kind = fuse_combine ? GK_GEMM2_COMBINE : GK_GEMM2;
    c.inject_stall = 0;
    MM_TRY(timed(ST_GEMM2, st, [&] { return launch_gemm(w, ws, c, st); }));
  }
  if (!fuse_combine)
    MM_TRY(timed(ST_COMBINE_Y, st, [&] {
      // GEMM2's rows already carry the routing weight (GEMM1 wrote w*h): an unweighted sum
      return launch_combine(w, ws, ws + w.off_o, nullptr, y, st, extra, extra_lo, true);
    }));
  return MM_OK;
}

static mm_status backward_impl(mm_dims d, const mm_shared_expert* se, const void* dy,
                               const void* x, const int32_t* topk_ids, const float* topk_weights,
                               const void* up_proj_weight, const void* down_proj_weight,
                               void* workspace, size_t workspace_bytes, void* dx,
                               float* d_topk_weights, void* d_up_proj_weight,
                               void* d_down_proj_weight, void* stream, uint32_t flags) {
  Plan p;
  mm_status s = check_common(d, se, workspace, workspace_bytes, &p);
  if (s != MM_OK) return s;
  const Workspace& w = p.w;
  if (d.T == 0)
    return backward_empty(p, se, up_proj_weight, down_proj_weight, d_up_proj_weight,
                          d_down_proj_weight, workspace, stream, flags);
  if (!dy || !x || !topk_ids || !topk_weights || !up_proj_weight || !down_proj_weight || !dx ||
      !d_topk_weights || !d_up_proj_weight || !d_down_proj_weight)
    return MM_ERR_INVALID_ARG;
  if (!aligned(dy, 16) || !aligned(x, 16) || !aligned(up_proj_weight, 16) ||
      !aligned(down_proj_weight, 16) || !aligned(dx, 16) || !aligned(d_up_proj_weight, 16) ||
      !aligned(d_down_proj_weight, 16) || !aligned(d_topk_weights, 4) || !aligned(topk_ids, 4) ||
      !aligned(topk_weights, 4))
    return MM_ERR_INVALID_ARG;
  if (se && (!se->up_proj_weight || !se->down_proj_weight || !se->d_up_proj_weight ||
             !se->d_down_proj_weight || !aligned(se->up_proj_weight, 16) ||
             !aligned(se->down_proj_weight, 16) || !aligned(se->d_up_proj_weight, 16) ||
             !aligned(se->d_down_proj_weight, 16)))
    return MM_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = reinterpret_cast<char*>(workspace);
  g_err[0] = 0;
  MM_TRY(bind_context());

  MM_TRY(timed(ST_GATHER_DY, st,
               [&] { return launch_gather_rows(w, ws, dy, ws + w.off_dy_slot, st); }));
  GemmCall c{GK_ACT_GRAD, up_proj_weight, down_proj_weight, nullptr, kDefaultTimeoutNs, 0, 0,
             nullptr, nullptr};
  const int accumulate = (flags & MM_FLAG_ACCUMULATE_WEIGHT_GRADS) ? 1 : 0;
  c.wgrad_f32 = (flags & MM_FLAG_FP32_WEIGHT_GRADS) ? 1 : 0;
  // CTA pairs: input_grad in either form; the weight gradients as pair MMAs only, and only when
  // the experts average 256 rows or more (below that the pair's lockstep over reductions of a
  // few 64-row blocks costs more than its halved operand traffic saves: measured on a GB300 at
  // 187 rows per expert, 2 % slower; at 256, 8-11 % faster)
  const int pair = pair_mode(flags);
  const int wgrad_pair = (pair == 2 && w.S >= 256 * w.E) ? 2 : 0;
  c.paired = pair == 2 ? 2 : 0;  // act_grad: pair MMAs or one CTA per tile
  MM_TRY(timed(ST_ACT_GRAD, st, [&] { return launch_gemm(w, ws, c, st); }));
  c.kind = GK_W2_GRAD;
  c.d_w = d_down_proj_weight;
  c.accumulate = accumulate;
  c.paired = wgrad_pair;
  // d_topk_weights: in W2Grad's launch (its epilogue warps, before their first tile), or, if
  // that grid is too small for the slots, a kernel of its own after it
  bool d_topk_taken = false;
  c.d_topk = d_topk_weights;
  c.d_topk_taken = &d_topk_taken;
  MM_TRY(timed(ST_W2_GRAD, st, [&] { return launch_gemm(w, ws, c, st); }));
  c.d_topk = nullptr;
  c.d_topk_taken = nullptr;
  if (!d_topk_taken)
    MM_TRY(timed(ST_D_TOPK, st, [&] { return launch_d_topk(w, ws, d_topk_weights, st); }));
  // split experts' W2Grad partial slices (in the o / dx row buffer) summed into the output
  // before input_grad writes its dx rows there
  if (wgrad_split_possible(w, WG_W2))
    MM_TRY(timed(ST_WGRAD_REDUCE, st, [&] {
      return launch_wgrad_reduce(w, ws, WG_W2, d_down_proj_weight, c.wgrad_f32 != 0,
                                 accumulate != 0, st);
    }));
  c.kind = GK_INPUT_GRAD;
  c.d_w = nullptr;
  c.accumulate = 0;
  c.paired = pair;
  MM_TRY(timed(ST_INPUT_GRAD, st, [&] { return launch_gemm(w, ws, c, st); }));
  c.paired = 0;
  const void* extra = nullptr;
  const void* extra_lo = nullptr;
  char* wss = ws + p.base_s;
  GemmCall cs{GK_ACT_GRAD, nullptr, nullptr, nullptr, kDefaultTimeoutNs, 0, 0, dy,
              reinterpret_cast<int*>(ws + w.off_hdr) + HDR_STATUS, 1, c.wgrad_f32};
  // the shared expert is one expert of T rows: the same pair rules
  const int shared_wgrad_pair = (pair == 2 && w.T >= 256) ? 2 : 0;
  if (p.shared) {  // shared expert: act_grad, W2Grad (rows = dy), input_grad
    cs.w_up = se->up_proj_weight;
    cs.w_down = se->down_proj_weight;
    MM_TRY(timed(ST_SHARED, st, [&] { return launch_gemm(p.ws_s, wss, cs, st); }));
    cs.kind = GK_W2_GRAD;
    cs.d_w = se->d_down_proj_weight;
    cs.accumulate = accumulate;
    cs.paired = shared_wgrad_pair;
    MM_TRY(timed(ST_SHARED, st, [&] { return launch_gemm(p.ws_s, wss, cs, st); }));
    cs.kind = GK_INPUT_GRAD;
    cs.d_w = nullptr;
    cs.accumulate = 0;
    cs.paired = pair;
    cs.rows = nullptr;
    MM_TRY(timed(ST_SHARED, st, [&] { return launch_gemm(p.ws_s, wss, cs, st); }));
    extra = wss + p.ws_s.off_o;
    extra_lo = wss + p.ws_s.off_o_lo;
  }
  // Combine(dX) is HBM-bound and independent of W1Grad (tensor-bound): it runs on the side
  // stream, forked after input_grad and joined back after W1Grad has been enqueued.
  SideStream* side = nullptr;
  MM_TRY(side_stream(&side));
  MM_TRY(cudaEventRecord(side->fork, st));
  MM_TRY(cudaStreamWaitEvent(side->s, side->fork, 0));
  const cudaError_t e_comb = timed(ST_COMBINE_DX, side->s, [&] {
    return launch_combine(w, ws, ws + w.off_o, nullptr, dx, side->s, extra, extra_lo);
  });
  c.kind = GK_W1_GRAD;
  c.d_w = d_up_proj_weight;
  c.accumulate = accumulate;
  c.paired = wgrad_pair;
  cudaError_t e_w1 = timed(ST_W1_GRAD, st, [&] { return launch_gemm(w, ws, c, st); });
  if (e_w1 == cudaSuccess && wgrad_split_possible(w, WG_W1))  // split experts' partial slices
    e_w1 = timed(ST_WGRAD_REDUCE, st, [&] {
      return launch_wgrad_reduce(w, ws, WG_W1, d_up_proj_weight, c.wgrad_f32 != 0,
                                 accumulate != 0, st);
    });
  MM_TRY(cudaEventRecord(side->join, side->s));  // the join is enqueued whatever happened above
  MM_TRY(cudaStreamWaitEvent(st, side->join, 0));
  MM_TRY(e_comb);
  MM_TRY(e_w1);
  if (p.shared) {  // shared expert W1Grad (rows = x)
    cs.kind = GK_W1_GRAD;
    cs.d_w = se->d_up_proj_weight;
    cs.accumulate = accumulate;
    cs.rows = x;
    cs.paired = shared_wgrad_pair;
    MM_TRY(timed(ST_SHARED, st, [&] { return launch_gemm(p.ws_s, wss, cs, st); }));
  }
  return MM_OK;
}

mm_status mm_forward(mm_dims d, const void* x, const int32_t* topk_ids, const float* topk_weights,
                     const void* up_proj_weight, const void* down_proj_weight, void* y,
                     void* workspace, size_t workspace_bytes, void* stream, uint32_t flags) {
  return forward_impl(d, nullptr, nullptr, x, topk_ids, topk_weights, up_proj_weight,
                      down_proj_weight, y, workspace, workspace_bytes, stream, flags);
}

mm_status mm_backward(mm_dims d, const void* dy, const void* x, const int32_t* topk_ids,
                      const float* topk_weights, const void* up_proj_weight,
                      const void* down_proj_weight, void* workspace, size_t workspace_bytes,
                      void* dx, float* d_topk_weights, void* d_up_proj_weight,
                      void* d_down_proj_weight, void* stream, uint32_t flags) {
  return backward_impl(d, nullptr, dy, x, topk_ids, topk_weights, up_proj_weight,
                       down_proj_weight, workspace, workspace_bytes, dx, d_topk_weights,
                       d_up_proj_weight, d_down_proj_weight, stream, flags);
}

size_t mm_workspace_size_ex(mm_dims d, const mm_options* opt, uint32_t flags) {
  (void)flags;
  const mm_shared_expert* se = opt ? opt->shared : nullptr;
  if (se != nullptr && se->I < 1) return 0;
  Plan p;
  if (!plan_all(d, se ? se->I : 0, &p)) return 0;
  return p.total;
}

mm_status mm_forward_ex(mm_dims d, const mm_options* opt, const void* x,
                        const int32_t* topk_ids, const float* topk_weights,
                        const void* up_proj_weight, const void* down_proj_weight, void* y,
                        void* workspace, size_t workspace_bytes, void* stream, uint32_t flags) {
  if (opt && opt->tokens_per_expert && !aligned(opt->tokens_per_expert, 4))
    return MM_ERR_INVALID_ARG;
  return forward_impl(d, opt ? opt->shared : nullptr, opt ? opt->tokens_per_expert : nullptr, x,
                      topk_ids, topk_weights, up_proj_weight, down_proj_weight, y, workspace,
                      workspace_bytes, stream, flags);
}

mm_status mm_backward_ex(mm_dims d, const mm_options* opt, const void* dy, const void* x,
                         const int32_t* topk_ids, const float* topk_weights,
                         const void* up_proj_weight, const void* down_proj_weight,
                         void* workspace, size_t workspace_bytes, void* dx,
                         float* d_topk_weights, void* d_up_proj_weight, void* d_down_proj_weight,
                         void* stream, uint32_t flags) {
  return backward_impl(d, opt ? opt->shared : nullptr, dy, x, topk_ids, topk_weights,
                       up_proj_weight, down_proj_weight, workspace, workspace_bytes, dx,
                       d_topk_weights, d_up_proj_weight, d_down_proj_weight, stream, flags);
}

mm_status mm_get_status(const void* workspace, void* stream) {
  if (workspace == nullptr || !aligned(workspace, 256)) return MM_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MM_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MM_ERR_CUDA;
  return static_cast<mm_status>(v);
}

mm_status mm_routing_export(mm_dims d, const void* workspace, int32_t* counts, int32_t* offsets,
                            int32_t* row_of_slot, void* stream) {
  Workspace w;
  if (!plan_workspace(d, &w)) return MM_ERR_UNSUPPORTED;
  if (workspace == nullptr || !aligned(workspace, 256)) return MM_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const char* ws = reinterpret_cast<const char*>(workspace);
  if (counts)
    MM_TRY(cudaMemcpyAsync(counts, ws + w.off_counts, w.E * sizeof(int32_t), cudaMemcpyDefault, st));
  if (offsets)
    MM_TRY(cudaMemcpyAsync(offsets, ws + w.off_offsets, (w.E + 1) * sizeof(int32_t),
                           cudaMemcpyDefault, st));
  if (row_of_slot && w.S > 0) {
    // converted into the backward-only p_part scratch, then copied out
    int32_t* tmp = reinterpret_cast<int32_t*>(const_cast<char*>(ws) + w.off_p_part);
    MM_TRY(launch_export_rows(w, ws, tmp, st));
    MM_TRY(cudaMemcpyAsync(row_of_slot, tmp, w.S * sizeof(int32_t), cudaMemcpyDefault, st));
  }
  MM_TRY(cudaStreamSynchronize(st));
  return MM_OK;
}

mm_status mm_timing_enable(int on) {
  g_timer.on = on != 0;
  return MM_OK;
}

mm_status mm_timing_select(uint32_t stage_mask) {
  g_timer.mask = stage_mask;
  return MM_OK;
}

int mm_timing_read(double* ms, int64_t* launches, int max_stages) {
  double acc[ST_COUNT] = {0};
  int64_t cnt[ST_COUNT] = {0};
  for (auto& r : g_timer.pending) {
    float t = 0.f;
    if (cudaEventSynchronize(r.stop) == cudaSuccess &&
        cudaEventElapsedTime(&t, r.start, r.stop) == cudaSuccess) {
      acc[r.stage] += t;
      cnt[r.stage] += 1;
    }
    g_timer.pool.push_back(r.start);
    g_timer.pool.push_back(r.stop);
  }
  g_timer.pending.clear();
  for (int i = 0; i < ST_COUNT && i < max_stages; ++i) {
    if (ms) ms[i] = acc[i];
    if (launches) launches[i] = cnt[i];
  }
  return ST_COUNT;
}

const char* mm_stage_name(int stage) {
  if (stage < 0 || stage >= ST_COUNT) return "";
  return kStageNames[stage];
}

mm_status mm_trace_set(void* device_buffer, size_t bytes) {
  if (device_buffer == nullptr) {
    g_trace = TraceState();
    return MM_OK;
  }
  if (!aligned(device_buffer, 32) || bytes < 64) return MM_ERR_INVALID_ARG;
  const size_t cap = bytes / 32 - 1;
  g_trace.buf = reinterpret_cast<uint32_t*>(device_buffer);
  g_trace.cap = cap > 0xFFFFFFFFull ? 0xFFFFFFFFu : (uint32_t)cap;
  g_trace.next_launch = 0;
  return MM_OK;
}

}  // extern "C"
