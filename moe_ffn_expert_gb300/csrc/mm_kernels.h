// Host launchers of the library's kernels (each enqueues exactly one kernel on `stream`).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mm_layout.h"

namespace mm {

// Launches `kernel` on `st` with programmatic stream serialization (see pdl_wait in
// mm_device.cuh): the launch may overlap the end of the stream's previous kernel.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---- routing, dispatch and combine (mm_route.cu)
cudaError_t launch_route_count(const Workspace& w, char* ws, const int32_t* ids, cudaStream_t st);
// tokens_per_expert (optional, device int32 [E]): compared with the computed counts; a
// mismatch records MM_ERR_TOKENS_PER_EXPERT in the status word.
cudaError_t launch_route_scan(const Workspace& w, char* ws, const int32_t* tokens_per_expert,
                              cudaStream_t st);
cudaError_t launch_route_rank(const Workspace& w, char* ws, const int32_t* ids, const float* topk_w,
                              cudaStream_t st);
// dst[r] = src[slot_of_row[r] / K] for every real row, zeros for pad rows.
cudaError_t launch_gather_rows(const Workspace& w, char* ws, const void* src, void* dst,
                               cudaStream_t st);
// out[t] = sum_k (weights ? weights[t,k] : 1) * rows[row_of_slot[t*K+k]], k ascending, fp32,
// plus extra[t] (weight 1) when extra is not null.
cudaError_t launch_combine(const Workspace& w, char* ws, const void* rows, const float* weights,
                           void* out, cudaStream_t st, const void* extra = nullptr,
                           const void* extra_lo = nullptr, bool row_table = false);
// Identity routing tables of the shared expert's sub-workspace (ws points at its base).
cudaError_t launch_shared_tables(const Workspace& ws_shared, char* ws, cudaStream_t st);
// d_topk[s] = sum over column tiles (ascending) of p_part[tile][row_of_slot[s]]. Launched only
// when the W2Grad launch, which normally computes these in its epilogue warps, has too few CTAs
// for the slots.
cudaError_t launch_d_topk(const Workspace& w, char* ws, float* d_topk, cudaStream_t st);
// Records MM_ERR_INVALID_ARG in the status word if the forward kept no gate|up (forward only):
// the check of a backward that launches no GEMM (T = 0).
cudaError_t launch_backward_check(const Workspace& w, char* ws, cudaStream_t st);
// Converts the padded row_of_slot table to positions in the unpadded expert-sorted order.
cudaError_t launch_export_rows(const Workspace& w, const char* ws, int32_t* out, cudaStream_t st);

// ---- grouped GEMMs on tcgen05 (mm_gemm.cu)
enum GemmKind {
  GK_GEMM1_SWIGLU = 0,  // gu = x_slot W_up[e]; h = silu(gate) * up
  GK_GEMM2 = 1,         // o = h W_down[e]
  GK_ACT_GRAD = 2,      // g = dy_slot W_down[e]^T, SwiGLU backward in the epilogue
  GK_INPUT_GRAD = 3,    // dx_slot = dgu W_up[e]^T
  GK_W2_GRAD = 4,       // dW_down[e] = hw_e^T dy_slot_e
  GK_W1_GRAD = 5,       // dW_up[e] = x_slot_e^T dgu_e
  GK_FWD_FUSED = 6,     // GEMM1 + SwiGLU and GEMM2 in one launch, GEMM2 row blocks released by
                        // ready counters that GEMM1's epilogue increments
  GK_GEMM2_COMBINE = 7, // GEMM2 with the weighted combine into y in its epilogue
};

struct GemmCall {
  GemmKind kind;
  const void* w_up;    // bf16 [E, H, 2I]
  const void* w_down;  // bf16 [E, I, H]
  void* d_w;           // weight-gradient output (W1/W2 grads)
  uint64_t timeout_ns;
  int inject_stall;    // test hook: withhold the first accumulator hand-off of CTA 0
  int accumulate;      // weight gradients: add into the output instead of overwriting it
  const void* rows;    // if set: token rows read directly (T of them) instead of x_slot/dy_slot
  int* status;         // if set: the status word errors are recorded in
  int split_out;       // GEMM2 / INPUT_GRAD: write o as bf16 hi (off_o) + lo (off_o_lo) rows
  int wgrad_f32;       // weight gradients: fp32 output arrays (else bf16)
  // GEMM2 / fused forward: when comb_y is set, the weighted combine into comb_y runs in the
  // epilogue (the per-(token, 128-column chunk) counters at off_cnt must be zero)
  int skip_gu = 0;     // GEMM1 / fused forward: do not store gate|up (forward only)
  int paired = 0;      // 2: clusters of two CTAs sharing one M = 256 MMA (row-grouped kinds: two
                       // row tiles of one expert; weight gradients: two row tiles of the weight);
                       // 0: one CTA per tile
  void* comb_y = nullptr;
  const float* comb_w = nullptr;
  const void* comb_extra = nullptr;
  const void* comb_extra_lo = nullptr;
  // W2Grad: d_topk_weights [T, K] may be computed by this launch's epilogue warps; if they take
  // it, *d_topk_taken is set and no d_topk kernel is needed
  float* d_topk = nullptr;
  bool* d_topk_taken = nullptr;
};

cudaError_t launch_gemm(const Workspace& w, char* ws, const GemmCall& c, cudaStream_t st);

// Records a description of a host-side failure for mm_last_error_detail (this thread).
void note_error(const char* fmt, ...);

// Trace context for the launch being enqueued on this thread (tracing off: buf == nullptr);
// every launcher passes it to its kernel.
TraceCtx trace_ctx();

// SMs of the current device (0 if it cannot be queried).
int device_sm_count();

// Whether the routing scan may split an expert's rows for weight-gradient `kind` (decided from
// the sizes alone; when false no expert is split and no sum needs launching).
bool wgrad_split_possible(const Workspace& w, int kind);

// The sums of split weight gradients (see WgKind): out[e] for every split expert e of `kind`
// from its fp32 partial slices, in chunk order; bf16 or fp32 output, optionally added in.
cudaError_t launch_wgrad_reduce(const Workspace& w, char* ws, int kind, void* out, bool out_f32,
                                bool accumulate, cudaStream_t st);

}  // namespace mm
