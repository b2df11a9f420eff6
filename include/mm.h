/*
 * mm.h -- C ABI of the fused MoE-FFN layer (forward and backward) for one GB300 GPU.
 *
 * The operation is the one defined by the RFC "HyperParallel Multicore HyperMegaMoE fused
 * forward/backward operator": §2.1 (forward chain Dispatch -> GMM1/up_proj -> SwiGLU ->
 * GMM2/down_proj -> Combine), §2.2 (backward graph and its gradient list), §2.3 and §10
 * (the ACLNN interface's two phases: a workspace-size query, then the call), §3.1
 * (the five public tensors) and §4 (routing semantics and boundary checks). On one GPU the
 * AllToAll dispatch/combine become a permute/unpermute of rows inside device memory.
 *
 * Shapes and layouts (all row-major, contiguous, device memory unless stated):
 *   T tokens, H hidden size, I intermediate size, E experts, K experts per token.
 *   x                 bf16 [T, H]
 *   topk_ids          int32 [T, K]   expert id of slot s = t*K + k, in [0, E)
 *   topk_weights      fp32 [T, K]    routing weight of each slot
 *   up_proj_weight    bf16 [E, H, 2I] gate in columns [0, I), up in [I, 2I)
 *                                     (layout from the multicore usage guide, "inputs and weights")
 *   down_proj_weight  bf16 [E, I, H]
 *   y, dy, dx         bf16 [T, H]
 *   d_topk_weights    fp32 [T, K]
 *   d_up_proj_weight  bf16 [E, H, 2I];  d_down_proj_weight bf16 [E, I, H]
 *                     (fp32, same shapes, with MM_FLAG_FP32_WEIGHT_GRADS)
 *
 * Math: h_s = silu(x_t W_gate[e]) * (x_t W_up[e]) with silu(z) = z*sigmoid(z),
 * o_s = h_s W_down[e], y_t = sum_k topk_weights[t,k] * o_{t*K+k} (k ascending, fp32, rounded
 * once to bf16). Products run on bf16 tensor cores with fp32 accumulation.
 *
 * Ownership: the caller allocates every buffer, including the workspace. The library allocates
 * no device memory. All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 * stream) and nothing synchronises with the host, except mm_get_status, mm_routing_export
 * (host destination) and mm_forward with MM_FLAG_VALIDATE_IDS. Host threads may call
 * concurrently on different workspaces (mm_backward forks work onto a library stream of the
 * calling thread and joins it back); the optional stage timer (mm_timing_*) is process-global
 * and for use from one thread while no other thread calls the library.
 *
 * Errors: host-side checks (null or misaligned pointers, sizes out of range, workspace too
 * small) return an error before anything is enqueued. An expert id outside [0, E) can only be
 * seen on the device: the first routing kernel records MM_ERR_BAD_EXPERT_ID in the workspace's
 * status word, every later kernel of the call sees it and does nothing (no out-of-bounds
 * access), and mm_get_status reports it. Outputs are then unspecified. Device waits are bounded;
 * a wait that runs out records MM_ERR_TIMEOUT the same way.
 */
#ifndef MM_H_
#define MM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mm_status {
  MM_OK = 0,
  MM_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size */
  MM_ERR_UNSUPPORTED = 2,   /* sizes this build does not handle (see mm_forward) */
  MM_ERR_WORKSPACE = 3,     /* workspace null, misaligned or smaller than mm_workspace_size */
  MM_ERR_CUDA = 4,          /* a CUDA runtime call failed (no device, launch error, ...) */
  MM_ERR_BAD_EXPERT_ID = 5, /* some topk_ids entry is outside [0, E) (found on the device) */
  MM_ERR_TIMEOUT = 6,       /* a bounded device-side wait ran out */
  MM_ERR_TOKENS_PER_EXPERT = 7 /* a caller's tokens_per_expert differs from the ids' histogram */
} mm_status;

/* Layer sizes. Supported: T >= 0, H and I multiples of 8 (16-byte rows), 1 <= E <= 1024,
 * 1 <= K <= 16, T*K + E*127 < 2^31. An empty batch (T = 0) is a valid call: the pointers of
 * T-sized tensors (x, topk_ids, topk_weights, y, dy, dx, d_topk_weights) may then be NULL, the
 * forward leaves empty routing tables (a caller's tokens_per_expert must be all zero), and the
 * backward writes zero weight gradients (leaves them unchanged with
 * MM_FLAG_ACCUMULATE_WEIGHT_GRADS). */
typedef struct mm_dims {
  int64_t T, H, I, E, K;
} mm_dims;

/* mm_forward flag: run the id check (and the tokens_per_expert check of mm_forward_ex) first
 * and wait for it on the host (one device-to-host read), returning MM_ERR_BAD_EXPERT_ID or
 * MM_ERR_TOKENS_PER_EXPERT before any GEMM is enqueued. */
#define MM_FLAG_VALIDATE_IDS 0x1u

/* mm_backward flag: add the weight gradients into d_up_proj_weight and d_down_proj_weight
 * (gradient accumulation over micro-batches, RFC §7.1) instead of overwriting them. The addition
 * is done in bf16 by the stores themselves (one rounding of each addend and of each sum); experts
 * with no slot leave their slices unchanged. dx and d_topk_weights are still overwritten. */
#define MM_FLAG_ACCUMULATE_WEIGHT_GRADS 0x2u

/* mm_backward flag: the weight-gradient outputs (d_up_proj_weight, d_down_proj_weight and a shared
 * expert's) are fp32 arrays of the same shapes instead of bf16, written straight from the fp32
 * accumulators. With MM_FLAG_ACCUMULATE_WEIGHT_GRADS the stores add in fp32: gradient
 * accumulation into fp32 "main grad" buffers with one rounding per addition. */
#define MM_FLAG_FP32_WEIGHT_GRADS 0x4u

/* mm_forward flag: run GEMM1 + SwiGLU and GEMM2 in one persistent launch in which a row block's
 * GEMM2 tiles start as soon as all of its GEMM1 tiles have stored their h rows (per-row-block
 * ready counters in the workspace, bounded waits; the RFC's event-counter release of dependent
 * tiles, §5.1) instead of two stream-ordered launches. Results are identical bit for bit in both
 * forms. Without this flag or MM_FLAG_SEPARATE_FORWARD_GEMMS, mm_forward picks the one launch by
 * itself where it measured faster on a GB300: CTA-pair launches (no MM_FLAG_SINGLE_CTA_TILES,
 * MM_FLAG_FUSED_COMBINE or MM_FLAG_TEST_STALL) whose two GEMMs come to 1 to 16 waves of work,
 * estimated from the sizes as ceil(T*K / 256) x (ceil(I / 128) + ceil(H / 256)) units over half
 * the SM count. There the one launch overlaps GEMM1's last partial wave with GEMM2's start; with
 * more waves its releases cost more than that, with less than one GEMM2 cannot start early. */
#define MM_FLAG_FUSED_FORWARD_GEMMS 0x8u

/* mm_forward flag: always run GEMM1 + SwiGLU and GEMM2 as two stream-ordered launches (never the
 * one launch above). Together with MM_FLAG_FUSED_FORWARD_GEMMS: MM_ERR_INVALID_ARG. */
#define MM_FLAG_SEPARATE_FORWARD_GEMMS 0x40u

/* mm_forward flag: fold the weighted combine into GEMM2's epilogue instead of running it as its
 * own kernel. Each epilogue warp, after its o rows are stored and visible, counts each row's token
 * once per 128-column chunk (counters in the workspace); the warp that brings a token's count to K
 * sums that token's K rows of the chunk in slot order and writes y (the RFC's per-token arrival
 * counting at Combine, §2.1, §5.1). y is identical bit for bit to the separate combine's. */
#define MM_FLAG_FUSED_COMBINE 0x10u

/* mm_forward flag: a forward with no backward to follow (inference). GEMM1 stores h only, not
 * the fp32 gate|up activations a backward needs. An mm_backward on that workspace records
 * MM_ERR_INVALID_ARG in the status word and its GEMMs do nothing (outputs unspecified). */
#define MM_FLAG_FORWARD_ONLY 0x20u

/* mm_forward / mm_backward flag: one CTA per 128-row tile in every grouped GEMM. By default
 * GEMM1, GEMM2 (forward), act_grad and input_grad (backward), and the weight gradients when the
 * experts average at least 256 rows, run 256-row tiles shared by the two CTAs of a cluster through one
 * tensor-core MMA (tcgen05 .cta_group::2): each CTA holds its 128 rows of A and half of the
 * weight tile's columns, and receives its own rows of the accumulator. Results are identical bit
 * for bit in both forms. */
#define MM_FLAG_SINGLE_CTA_TILES 0x100u

/* mm_forward flag, a test hook for the failure path only: the first grouped GEMM withholds one
 * accumulator hand-off (first tile of its first CTA) and every device wait of the call is bounded
 * by 50 ms instead of 2 s. The call then ends with MM_ERR_TIMEOUT in the status word (and y is
 * unspecified) instead of hanging; the next call on the same workspace runs normally. */
#define MM_FLAG_TEST_STALL 0x80000000u

/* Bytes of workspace mm_forward/mm_backward need for `d` (RFC §2.3 workspace query).
 * Returns 0 if `d` is unsupported. The workspace holds the routing tables, the dispatched
 * rows x_slot and the saved gate|up activations (kept from mm_forward for mm_backward),
 * and the scratch of both calls. Its contents need no initialisation. */
size_t mm_workspace_size(mm_dims d, uint32_t flags);

/* Forward pass (RFC §2.1): routing (per-expert histogram, prefix offsets, stable permute of
 * the T*K slots), dispatch, GMM1 + SwiGLU, GMM2, weighted combine into y.
 * `workspace` (>= mm_workspace_size bytes, 256-byte aligned) must not be touched by
 * anything else until the last mm_backward for it has been enqueued; two forwards whose
 * backwards are still pending need two workspaces. All tensor pointers 16-byte aligned. */
mm_status mm_forward(mm_dims d, const void* x, const int32_t* topk_ids,
                     const float* topk_weights, const void* up_proj_weight,
                     const void* down_proj_weight, void* y, void* workspace,
                     size_t workspace_bytes, void* stream, uint32_t flags);

/* Backward pass (RFC §2.2) for the forward that last used `workspace`, with upstream
 * gradient dy. Writes (the weight gradients are added in with MM_FLAG_ACCUMULATE_WEIGHT_GRADS):
 *   dx                 = sum over k of the input_grad rows of the token's slots,
 *   d_topk_weights[t,k] = <dy[t], o_{t*K+k}>,
 *   d_up_proj_weight[e]  = x_slot_e^T [d_gate | d_up]   (zero for an expert with no slot),
 *   d_down_proj_weight[e] = (w * h)_e^T dy_slot_e        (zero for an expert with no slot).
 * x, topk_ids, topk_weights and the two weights must be the forward's (the dispatched x rows
 * and the routing are read back from the workspace; x itself is only checked). A backward only
 * reads what mm_forward kept (routing, dispatched x rows, gate|up) and overwrites its own scratch,
 * so one forward may be followed by several backwards (another dy: a retained autograd graph),
 * each giving what a single one would, bit for bit. An expert with far more rows than the
 * average (skewed routing) may have its weight-gradient reduction cut into row chunks whose fp32
 * partial sums are added in a fixed order before the output's one rounding: still deterministic,
 * and the same in every CTA layout (the chunks follow the routing, the sizes and the device's SM
 * count, so GPUs with different SM counts may round such an expert's gradient differently). */
mm_status mm_backward(mm_dims d, const void* dy, const void* x, const int32_t* topk_ids,
                      const float* topk_weights, const void* up_proj_weight,
                      const void* down_proj_weight, void* workspace, size_t workspace_bytes,
                      void* dx, float* d_topk_weights, void* d_up_proj_weight,
                      void* d_down_proj_weight, void* stream, uint32_t flags);

/* Optional shared expert (RFC §6.1, shared-expert fusion): one SwiGLU FFN applied to every token,
 * whose output the combine adds to y with weight 1 (y_t = sum_k w[t,k] o_{t,k} + o_shared_t, one
 * fp32 sum rounded once), and whose input-gradient rows are added into dx the same way. Its
 * intermediate size may differ from the routed experts'. */
typedef struct mm_shared_expert {
  int64_t I;                      /* shared intermediate size I_s (a multiple of 8) */
  const void* up_proj_weight;     /* bf16 [H, 2*I_s]: gate in columns [0, I_s), up in [I_s, 2*I_s) */
  const void* down_proj_weight;   /* bf16 [I_s, H] */
  void* d_up_proj_weight;         /* [H, 2*I_s], written by mm_backward_ex (unused forward) */
  void* d_down_proj_weight;       /* [I_s, H], written by mm_backward_ex (unused forward);
                                     both bf16, or fp32 with MM_FLAG_FP32_WEIGHT_GRADS */
} mm_shared_expert;

/* Optional inputs of the extended entry points. A NULL mm_options, or one whose fields are all
 * NULL, means the plain mm_forward / mm_backward. */
typedef struct mm_options {
  /* A shared expert (NULL: none). The same one must be given to the workspace query, the forward
   * and its backward. */
  const mm_shared_expert* shared;
  /* Forward only, NULL: none. The caller's per-expert slot histogram, device int32 [E], which the
   * multicore usage guide lets a caller pass when it already has it. The layer still computes
   * its own histogram (the routing tables need per-chunk counts) and only compares: a mismatch
   * records MM_ERR_TOKENS_PER_EXPERT in the status word and the rest of the call does nothing. */
  const int32_t* tokens_per_expert;
} mm_options;

/* Workspace bytes for mm_forward_ex / mm_backward_ex with options `opt` (0 if unsupported). The
 * routed part's layout is the same as mm_workspace_size's, followed, with a shared expert, by its
 * saved activations and scratch. */
size_t mm_workspace_size_ex(mm_dims d, const mm_options* opt, uint32_t flags);

/* mm_forward with options: same arguments, errors and workspace rule. */
mm_status mm_forward_ex(mm_dims d, const mm_options* opt, const void* x,
                        const int32_t* topk_ids, const float* topk_weights,
                        const void* up_proj_weight, const void* down_proj_weight, void* y,
                        void* workspace, size_t workspace_bytes, void* stream, uint32_t flags);

/* mm_backward with options. With a shared expert it also writes opt->shared->d_up_proj_weight and
 * d_down_proj_weight (subject to the same flags as the routed weight gradients) and adds the
 * shared expert's input gradient into dx. The workspace must come from mm_forward_ex with the
 * same shared expert. */
mm_status mm_backward_ex(mm_dims d, const mm_options* opt, const void* dy, const void* x,
                         const int32_t* topk_ids, const float* topk_weights,
                         const void* up_proj_weight, const void* down_proj_weight,
                         void* workspace, size_t workspace_bytes, void* dx,
                         float* d_topk_weights, void* d_up_proj_weight, void* d_down_proj_weight,
                         void* stream, uint32_t flags);

/* Synchronises `stream`, then returns the device-side status word of `workspace`
 * (MM_OK, MM_ERR_BAD_EXPERT_ID, MM_ERR_TOKENS_PER_EXPERT or MM_ERR_TIMEOUT), or MM_ERR_CUDA if
 * the stream failed.
 * The word is cleared at the start of every mm_forward. */
mm_status mm_get_status(const void* workspace, void* stream);

/* Copies the routing tables of the last mm_forward on `workspace` into caller buffers
 * (device or host memory; the call synchronises `stream` when any destination is host):
 *   counts[E]        slots per expert,
 *   offsets[E+1]     exclusive prefix sum of counts (offsets[E] = T*K),
 *   row_of_slot[T*K] position of slot s in the expert-sorted order, stable in s.
 * Any destination may be NULL. */
mm_status mm_routing_export(mm_dims d, const void* workspace, int32_t* counts,
                            int32_t* offsets, int32_t* row_of_slot, void* stream);

/* Routing tables for callers that cannot allocate device memory.
 * The paper has no counterpart to this entry point. It exists for callers that may not call
 * cudaMalloc at the point where they need the routing (code inside a framework that owns the
 * device heap, or work prepared ahead of time that may only use pointers it already holds).
 * It computes exactly what mm_forward + mm_routing_export give: counts[E], offsets[E+1] and
 * row_of_slot[T*K] (stable expert-sorted position of each slot), written to caller-provided
 * DEVICE buffers (4-byte aligned); H and I of `d` are ignored. It allocates nothing: its
 * scratch is a static device array of 4 MiB + 256 B that every GPU loading this library holds
 * until the process exits. Limits: T*K <= 2^20, E <= 1024, K <= 16; larger sizes return
 * MM_ERR_UNSUPPORTED (use mm_forward with a workspace). An expert id outside [0, E) makes every
 * output entry -1. All calls share the static scratch: calls whose kernels overlap on the GPU
 * (different streams or host threads) race and must be serialised by the caller. The first call
 * on each device looks up the scratch's device address (cudaGetSymbolAddress); make that first
 * call before any stream capture. Nothing is synchronised with the host. */
mm_status mm_route_noalloc(mm_dims d, const int32_t* topk_ids, int32_t* counts,
                           int32_t* offsets, int32_t* row_of_slot, void* stream);

/* The step and CUDA error of the last MM_ERR_CUDA returned to the calling thread ("" if none). */
const char* mm_last_error_detail(void);

/* Human-readable name of a status code. */
const char* mm_status_string(mm_status s);

/* ABI version of this library (bumped on any change of the exported functions or structs). */
int mm_abi_version(void);

/* Optional per-stage timer. When enabled, every kernel the library enqueues is bracketed by
 * CUDA events on its stream. mm_timing_read synchronises those events, writes for each stage
 * (up to max_stages) the summed milliseconds and the number of launches since the last read,
 * clears them, and returns the number of stages (MM_NUM_STAGES). mm_stage_name names a stage. */
#define MM_NUM_STAGES 17
mm_status mm_timing_enable(int on);
/* Restricts the timer to the stages whose bit (1 << stage) is set in stage_mask (default: all),
 * so that a timed run can bracket only the kernel it reports on. */
mm_status mm_timing_select(uint32_t stage_mask);
int mm_timing_read(double* ms, int64_t* launches, int max_stages);
const char* mm_stage_name(int stage);

/* Optional per-tile trace: when and where each piece of work ran. The RFC's performance
 * acceptance (§8) asks for the concurrency and utilisation of the cube (matrix) and vector
 * units over time; on a GB300 each grouped-GEMM CTA has both in one SM: the tensor-core
 * mainloop, and the epilogue warps that apply the elementwise math and store the tile. While a
 * trace buffer is set, every kernel that mm_forward / mm_backward (and their _ex forms) enqueue
 * writes records into it:
 *   MM_TRACE_CTA       one per CTA: from its start (after the stream's previous kernel completed)
 *                      to the end of its work (the CTA's first thread);
 *   MM_TRACE_MAINLOOP  one per grouped-GEMM tile (per unit of two row tiles for the CTA-pair
 *                      MMAs, recorded by the even CTA that issues them): from the MMA-issuing
 *                      thread taking a free accumulator to its commit of the tile's last MMA;
 *   MM_TRACE_EPILOGUE  one per tile and CTA: from the accumulator being ready to the end of the
 *                      first epilogue warp's work on it (the other warps' spans are alike).
 * Times are %globaltimer nanoseconds (one clock for all SMs). The buffer is device memory,
 * 32-byte aligned: a 32-byte header whose first uint32 counts the records offered, then
 * bytes / 32 - 1 record slots; records past the last slot are dropped (the count still
 * includes them). The caller zeroes the header before the calls it wants traced (records are
 * placed at the count's value). Each traced launch gets the next sequence number
 * (`launch`), starting at 0 when the buffer is set. A kernel captured into a CUDA graph keeps
 * the buffer and sequence number it was captured with. Process-global, for use from one thread
 * while no other thread calls the library (like the stage timer). Each record costs an atomic
 * add and two stores: time untraced runs. mm_trace_set(NULL, 0) turns tracing off. */
typedef struct mm_trace_record {
  uint16_t stage;   /* mm_stage_name(stage) */
  uint16_t role;    /* MM_TRACE_CTA, MM_TRACE_MAINLOOP or MM_TRACE_EPILOGUE */
  uint16_t sm;      /* %smid of the SM that ran it */
  uint16_t rank;    /* the CTA's rank in its pair (CTA-pair MMAs), else 0 */
  int32_t unit;     /* MM_TRACE_CTA: blockIdx.x; else the tile (or pair unit) index in the launch */
  uint32_t launch;  /* sequence number of the launch */
  uint64_t t0, t1;  /* %globaltimer at start and end, ns */
} mm_trace_record;
#define MM_TRACE_CTA 0
#define MM_TRACE_MAINLOOP 1
#define MM_TRACE_EPILOGUE 2
/* Sets (or with NULL clears) the trace buffer. MM_ERR_INVALID_ARG if the pointer is not 32-byte
 * aligned or bytes < 64 (a header and one record). */
mm_status mm_trace_set(void* device_buffer, size_t bytes);

#ifdef __cplusplus
}
#endif

#endif /* MM_H_ */
