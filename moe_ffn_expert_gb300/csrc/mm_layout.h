// Workspace layout and launch-side declarations shared by the library's translation units.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/mm.h"

namespace mm {

// Row tiles of the grouped GEMMs. Every expert's rows are padded up to a multiple of BM in
// the expert-sorted buffers, so a row tile never straddles two experts and pad rows hold
// zeros (they then add nothing to the weight-gradient reductions).
constexpr int BM = 128;
constexpr int BK = 64;   // 64 bf16 = 128 bytes: one 128B-swizzle row
constexpr int BN = 256;  // accumulator columns per tile (fp32, one TMEM column each)

// Slots handled by one warp in the routing kernels.
constexpr int ROUTE_CHUNK = 512;

// Header words (int32) at the start of the workspace.
enum HeaderWord {
  HDR_STATUS = 0,      // mm_status of the call (0 = OK)
  HDR_NUM_MTILES = 1,  // number of BM-row tiles over all experts (padded rows / BM)
  HDR_BAD_SLOT = 2,    // first slot seen with an invalid expert id (diagnostics)
  HDR_NO_BACKWARD = 3, // nonzero: the forward kept no gate|up (MM_FLAG_FORWARD_ONLY)
  HDR_NUM_MPAIRS = 4,  // pairs of row tiles of one expert (the paired GEMMs' work units)
  HDR_WG_CHUNKS = 5,   // 2 words: row chunks of the weight-gradient plan (W2Grad, W1Grad)
  HDR_WG_SPLITS = 7,   // 2 words: experts whose weight gradient is split into several chunks
  HDR_WORDS = 64
};

// Weight-gradient plan (one per weight-gradient kind, written by the routing scan): the
// reduction over an expert's rows runs as one or more row chunks. An expert whose rows are long
// against the launch's average load per CTA pair is split into chunks of whole 64-row blocks;
// each chunk's tile goes to an fp32 partial slice and a reduce kernel sums the slices in chunk
// order. Chunk c: {expert, first padded row, rows, slice (-1: the output itself)}; split expert
// j: {expert, first slice, slices, 0}. Split chunks come first, then the other experts' chunks
// in expert order.
enum WgKind { WG_W2 = 0, WG_W1 = 1 };

// What the routing scan needs to write the plans (int32 quadruples).
struct WgPlanArgs {
  int32_t* plan;    // [2][plan_stride][4] row chunks
  int32_t* red;     // [2][E][4] split experts
  int units[2];     // CTA-pair work units per row chunk (row-tile pairs x column tiles)
  int slices[2];    // partial slices that fit for each kind
  int plan_stride;  // E + the larger slice count
  int pairs;        // CTA pairs the weight-gradient launches run on
};

// Stage ids of the per-stage timer.
enum Stage {
  ST_ROUTE_COUNT = 0,
  ST_ROUTE_SCAN,
  ST_ROUTE_RANK,
  ST_GATHER_X,
  ST_GEMM1_SWIGLU,
  ST_GEMM2,
  ST_COMBINE_Y,
  ST_GATHER_DY,
  ST_ACT_GRAD,
  ST_D_TOPK,
  ST_W2_GRAD,
  ST_INPUT_GRAD,
  ST_COMBINE_DX,
  ST_W1_GRAD,
  ST_SHARED,     // every launch of the shared expert (forward and backward)
  ST_FWD_GEMMS,  // the fused GEMM1 + SwiGLU -> GEMM2 launch
  ST_WGRAD_REDUCE,  // the sums of split weight gradients' partial slices
  ST_COUNT
};
static_assert(ST_COUNT == MM_NUM_STAGES, "stage table");

// Trace context of one launch (a kernel argument): the caller's buffer (a header word counting
// the records offered, then 32-byte mm_trace_record slots from byte 32), its record capacity,
// and the launch's stage and sequence number. buf == nullptr: tracing is off.
struct TraceCtx {
  uint32_t* buf;
  uint32_t cap;
  uint32_t stage;
  uint32_t launch;
};

// Byte offsets of every region in the caller's workspace (all 256-byte aligned).
struct Workspace {
  int64_t T, H, I, E, K, S;
  int64_t S_pad;        // worst-case padded rows (multiple of BM)
  int64_t n_chunks;     // routing chunks of ROUTE_CHUNK slots
  int64_t n_act_tiles;  // rows of the d_topk partials: 2 column halves x ceil(I / BN) tiles
  size_t off_hdr, off_counts, off_offsets, off_poff, off_chunk, off_tile_expert;
  size_t off_ready;  // int32 [S_pad / BM] fused forward: GEMM1 epilogue warps done per row tile
  size_t off_cnt;    // int32 [T][ceil(H / 128)] fused combine: slots stored per token and chunk
  size_t off_pair_tile;  // int32 [S_pad / BM] first row tile of each pair; ~tile if the pair's
                         // second tile belongs to another expert
  size_t off_row_of_slot, off_slot_of_row, off_w_row;
  size_t off_x_slot;   // bf16 [S_pad, H]   dispatched x rows (kept for W1Grad)
  size_t off_gu;       // fp32 [S_pad, 2I]  gate|up accumulators (kept for the backward)
  size_t off_h;        // bf16 [S_pad, I]   hi part of w*h (kept for the backward)
  size_t off_hw_lo;    // bf16 [S_pad, I]   lo part of w*h (kept for the backward)
  size_t off_o;        // bf16 [S_pad, H]   forward: w*o;  backward: dx rows
  size_t off_dy_slot;  // bf16 [S_pad, H]   dispatched dy rows
  size_t off_dgu;      // bf16 [S_pad, 2I]  hi part of [d_gate | d_up]
  size_t off_dgu_lo;   // bf16 [S_pad, 2I]  lo part of [d_gate | d_up]
  size_t off_p_part;   // fp32 [n_act_tiles, S_pad] per-column-half partials of <g, h>
  size_t off_o_lo;     // bf16 [S_pad, H]   direct-row layout only: lo part of o / dx rows
  size_t off_wg_plan;  // int4 [2][E + wg_slices_max] weight-gradient row chunks (see WgKind)
  size_t off_wg_red;   // int4 [2][E] split experts of each weight-gradient kind
  // fp32 partial slices of split weight gradients: W2Grad's in the o / dx row buffer (free from
  // the forward's combine until input_grad writes it), W1Grad's in the dy row buffer (free
  // after act_grad and W2Grad); how many slices of each kind fit (0: no split)
  int64_t wg_slices[2];
  int64_t wg_slices_max;
  size_t total;
};

// Fills `w` for the sizes in `d`; returns false if the sizes are unsupported. With direct_rows
// the layout has no dispatched-row buffers (x_slot, dy_slot): the shared expert's GEMMs read the
// token rows of x and dy themselves (its routing is the identity).
bool plan_workspace(const mm_dims& d, Workspace* w, bool direct_rows = false);

}  // namespace mm
