// Grouped GEMMs of the MoE-FFN layer on the sm_103a tensor cores (tcgen05 + TMEM), fed by TMA.
//
// One persistent, warp-specialised kernel template serves all products of the layer (RFC
// "HyperParallel Multicore HyperMegaMoE fused forward/backward operator", §2.1 GMM1/GMM2, §2.2
// act_grad, input_grad, W2Grad and W1Grad), every one on 128 x 256 accumulator tiles:
//
//   kind          A (rows x red.)            B (red. x cols)              epilogue
//   GEMM1         x_slot [rows,H]  K-maj     W_up[e]   [H,2I]  N-major    gu = [gate|up] (fp32), w*h
//   GEMM2         w*h    [rows,I]  K-maj     W_down[e] [I,H]   N-major    w*o (bf16; hi + lo if split)
//   ACT_GRAD      dy_slot[rows,H]  K-maj     W_down[e]^T       K-major    SwiGLU backward: dgu, <g,h>
//   INPUT_GRAD    dgu    [rows,2I] K-maj     W_up[e]^T         K-major    dx_slot (bf16)
//   W2_GRAD       hw_e^T [I,M_e]   M-maj x2  dy_slot_e [M_e,H] N-major    dW_down[e]
//   W1_GRAD       dgu_e^T[2I,M_e]  M-maj x2  x_slot_e [M_e,H]  N-major    dW_up[e] (stored transposed)
//   FWD_FUSED     GEMM1 and GEMM2 tiles in one launch (GEMM2 row blocks released by counters)
//   GEMM2_COMBINE GEMM2 whose epilogue also sums y for the tokens whose last slot it stores
//
// The routing weight w of a row is applied where its h is made: GEMM1's epilogue writes w*h, so
// GEMM2 gives the weighted expert output w*o and the combine sums a token's rows with weight 1
// (the same products, one rounding of w*h instead of h; the RFC's weighted merge, §4.1).
//
// Precision of the weight gradients. They reduce over all rows of an expert (hundreds to
// thousands), so a bf16 rounding of every row of an operand would leave errors of ~0.5% of the
// gradient's rms. The forward therefore keeps the gate|up accumulators in fp32 and writes w*h,
// and the act_grad epilogue [d_gate|d_up], as two bf16 planes, hi = bf16(v) and
// lo = bf16(v - hi), which together carry ~16 mantissa bits (GEMM2 and input_grad read hi
// only). Both weight gradients put that pair on the A side ("x2" above) and issue two MMAs per
// k-step (hi and lo against the same B tile) into one fp32 accumulator; W1_GRAD therefore
// computes dW_up^T and its epilogue transposes.
// Their stages hold A hi, A lo and B: 64 KB, three of them.
//
// Row-grouped kinds walk 128-row tiles of the expert-sorted (padded) row buffers; each tile
// belongs to one expert, whose weight slab is the third coordinate of a 3-D tensor map.
// Weight-gradient kinds walk (expert, row tile, column tile) of the weight, reducing over
// the expert's rows (the last 64-row block trimmed to 16-row MMA steps; pad rows are zero, an
// expert with no rows gets a zero tile).
//
// CTA pairs (template argument PAIR = 2, the default for GEMM1, GEMM2, ACT_GRAD, INPUT_GRAD and
// long weight gradients): two CTAs of a cluster share one 256 x 256 tcgen05.mma.cta_group::2 per
// 16-deep step. Each holds its own 128 rows of A and half of B's columns (32 KB stages, six
// deep, four for act_grad beside its epilogue's staging; 48 KB and four deep for the split
// weight gradients), both CTAs' TMA loads complete on
// the even CTA's stage barrier, the even CTA's MMA thread issues the MMAs and signals its
// commits to both CTAs' barriers, and each CTA's epilogue drains its own 128 accumulator rows.
// Every TMA load of a CTA writes only its own shared memory and reads only this GPU's memory.
//
// Warp roles (320 threads, one CTA per SM, grid <= SM count, static round-robin over tiles):
//   warp 0      one thread issues TMA loads into a 4-stage (3 for act_grad and the weight
//               gradients; the pair counts above) shared-memory ring (mbarrier per stage,
//               transaction-count completion);
//   warp 1      allocates 2*BN TMEM columns (two 128xBN fp32 accumulators); one thread issues
//               tcgen05.mma (128xBNx16 per instruction; 256xBNx16 over a pair, from the even CTA)
//               and tcgen05.commit's the stage and accumulator barriers;
//   warps 2-9   epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes 32*(w%4)..+31,
//               32 tile rows; warps w and w+4 take one column half each), apply the kind's
//               epilogue through per-warp shared-memory staging (TMA or coalesced stores), and
//               release the accumulator so the next tile's MMAs overlap this epilogue.
// All operand tiles use the 128-byte swizzle; every mbarrier wait is bounded by %globaltimer and
// a wait that runs out records MM_ERR_TIMEOUT, stops the role and still frees TMEM.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "mm_device.cuh"
#include "mm_kernels.h"

namespace mm {
namespace {

constexpr int STAGE_BYTES = 48 * 1024;       // one CTA per tile: A (128 x 64) and B (256 x 64)
constexpr int A_BYTES = BM * BK * 2;         // 16 KB
constexpr int MN_BLOCK_BYTES = 64 * BK * 2;  // one 64-wide MN block of an MN-major tile: 8 KB
constexpr int NUM_EPI_WARPS = 8;             // two per TMEM lane quarter, one per column half
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr int BAR_BYTES = 512;
constexpr int GU_CHUNK_BYTES = 2 * 32 * 16 * 4;  // act_grad: 32 rows x 16 fp32 of gate and of up
constexpr int OUT_PLANE_BYTES = 32 * 16 * 2;     // act_grad: 32 rows x 16 bf16 of one output plane
constexpr int OUT_CHUNK_BYTES = 4 * OUT_PLANE_BYTES;  // d_gate and d_up; hi and lo each

// Store maps of the act_grad epilogue: [d_gate|d_up] hi and lo as [rows][2][I] (so a store
// never crosses from the gate half into the up half).
struct alignas(128) EpiMaps {
  CUtensorMap dgu_hi, dgu_lo;
  CUtensorMap out;  // the bf16 output of GEMM2, INPUT_GRAD and the weight gradients
  CUtensorMap out_lo;  // its lo part (GEMM2 / INPUT_GRAD with split_out)
  CUtensorMap a2, b2;  // the fused forward's second GEMM: h rows and W_down
  CUtensorMap part;    // weight gradients: fp32 partial slices of split experts' row chunks
};

static_assert(offsetof(EpiMaps, out_lo) == offsetof(EpiMaps, out) + sizeof(CUtensorMap),
              "the split output's lo map follows its hi map");

constexpr int OUT_TILE_BYTES = 32 * 32 * 2;  // 32 rows x 32 bf16 of staged output (64-byte rows)
constexpr int B_HALF_ROWS = BN / 2;          // a CTA of a pair loads half of B's N extent
static_assert(BK == 64, "one 128-byte swizzle row per k-block");

struct Args {
  const int* hdr;
  const int32_t* tile_expert;
  const int32_t* poff;
  const int32_t* counts;  // weight-gradient kinds: rows of each expert (without padding)
  int* status;
  int n_tiles_n;   // column tiles
  int k_iters;     // row-grouped kinds: reduction blocks of BK
  int E;
  int m_tiles_w;   // weight-gradient kinds: row tiles of the weight
  int N;           // valid output columns
  int M;           // weight-gradient kinds: valid output rows
  int I;           // intermediate size
  void* out0;  // bf16, except fp32 gate|up of GEMM1 and fp32 weight gradients (wgrad_f32)
  int64_t ld0;
  __nv_bfloat16* out1;
  int64_t ld1;
  __nv_bfloat16* out2;  // lo plane of the act_grad epilogue
  __nv_bfloat16* out3;  // GEMM1: lo plane of w*h
  const float* gu;
  int64_t ld_gu;
  const float* w_row;  // routing weight of every padded row (0 for pad rows)
  float* p_part;
  int64_t S_pad;
  int64_t out_expert_stride;
  uint64_t timeout_ns;
  int inject_stall;
  int accumulate;  // weight gradients: reduce-add into the output
  int split_out;   // GEMM2 / INPUT_GRAD: store the output as bf16 hi and lo planes
  int wgrad_f32;   // weight gradients: fp32 output (else bf16)
  // fused forward: GEMM2 column tiles, reduction blocks, window of row tiles, ready counters
  int n2, k2, win;
  int* ready;
  int ready_target;
  // GEMM2 with the combine fused into its epilogue (y[t] summed by the last of its K slots)
  int fuse_combine;
  int* cnt;                       // [T][comb_nch] slots stored so far per 128-column chunk
  const int32_t* slot_of_row;
  const int32_t* row_of_slot;
  const float* comb_w;            // routing weights [T][K]
  const __nv_bfloat16* comb_o;    // o rows [S_pad][H]
  const __nv_bfloat16* comb_extra;     // optional row per token added with weight 1 (hi)
  const __nv_bfloat16* comb_extra_lo;  // and its lo part
  __nv_bfloat16* comb_y;          // [T][H]
  int comb_K, comb_H, comb_nch;
  int skip_gu;  // GEMM1: forward only, gate|up are not stored
  const int32_t* pair_tile;  // paired launches: first row tile of each pair (~tile: no second)
  TraceCtx trace;            // optional per-tile trace (trace.buf == nullptr: off)
  const int4* wg_plan;       // weight gradients: the row chunks of this kind (see WgKind)
  int wg_kind;               // WG_W2 or WG_W1
  // W2Grad: d_topk_weights computed by the epilogue warps before their first tile (see
  // epilogue_d_topk); null when a separate kernel does it
  float* d_topk;
  const int32_t* row_of_slot_d;
  int d_topk_S;
  int d_topk_tiles;
};

template <int KIND>
struct Traits {
  static constexpr bool WGRAD = (KIND == GK_W2_GRAD || KIND == GK_W1_GRAD);
  static constexpr bool A_MN = WGRAD;
  static constexpr bool FUSED = (KIND == GK_FWD_FUSED);
  static constexpr bool GEMM2_LIKE = (KIND == GK_GEMM2 || KIND == GK_GEMM2_COMBINE);
  static constexpr bool B_MN = (KIND == GK_GEMM1_SWIGLU || GEMM2_LIKE || FUSED ||
                                KIND == GK_W2_GRAD || KIND == GK_W1_GRAD);
  // The weight gradients' split operand (bf16 hi + lo, two MMAs per k-step into one fp32
  // accumulator) is always A: W2Grad computes (w h)^T dy_rows with A = w h; W1Grad computes the
  // transpose dW_up^T = [d_gate|d_up]^T x_rows with A = [d_gate|d_up] and its epilogue stores the
  // transpose. Both then run 128 x 256 tiles like the row-grouped kinds.
  static constexpr bool A_SPLIT = WGRAD;
  static constexpr bool TRANSPOSED_OUT = (KIND == GK_W1_GRAD);
  // GEMM1 runs an expert's lone last row tile as an M = 128 pair MMA (64 rows per CTA). GEMM2 and
  // input_grad could too (their epilogues follow epi_geom), but measured on a GB300 GEMM2 got 7 %
  // slower (its 12-block reductions make a half unit's mainloop shorter than the epilogue it
  // overlaps) and input_grad stayed the same; act_grad and the fused forward keep per-row state
  // over a CTA's 128 rows (<g,h> partials, ready counts)
  static constexpr bool HALF = (KIND == GK_GEMM1_SWIGLU);
  static_assert(!HALF || (!WGRAD && !FUSED), "half units are row tiles of the row-grouped GEMM1");
  static_assert(!TRANSPOSED_OUT || WGRAD, "only a weight gradient is stored transposed");
  static constexpr int TN = BN;  // accumulator columns per tile
  static constexpr int B_BYTES = TN * BK * 2;
  static constexpr int A_LO_OFF = A_BYTES;                                   // if A_SPLIT
  static constexpr int B_OFF = A_BYTES * (A_SPLIT ? 2 : 1);
  static constexpr int STAGE_BYTES = B_OFF + B_BYTES;  // 48 KB, 64 KB with the A lo plane
  static constexpr uint32_t TMEM_COLS = 2 * TN;
  static constexpr uint32_t IDESC = idesc_bf16_f32(BM, TN, A_MN ? 1 : 0, B_MN ? 1 : 0);
  static_assert(A_SPLIT || STAGE_BYTES == ::mm::STAGE_BYTES, "stage layout");
  static_assert(!A_SPLIT || A_LO_OFF + A_BYTES == B_OFF, "A lo plane layout");
  // act_grad trades one mainloop stage for per-warp staging of its gate|up input and of its
  // four output planes (TMA in, TMA out); the weight gradients' 64 KB stages fit three times
  static constexpr bool GU_STAGING = (KIND == GK_ACT_GRAD);
  static constexpr int STAGES = (GU_STAGING || WGRAD) ? 3 : 4;
  // GEMM2, INPUT_GRAD and the weight gradients stage their bf16 output per warp (two 32x32
  // buffers) and store it with TMA
  static constexpr bool OUT_STAGING =
      (GEMM2_LIKE || KIND == GK_INPUT_GRAD || WGRAD || FUSED);
  // GEMM1 copies its outputs out through a 4 KB per-warp buffer with coalesced stores (the
  // fused forward uses the same 4 KB for both of its epilogues)
  static constexpr bool ROW_STAGING = (KIND == GK_GEMM1_SWIGLU || FUSED);
  static constexpr int EPI_BYTES = GU_STAGING    ? NUM_EPI_WARPS * (GU_CHUNK_BYTES + OUT_CHUNK_BYTES)
                                   : OUT_STAGING ? NUM_EPI_WARPS * 2 * OUT_TILE_BYTES
                                   : ROW_STAGING ? NUM_EPI_WARPS * 4096
                                                 : 0;
  static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + EPI_BYTES + 1024 + BAR_BYTES;
  static_assert(SMEM <= 232448, "shared memory budget");
  // a CTA of a pair MMA (M = 256 over two CTAs) holds its A rows (hi and lo) and half of B's
  // columns per stage: 32 KB six deep (four beside act_grad's staging), 48 KB four deep for the
  // weight gradients
  static constexpr int PAIR_STAGE_BYTES = B_OFF + B_BYTES / 2;
  static constexpr int PAIR_STAGES = (WGRAD || GU_STAGING) ? 4 : 6;
  // with half of B per stage, act_grad's epilogue warps keep two gate|up chunks in flight
  static constexpr int PAIR_GU_BUFS = GU_STAGING ? 2 : 1;
  static constexpr int PAIR_EPI_BYTES =
      GU_STAGING ? NUM_EPI_WARPS * (PAIR_GU_BUFS * GU_CHUNK_BYTES + OUT_CHUNK_BYTES) : EPI_BYTES;
  static constexpr size_t PAIR_SMEM =
      (size_t)PAIR_STAGES * PAIR_STAGE_BYTES + PAIR_EPI_BYTES + 1024 + BAR_BYTES;
  static_assert(PAIR_SMEM <= 232448, "pair-MMA shared memory budget");
};

struct Tile {
  int e, m0, n0, kiters, row0;
  int klast;  // 16-deep MMA steps issued for the last reduction block (BK / 16 unless trimmed)
  int part;  // fused forward: 0 = GEMM1 + SwiGLU tile, 1 = GEMM2 tile
  int half;  // pair MMAs: 1 = an M = 128 unit over one row tile, this CTA's 64 rows from m0
  int slot;  // weight gradients: the fp32 partial slice of a split expert's chunk, -1: the output
};

// Where one epilogue warp's share of a tile's accumulator sits and where it goes: 32 rows from
// row0; nch chunks of 32 columns, chunk j read from tensor-memory column tcol0 + 32 j (GEMM1: its
// up values from tcol0 + up_off + 32 j) and written to output column ocol0 + 32 j.
struct EpiGeom {
  int row0, nch, tcol0, up_off, ocol0;
};

// Warp (q = lane quarter, hf = column half) of a tile. An M = 256 pair unit (or a one-CTA tile)
// leaves rows 32 q .. 32 q + 31 of the CTA's 128 in the warp's lanes with all of the unit's
// columns. An M = 128 pair unit leaves the CTA's 64 rows in lanes 0-63 with the unit's first N/2
// columns and again in lanes 64-127 with the last N/2, both in tensor-memory columns 0 .. N/2 - 1
// (measured once on a GB300 with an MMA whose accumulator held its own coordinates).
template <bool GATE_UP>
__device__ __forceinline__ EpiGeom epi_geom(const Tile& t, int q, int hf, int TN) {
  EpiGeom g;
  if (!t.half) {
    g.row0 = t.m0 + 32 * q;
    g.nch = GATE_UP ? 2 : TN / 64;
    g.tcol0 = GATE_UP ? 64 * hf : (TN / 2) * hf;
    g.up_off = GATE_UP ? 128 : 0;
    g.ocol0 = t.n0 + g.tcol0;
  } else {
    g.row0 = t.m0 + 32 * (q & 1);
    g.nch = GATE_UP ? 1 : TN / 128;
    // GEMM1: a CTA's B half holds 64 gate and the matching 64 up columns
    g.tcol0 = GATE_UP ? 32 * hf : (TN / 4) * hf;
    g.up_off = GATE_UP ? 64 : 0;
    g.ocol0 = GATE_UP ? t.n0 + 64 * (q >> 1) + 32 * hf : t.n0 + (TN / 2) * (q >> 1) + (TN / 4) * hf;
  }
  return g;
}

// Work order of the fused forward over nm row blocks (row tiles, or pairs of row tiles for the
// pair MMAs): GEMM1 units of row-block window 0, then for each later window w its GEMM1 units
// followed by window w-1's GEMM2 units, then the last window's GEMM2 units. Every GEMM2 unit of a
// row block comes after all of that block's GEMM1 units, and about a window of GEMM1 work
// separates them. Unit i -> row block m, part (0 = GEMM1, 1 = GEMM2), column tile nt.
__device__ __forceinline__ void fused_order(const Args& a, int nm, int i, int& m, int& part,
                                            int& nt) {
  const int W = a.win, n1 = a.n_tiles_n, n2 = a.n2;
  const int nw = (nm + W - 1) / W;
  const int mL = nm - (nw - 1) * W;  // row blocks of the last window
  const int A = W * n1, B = W * n2;
  int w, r;
  const int first = (nw == 1 ? mL : W) * n1;
  if (i < first) {
    w = 0, part = 0, r = i;
  } else {
    i -= first;
    const int full_pairs = nw >= 2 ? nw - 2 : 0;
    if (i < full_pairs * (A + B)) {
      const int p = i / (A + B), q = i - p * (A + B);
      if (q < A)
        w = p + 1, part = 0, r = q;
      else
        w = p, part = 1, r = q - A;
    } else {
      i -= full_pairs * (A + B);
      if (nw >= 2 && i < mL * n1) {
        w = nw - 1, part = 0, r = i;
      } else {
        if (nw >= 2) i -= mL * n1;
        if (nw >= 2 && i < B) {
          w = nw - 2, part = 1, r = i;
        } else {
          if (nw >= 2) i -= B;
          w = nw - 1, part = 1, r = i;
        }
      }
    }
  }
  const int n = part ? n2 : n1;
  m = w * W + r / n;
  nt = r - (r / n) * n;
}

template <int KIND>
__device__ __forceinline__ Tile decode_tile(const Args& a, int tile) {
  Tile t;
  t.part = 0;
  t.half = 0;
  t.slot = -1;
  t.klast = BK / 16;
  if constexpr (Traits<KIND>::FUSED) {
    int mt, part, nt;
    fused_order(a, __ldg(a.hdr + HDR_NUM_MTILES), tile, mt, part, nt);
    t.part = part;
    t.e = __ldg(a.tile_expert + mt);
    t.m0 = mt * BM;
    t.n0 = part ? nt * BN : nt * (BN / 2);
    t.row0 = t.m0;
    t.kiters = part ? a.k2 : a.k_iters;
  } else if constexpr (Traits<KIND>::WGRAD) {
    // tile = (row chunk of the plan, row tile of the weight, column tile); a chunk is an
    // expert's rows or, for a split expert, a run of whole 64-row blocks of them
    const int per_c = a.m_tiles_w * a.n_tiles_n;
    const int c = tile / per_c;
    const int rem = tile - c * per_c;
    const int mt = rem / a.n_tiles_n;
    const int nt = rem - mt * a.n_tiles_n;
    const int4 ch = __ldg(a.wg_plan + c);  // {expert, first padded row, rows, slice}
    t.e = ch.x;
    t.m0 = mt * BM;
    t.n0 = nt * Traits<KIND>::TN;
    t.row0 = ch.y;
    t.slot = ch.w;
    // the reduction runs over the chunk's rows only: whole blocks of BK rows, then as many
    // 16-row MMA steps as the last block needs (its pad rows are zero and add nothing)
    const int rows = ch.z;
    t.kiters = (rows + BK - 1) / BK;
    if (t.kiters > 0) t.klast = (rows - (t.kiters - 1) * BK + 15) / 16;
  } else {
    const int mt = tile / a.n_tiles_n;
    const int nt = tile - mt * a.n_tiles_n;
    t.e = __ldg(a.tile_expert + mt);
    t.m0 = mt * BM;
    t.n0 = (KIND == GK_GEMM1_SWIGLU) ? nt * (BN / 2) : nt * BN;
    t.row0 = t.m0;
    t.kiters = a.k_iters;
  }
  return t;
}

// Work units of the paired launches. Row-grouped kinds: a unit is two row tiles of the same
// expert and one column tile, so both CTAs need the same B tile (the expert's weights); CTA r of
// the pair takes row tile mt0 + r. When an expert has an odd number of row tiles its last row
// tile is a unit of its own: for GEMM1 an M = 128 MMA over the pair (HALF kinds: CTA r takes rows
// 64 r .. 64 r + 63 of the tile; t.half = 1), for the other kinds an M = 256 MMA whose second CTA
// loads other rows of the buffer (or zeros past it), takes part in the MMAs and stores nothing.
// Weight gradients: a unit is two 128-row tiles of the weight (same expert, same column tile);
// a second tile past the weight's rows is likewise computed and not stored.
template <int KIND>
__device__ __forceinline__ Tile decode_pair(const Args& a, int unit, uint32_t rank, bool& valid) {
  if constexpr (Traits<KIND>::WGRAD) {
    // unit = (row chunk, pair of weight row tiles, column tile); rank r takes row tile 2p + r
    const int mp = (a.m_tiles_w + 1) / 2;
    const int per_c = mp * a.n_tiles_n;
    const int c = unit / per_c;
    const int rem = unit - c * per_c;
    const int p = rem / a.n_tiles_n;
    const int nt = rem - p * a.n_tiles_n;
    Tile t = decode_tile<KIND>(a, (c * a.m_tiles_w + 2 * p) * a.n_tiles_n + nt);
    t.m0 += (int)rank * BM;
    valid = t.m0 < a.M;
    return t;
  }
  int p, nt, part = 0;
  if constexpr (Traits<KIND>::FUSED) {  // the fused order over pairs of row tiles
    fused_order(a, __ldg(a.hdr + HDR_NUM_MPAIRS), unit, p, part, nt);
  } else {
    p = unit / a.n_tiles_n;
    nt = unit - p * a.n_tiles_n;
  }
  const int pt = __ldg(a.pair_tile + p);
  const int mt0 = pt >= 0 ? pt : ~pt;
  Tile t;
  t.half = Traits<KIND>::HALF && pt < 0;
  valid = rank == 0 || pt >= 0 || t.half;
  t.part = part;
  t.klast = BK / 16;
  t.e = __ldg(a.tile_expert + mt0);
  t.m0 = t.half ? mt0 * BM + (BM / 2) * (int)rank : (mt0 + (int)rank) * BM;
  const bool gate_up = KIND == GK_GEMM1_SWIGLU || (Traits<KIND>::FUSED && part == 0);
  t.n0 = gate_up ? nt * (BN / 2) : nt * BN;
  t.row0 = t.m0;
  t.kiters = part ? a.k2 : a.k_iters;
  return t;
}

__device__ __forceinline__ uint4 pack8_bf16(const float* v) {
  uint4 q;
  q.x = pack_bf16(v[0], v[1]);
  q.y = pack_bf16(v[2], v[3]);
  q.z = pack_bf16(v[4], v[5]);
  q.w = pack_bf16(v[6], v[7]);
  return q;
}

// hi = bf16(v), lo = bf16(v - hi), 8 values each packed into one 16-byte word.
__device__ __forceinline__ void split8_bf16(const float* v, uint4& hi, uint4& lo) {
  float h[8], l[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    h[j] = __bfloat162float(__float2bfloat16_rn(v[j]));
    l[j] = v[j] - h[j];
  }
  hi = pack8_bf16(h);
  lo = pack8_bf16(l);
}

// Coalesced copy-out through a per-warp 4 KB staging buffer. A lane first writes its own row
// (32 values) into the buffer; after __syncwarp the warp reads it back row-major so that each
// store instruction covers whole 128-byte lines of consecutive rows, instead of 32 rows at
// 16 bytes each. The stores are streaming (evict-first) unless asked otherwise: GEMM1's outputs
// are next read by a later kernel, after far more data than L2 holds has passed through it, so
// they need not displace the GEMMs' operand tiles there. 16-byte unit u of row r sits at unit
// u ^ (r & 7) (fp32, 128-byte rows) or u ^ ((r >> 1) & 3) (bf16, 64-byte rows), so both the row
// writes and the line reads are free of bank conflicts.
__device__ __forceinline__ void stage_row_f32(uint8_t* stage, int lane, const float* v) {
  uint8_t* rowp = stage + lane * 128;
#pragma unroll
  for (int u = 0; u < 8; ++u)
    *reinterpret_cast<float4*>(rowp + ((u ^ (lane & 7)) << 4)) =
        make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
}

// Rows row0..row0+31 of an fp32 matrix (leading dimension ld), columns n..n+31 masked at N.
__device__ __forceinline__ void copy_out_f32(const uint8_t* stage, int lane, float* base,
                                             int64_t row0, int64_t ld, int n, int N) {
  const int u = lane & 7;
  if (n + 4 * u >= N) return;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 4 * i + (lane >> 3);
    const float4 v = *reinterpret_cast<const float4*>(stage + r * 128 + ((u ^ (r & 7)) << 4));
    __stcs(reinterpret_cast<float4*>(base + (row0 + r) * ld + n + 4 * u), v);
  }
}

__device__ __forceinline__ void stage_row_bf16(uint8_t* stage, int lane, const float* v) {
  uint8_t* rowp = stage + lane * 64;
#pragma unroll
  for (int u = 0; u < 4; ++u)
    *reinterpret_cast<uint4*>(rowp + ((u ^ ((lane >> 1) & 3)) << 4)) = pack8_bf16(v + 8 * u);
}

__device__ __forceinline__ void copy_out_bf16(const uint8_t* stage, int lane, __nv_bfloat16* base,
                                              int64_t row0, int64_t ld, int n, int N,
                                              bool streaming = true) {
  const int u = lane & 3;
  if (n + 8 * u >= N) return;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + (lane >> 2);
    const uint4 v = *reinterpret_cast<const uint4*>(stage + r * 64 + ((u ^ ((r >> 1) & 3)) << 4));
    uint4* dst = reinterpret_cast<uint4*>(base + (row0 + r) * ld + n + 8 * u);
    if (streaming)
      __stcs(dst, v);
    else
      *dst = v;
  }
}

// GEMM1 + SwiGLU epilogue of one warp: 32 tile rows (quarter q) x one column half. Accumulator
// columns [0,128) are gate columns n0.., [128,256) up columns n0..; each 32-column chunk writes
// the fp32 gate, the fp32 up and w * silu(gate) * up (w: the row's routing weight) as a bf16 hi
// plane and, for a backward, its bf16 lo residual, all through the staging buffer (hi in its
// first 2 KB, lo in the second). The accumulator is released (`acce`) right after the last TMEM
// read, before the last stores. `fused`: the one-launch forward, whose GEMM2 tiles read the w*h
// hi rows back within the same launch, so those are stored without the streaming hint.
__device__ __forceinline__ void gemm1_epilogue_staged(const Args& a, const EpiGeom& eg,
                                                      uint32_t tacc, int lane, uint8_t* stage,
                                                      uint32_t acce, bool acce_remote = false,
                                                      bool fused = false) {
  const int64_t row0 = eg.row0;
  float* gu = reinterpret_cast<float*>(a.out0);
  const float w = __ldg(a.w_row + row0 + lane);
#pragma unroll 1
  for (int c = 0; c < eg.nch; ++c) {
    uint32_t ga[32], ub[32];
    tmem_ld_32x32(tacc + eg.tcol0 + c * 32, ga);
    tmem_ld_32x32(tacc + eg.tcol0 + eg.up_off + c * 32, ub);
    tmem_ld_wait();
    if (c == eg.nch - 1) {  // last TMEM read of this warp for the tile
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (acce_remote)  // the odd CTA of a pair MMA: the even CTA's barrier
          mbar_arrive_remote_relaxed(acce);
        else
          mbar_arrive(acce);
      }
    }
    const int n = eg.ocol0 + c * 32;
    float g[32], u[32], h[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      g[j] = __uint_as_float(ga[j]);
      u[j] = __uint_as_float(ub[j]);
      h[j] = w * (g[j] * sigmoidf_(g[j]) * u[j]);
    }
    if (!a.skip_gu) {  // gate|up and the lo plane of w*h are kept only for a backward
      stage_row_f32(stage, lane, g);
      __syncwarp();
      copy_out_f32(stage, lane, gu, row0, a.ld0, n, a.I);
      __syncwarp();
      stage_row_f32(stage, lane, u);
      __syncwarp();
      copy_out_f32(stage, lane, gu + a.I, row0, a.ld0, n, a.I);
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 32; ++j) g[j] = h[j] - __bfloat162float(__float2bfloat16_rn(h[j]));
      stage_row_bf16(stage + 2048, lane, g);
    }
    stage_row_bf16(stage, lane, h);
    __syncwarp();
    // the one-launch forward's GEMM2 tiles read the w*h rows back soon: normal stores there
    copy_out_bf16(stage, lane, a.out1, row0, a.ld1, n, a.I, !fused);
    if (!a.skip_gu) copy_out_bf16(stage + 2048, lane, a.out3, row0, a.ld1, n, a.I);
    __syncwarp();
  }
}

// SwiGLU backward of one 16-column chunk of one row: g from TMEM, gate (cur[0..3]) and up
// (cur[4..7]) from the staged fp32 values. Writes this row of the four output planes (d_gate,
// d_up; hi and lo each) into the warp's staging planes (32 rows x 32 bytes, 32-byte swizzle:
// 16-byte half h of row r sits at half h ^ ((r >> 2) & 1)) and accumulates <g, h>.
__device__ __forceinline__ void act_grad_chunk(uint32_t taddr, const float4 (&cur)[8], float w,
                                               float& p, uint8_t* out_row, int lane) {
  uint32_t v[16];
  tmem_ld_32x16(taddr, v);
  tmem_ld_wait();
  const int swz = (lane >> 2) & 1;
#pragma unroll
  for (int g8 = 0; g8 < 2; ++g8) {
    const float4 a0 = cur[2 * g8], a1 = cur[2 * g8 + 1];
    const float4 b0 = cur[4 + 2 * g8], b1 = cur[4 + 2 * g8 + 1];
    const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    float da[8], db[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float ga = av[j], ub = bv[j];
      const float gv = __uint_as_float(v[8 * g8 + j]);
      const float sg = sigmoidf_(ga);
      const float sl = ga * sg;
      const float h = sl * ub;
      p += gv * h;  // columns past I carry ga = ub = 0, so h = 0
      const float dh = w * gv;
      da[j] = dh * ub * sg * (1.0f + ga * (1.0f - sg));
      db[j] = dh * sl;
    }
    uint8_t* o = out_row + ((g8 ^ swz) << 4);
    uint4 hi, lo;
    split8_bf16(da, hi, lo);
    *reinterpret_cast<uint4*>(o + 0 * OUT_PLANE_BYTES) = hi;
    *reinterpret_cast<uint4*>(o + 2 * OUT_PLANE_BYTES) = lo;
    split8_bf16(db, hi, lo);
    *reinterpret_cast<uint4*>(o + 1 * OUT_PLANE_BYTES) = hi;
    *reinterpret_cast<uint4*>(o + 3 * OUT_PLANE_BYTES) = lo;
  }
}

// act_grad epilogue of one warp: g = dy_slot W_down^T (from TMEM) and the SwiGLU backward.
// The warp streams the (tile, 16-column chunk) pairs of its 32 rows and column half. Input:
// lane 0 TMA-loads the fp32 gate and up values of a chunk (two 32x16 boxes, 64-byte swizzle)
// into one of the warp's GU_BUFS staging buffers (chunk i in buffer i % GU_BUFS, on that
// buffer's barrier), GU_BUFS chunks ahead, and refills a buffer as soon as the warp has read it.
// Output: the warp writes the chunk's four 32x16 bf16 planes to its output staging buffer and
// lane 0 stores them with TMA (the tensor maps clip columns past I).
// PAIR = 2: the tiles are the CTA's halves of CTA-pair MMA tiles (units first, first + step, ..;
// this CTA is `rank` of its pair); a half past the expert is consumed but stores nothing.
template <int PAIR, int GU_BUFS>
__device__ __forceinline__ void act_grad_epilogue(const Args& a, const CUtensorMap* tm_gu,
                                                  const EpiMaps* em, int total, uint32_t tmem_base,
                                                  uint32_t accf0, uint32_t accf1, uint32_t acce0,
                                                  uint32_t acce1, uint32_t gbar, uint32_t gbuf,
                                                  const uint8_t* gbuf_ptr, uint32_t obuf,
                                                  uint8_t* obuf_ptr, int warp, int lane, int first,
                                                  int step, uint32_t rank) {
  constexpr int KIND = GK_ACT_GRAD;
  auto tile_at = [&](int unit, bool& valid) -> Tile {
    if constexpr (PAIR == 2) {
      return decode_pair<KIND>(a, unit, rank, valid);
    } else {
      valid = true;
      return decode_tile<KIND>(a, unit);
    }
  };
  constexpr int NC = BN / 32;      // 16-column chunks per column half
  const int q = warp & 3;          // TMEM lane quarter = rows 32q..32q+31 of the tile
  const int hf = (warp - 2) >> 2;  // column half
  const int c0 = hf * NC;
  const uint64_t tmo = a.timeout_ns;
  auto chunk_end = [&](int n0) {   // chunks entirely past I are skipped
    int ce = c0 + NC;
    while (ce > c0 && n0 + (ce - 1) * 16 >= a.I) --ce;
    return ce;
  };
  static_assert(GU_BUFS == 1 || GU_BUFS == 2, "gate|up staging depth");
  int ld_tile = first, ld_c = c0;  // next (unit, chunk) to load
  uint32_t issued = 0;             // chunks loaded so far (the next goes to buffer issued % GU_BUFS)
  // ld_tile decoded once per unit (decoding it for every chunk put the table reads' latency
  // in front of each chunk's load)
  bool ld_v;
  Tile tn{};
  if (first < total) tn = tile_at(first, ld_v);
  auto issue_next = [&]() {
    while (ld_tile < total && ld_c >= chunk_end(tn.n0)) {
      ld_tile += step;
      ld_c = c0;
      if (ld_tile < total) tn = tile_at(ld_tile, ld_v);
    }
    if (ld_tile >= total) return;
    if (lane == 0) {
      const uint32_t b = issued % GU_BUFS;
      const uint32_t bar = gbar + 8u * b, dst = gbuf + b * GU_CHUNK_BYTES;
      fence_proxy_async_smem();  // the buffer's previous contents were read by the warp
      mbar_arrive_expect_tx(bar, GU_CHUNK_BYTES);
      tma_load_2d(dst, tm_gu, bar, tn.n0 + ld_c * 16, tn.m0 + q * 32);
      tma_load_2d(dst + GU_CHUNK_BYTES / 2, tm_gu, bar, a.I + tn.n0 + ld_c * 16, tn.m0 + q * 32);
    }
    ++issued;
    ++ld_c;
  };
#pragma unroll
  for (int b = 0; b < GU_BUFS; ++b) issue_next();
  uint32_t acc_it = 0, used = 0;
  bool failed = false;
  uint8_t* out_row = obuf_ptr + lane * 32;
  TraceSpan ep_sp{0u, 0ull};  // the first epilogue warp's span on each accumulator
  bool ep_open = false;
  int ep_unit = 0;
  auto ep_close = [&]() {
    if (ep_open && lane == 0) trace_end(a.trace, ep_sp, MM_TRACE_EPILOGUE, ep_unit, rank);
    ep_open = false;
  };
  for (int tile = first; tile < total; tile += step) {
    ep_close();
    bool tile_ok;
    const Tile t = tile_at(tile, tile_ok);
    const uint32_t buf = acc_it & 1u, aph = (acc_it >> 1) & 1u;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(buf ? accf1 : accf0, aph, tmo) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) set_status(a.status, MM_ERR_TIMEOUT);
      break;
    }
    __syncwarp();
    tc_fence_after();
    if (warp == 2 && a.trace.buf != nullptr) {
      if (lane == 0) ep_sp = trace_begin(a.trace);
      ep_open = true;
      ep_unit = tile;
    }
    const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN;
    const int row0 = t.m0 + q * 32;
    const int64_t row = (int64_t)row0 + lane;
    const float w = __ldg(a.w_row + row);
    float p = 0.f;
    const int c_end = chunk_end(t.n0);
    for (int c = c0; c < c_end; ++c) {
      const uint32_t gb = used % GU_BUFS;
      int okg = 1;
      if (lane == 0) okg = mbar_wait(gbar + 8u * gb, (used / GU_BUFS) & 1u, tmo) ? 1 : 0;
      okg = __shfl_sync(0xffffffffu, okg, 0);
      if (!okg) {
        if (lane == 0) set_status(a.status, MM_ERR_TIMEOUT);
        failed = true;
        break;
      }
      __syncwarp();
      // row `lane` of the two 32x16 fp32 boxes; with the 64-byte swizzle the 16-byte unit u of
      // row r sits at unit u ^ ((r >> 1) & 3)
      const uint8_t* base = gbuf_ptr + gb * GU_CHUNK_BYTES + lane * 64;
      const int n = t.n0 + c * 16;
      float4 cur[8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int pu = (u ^ ((lane >> 1) & 3)) * 16;
        const bool in = n + 4 * u < a.I;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        cur[u] = in ? *reinterpret_cast<const float4*>(base + pu) : z;
        cur[4 + u] = in ? *reinterpret_cast<const float4*>(base + GU_CHUNK_BYTES / 2 + pu) : z;
      }
      ++used;
      __syncwarp();
      issue_next();  // this staging buffer is free again: start the load GU_BUFS chunks ahead
      if (!tile_ok) continue;  // a pair half past the expert: nothing to compute or store
      // the previous chunk's stores must have finished reading the output staging buffer
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
      act_grad_chunk(tacc + c * 16, cur, w, p, out_row, lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&em->dgu_hi, obuf + 0 * OUT_PLANE_BYTES, n, 0, row0);
        tma_store_3d(&em->dgu_hi, obuf + 1 * OUT_PLANE_BYTES, n, 1, row0);
        tma_store_3d(&em->dgu_lo, obuf + 2 * OUT_PLANE_BYTES, n, 0, row0);
        tma_store_3d(&em->dgu_lo, obuf + 3 * OUT_PLANE_BYTES, n, 1, row0);
        bulk_commit();
      }
    }
    if (failed) break;
    // one partial per (column tile, half), summed in a fixed order by W2Grad's epilogue warps
    // (epilogue_d_topk) or the d_topk kernel
    if (tile_ok) a.p_part[(int64_t)(2 * (t.n0 / BN) + hf) * a.S_pad + row] = p;
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (PAIR == 2 && rank != 0)  // the odd CTA of a pair MMA: the even CTA's barrier
        mbar_arrive_remote_relaxed(mapa_shared(buf ? acce1 : acce0, 0));
      else
        mbar_arrive(buf ? acce1 : acce0);
    }
    ++acc_it;
  }
  ep_close();
  if (lane == 0) bulk_wait_all();  // this warp's output stores are complete before it exits
  __syncwarp();
}

// d_topk_weights[s] = the sum, in column-tile order, of act_grad's <g, h> partials of slot s's
// row (the separate d_topk kernel's arithmetic, bit for bit). Run by the epilogue warps of the
// W2Grad launch, the first after act_grad, before they wait for their first accumulator: the
// partials are complete (the launch waited for act_grad) and the wait is otherwise idle time.
// `et` is the thread's index among the CTA's epilogue threads; slots are spread over the grid.
__device__ __forceinline__ void epilogue_d_topk(const Args& a, int et) {
  constexpr int ET = NUM_EPI_WARPS * 32;
  const int nt = a.d_topk_tiles;
  for (int s = (int)blockIdx.x * ET + et; s < a.d_topk_S; s += (int)gridDim.x * ET) {
    const int64_t r = __ldg(a.row_of_slot_d + s);
    float acc = 0.f;
    for (int j0 = 0; j0 < nt; j0 += 8) {  // eight loads in flight, then the sum in tile order
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = j0 + u < nt ? a.p_part[(int64_t)(j0 + u) * a.S_pad + r] : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (j0 + u < nt) acc += v[u];
    }
    a.d_topk[s] = acc;
  }
}

// Output epilogue of one warp for the kinds with a TMA-stored output (GEMM2, INPUT_GRAD, the
// weight gradients): 32 tile rows (quarter q) x one column half, in 32-column chunks. Each chunk
// is converted, written to the warp's staging buffers and stored (or, for accumulated weight
// gradients, reduce-added) with TMA by lane 0; the tensor map clips rows and columns outside the
// output.
//  * bf16 (default): 32 x 32 bf16 (64-byte rows, 64-byte swizzle: 16-byte unit u of row r at
//    u ^ ((r >> 1) & 3)), alternating between the warp's two 2 KB buffers; before a buffer is
//    rewritten, the store that used it two chunks earlier must have finished reading it
//    (`chunk_no` counts the warp's chunks).
//  * a.split_out (GEMM2 / INPUT_GRAD): bf16 hi in buffer 0 and the residual lo in buffer 1, stored
//    through map[0] and map[1].
//  * a.wgrad_f32 (weight gradients): 32 x 32 fp32 (128-byte rows, 128-byte swizzle: unit u of
//    row r at u ^ (r & 7)) across both buffers.
// W1Grad's accumulator holds dW_up^T (rows = columns of dW_up): its chunks are written to the
// staging buffer transposed (lane = output column, value j = output row) and stored at the
// swapped coordinates. `zero` stores zeros without reading TMEM (an expert with no rows).
// PART (weight gradients): the tile of a split expert's row chunk goes in fp32 to its partial
// slice t.slot through `map` (the partial slices' map: the output's layout, the slice as the
// third coordinate), never added in; the reduce kernel sums the slices into the output. Each
// instantiation stores through the one map it is given (no choice between maps at run time).
template <int KIND, bool PART = false>
__device__ __forceinline__ void staged_store_tile(const Args& a, const Tile& t,
                                                  const EpiGeom& eg, uint32_t tacc, int lane,
                                                  const CUtensorMap* map, uint32_t sbuf,
                                                  uint8_t* sbuf_ptr, uint32_t& chunk_no,
                                                  bool zero = false) {
  using TR = Traits<KIND>;
  static_assert(!PART || TR::WGRAD, "partial slices are weight-gradient tiles");
  const int row0 = eg.row0;
  const bool f32 = TR::WGRAD && (PART || a.wgrad_f32);
  const bool split = !TR::WGRAD && a.split_out;
#pragma unroll 1
  for (int c = 0; c < eg.nch; ++c) {
    uint32_t v[32];
    if (zero) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0u;
    } else {
      tmem_ld_32x32(tacc + eg.tcol0 + c * 32, v);
      tmem_ld_wait();
    }
    // both buffers for the fp32 and split forms, else the one used two chunks ago
    const uint32_t b = (f32 || split) ? 0u : (chunk_no & 1u);
    if (lane == 0) {
      if (f32 || split)
        bulk_wait_read_all();
      else
        bulk_wait_read_le1();
    }
    __syncwarp();
    uint8_t* buf = sbuf_ptr + b * OUT_TILE_BYTES;
    if constexpr (TR::TRANSPOSED_OUT) {
      if (f32) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          *reinterpret_cast<uint32_t*>(buf + j * 128 + (((lane >> 2) ^ (j & 7)) << 4) +
                                       (lane & 3) * 4) = v[j];
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          *reinterpret_cast<__nv_bfloat16*>(buf + j * 64 + (((lane >> 3) ^ ((j >> 1) & 3)) << 4) +
                                            (lane & 7) * 2) =
              __float2bfloat16_rn(__uint_as_float(v[j]));
      }
    } else if (f32) {
      uint8_t* rowp = buf + lane * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<uint4*>(rowp + ((u ^ (lane & 7)) << 4)) =
            make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
    } else {
      uint8_t* rowp = buf + lane * 64;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float f[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = __uint_as_float(v[8 * u + j]);
        const int off = (u ^ ((lane >> 1) & 3)) << 4;
        if (split) {
          uint4 hi, lo;
          split8_bf16(f, hi, lo);
          *reinterpret_cast<uint4*>(rowp + off) = hi;
          *reinterpret_cast<uint4*>(rowp + OUT_TILE_BYTES + off) = lo;
        } else {
          *reinterpret_cast<uint4*>(rowp + off) = pack8_bf16(f);
        }
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      const int n = eg.ocol0 + c * 32;
      const uint32_t src = sbuf + b * OUT_TILE_BYTES;
      if constexpr (TR::WGRAD) {
        const int x = TR::TRANSPOSED_OUT ? row0 : n, y = TR::TRANSPOSED_OUT ? n : row0;
        if (PART)
          tma_store_3d(map, src, x, y, t.slot);
        else if (a.accumulate)
          tma_reduce_add_3d(map, src, x, y, t.e);
        else
          tma_store_3d(map, src, x, y, t.e);
      } else {
        tma_store_2d(map, src, n, row0);
        if (split) tma_store_2d(map + 1, src + OUT_TILE_BYTES, n, row0);
      }
      bulk_commit();
    }
    ++chunk_no;
  }
  // A bf16 tile may come next in this warp, and its chunks wait only for the store before last
  // (one buffer each); the fp32 partial stores read both buffers, so they must be done reading.
  if constexpr (PART) {
    if (!a.wgrad_f32 && lane == 0) bulk_wait_read_all();
  }
}

// Combine fused into GEMM2's epilogue, for one warp's 32 rows x 128 columns (chunk j of H)
// after its o stores: the warp waits for them to complete, makes them visible device-wide, and
// counts each real row's token once for chunk j. The lane that brings a token's count to K holds
// its last slot; the warp then sums that token's K rows of chunk j in slot order (fp32, weights,
// then the optional extra rows) and stores y, with the separate combine kernel's arithmetic.
__device__ __forceinline__ void fused_combine_warp(const Args& a, const Tile& t, int q, int hf,
                                                   int lane) {
  if (lane == 0) bulk_wait_all();
  __syncwarp();
  fence_proxy_async_global();
  __threadfence();
  const int j = (t.n0 >> 7) + hf;  // 128-column chunk
  if (j >= a.comb_nch) return;     // this column half lies past H
  const int K = a.comb_K, H = a.comb_H;
  const int s = __ldg(a.slot_of_row + t.m0 + q * 32 + lane);
  int tok = -1;
  bool last = false;
  if (s >= 0) {
    tok = s / K;
    last = atomicAdd(a.cnt + (size_t)tok * a.comb_nch + j, 1) == K - 1;
  }
  unsigned m = __ballot_sync(0xffffffffu, last);
  if (m == 0) return;
  __threadfence();  // the other slots' rows, counted before ours, are visible
  const int col = j * 128 + lane * 4;
  while (m) {
    const int src = __ffs(m) - 1;
    m &= m - 1;
    const int tk = __shfl_sync(0xffffffffu, tok, src);
    if (col < H) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int k0 = 0; k0 < K; k0 += 8) {  // eight slots' loads in flight at a time
        uint2 v[8];
        float wk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (k0 + k < K) {
            const size_t sk = (size_t)tk * K + k0 + k;
            wk[k] = a.comb_w ? __ldg(a.comb_w + sk) : 1.0f;
            v[k] = __ldcg(reinterpret_cast<const uint2*>(
                a.comb_o + (size_t)__ldg(a.row_of_slot + sk) * H + col));
          }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (k0 + k < K) {
            acc[0] += wk[k] * bf16_lo(v[k].x);
            acc[1] += wk[k] * bf16_hi(v[k].x);
            acc[2] += wk[k] * bf16_lo(v[k].y);
            acc[3] += wk[k] * bf16_hi(v[k].y);
          }
        }
      }
      const __nv_bfloat16* ex[2] = {a.comb_extra, a.comb_extra_lo};
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (ex[x] != nullptr) {
          const uint2 e = __ldg(reinterpret_cast<const uint2*>(ex[x] + (size_t)tk * H + col));
          acc[0] += 1.0f * bf16_lo(e.x);
          acc[1] += 1.0f * bf16_hi(e.x);
          acc[2] += 1.0f * bf16_lo(e.y);
          acc[3] += 1.0f * bf16_hi(e.y);
        }
      }
      *reinterpret_cast<uint2*>(a.comb_y + (size_t)tk * H + col) =
          make_uint2(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]));
    }
  }
}


// PAIR: 0 = one CTA per tile; 2 = clusters of two CTAs sharing one M = 256 MMA (tcgen05
// .cta_group::2): each CTA holds its 128 rows of A and half of B's columns, the even CTA issues
// the MMAs, each CTA's tensor memory receives its own 128 accumulator rows.
template <int KIND, int PAIR = 0>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
           const __grid_constant__ CUtensorMap tmL, const __grid_constant__ EpiMaps em,
           const Args a) {
  using TR = Traits<KIND>;
  static_assert(PAIR == 0 || PAIR == 2, "one CTA per tile, or CTA-pair MMAs");
  constexpr bool PAIRED = PAIR == 2;
  constexpr bool MMA2 = PAIRED;
  pdl_wait();  // the stream's previous kernels are complete (see mm_device.cuh)
  const TraceCta trace_cta(a.trace, PAIRED ? cluster_ctarank() : 0u);
  static_assert(!PAIRED || KIND == GK_GEMM1_SWIGLU || KIND == GK_GEMM2 || KIND == GK_INPUT_GRAD ||
                    TR::WGRAD || KIND == GK_ACT_GRAD || TR::FUSED,
                "pair MMAs: GEMM1, GEMM2, the fused forward, act_grad, input_grad and the weight "
                "gradients");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if constexpr (KIND == GK_ACT_GRAD) {
    // the forward on this workspace kept no gate|up (forward-only): no backward from it
    if (__syncthreads_or(a.hdr[HDR_NO_BACKWARD] != 0)) {
      if (threadIdx.x == 0) set_status(a.status, MM_ERR_INVALID_ARG);
      return;
    }
  }
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  constexpr int STAGES = MMA2 ? TR::PAIR_STAGES : TR::STAGES;
  constexpr uint32_t PAIR_IDESC = idesc_bf16_f32(2 * BM, TR::TN, TR::A_MN ? 1 : 0, TR::B_MN ? 1 : 0);
  constexpr uint32_t PAIR_IDESC_HALF = idesc_bf16_f32(BM, TR::TN, TR::A_MN ? 1 : 0, TR::B_MN ? 1 : 0);
  constexpr uint32_t STAGE_BYTES = MMA2 ? TR::PAIR_STAGE_BYTES : TR::STAGE_BYTES;
  constexpr int GU_BUFS = MMA2 ? TR::PAIR_GU_BUFS : 1;  // act_grad gate|up buffers per warp
  const uint32_t epi_base = sbase + STAGES * STAGE_BYTES;  // act_grad gate|up staging
  const uint32_t bars = epi_base + (MMA2 ? TR::PAIR_EPI_BYTES : TR::EPI_BYTES);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (2 * STAGES + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (2 * STAGES + 2 + b); };
  auto gu_bar = [&](int ew) { return bars + 8u * (2 * STAGES + 4 + GU_BUFS * ew); };
  const uint32_t tmem_holder = bars + 8u * (2 * STAGES + 4 + GU_BUFS * NUM_EPI_WARPS);
  static_assert(8 * (2 * STAGES + 4 + GU_BUFS * NUM_EPI_WARPS) + 8 <= BAR_BYTES - 8,
                "barrier area");
  volatile uint32_t* tmem_holder_ptr =
      reinterpret_cast<volatile uint32_t*>(smem_raw + (tmem_holder - raw));

  // an earlier kernel of this call failed (a CTA-wide vote keeps the exit uniform); the status
  // word is the call's (the shared expert's launches point at the routed layout's word too).
  // The two CTAs of a pair take the same decision (two words at the end of the barrier area):
  // neither may leave while the other waits for it at a cluster barrier or in the pair's
  // tensor-memory allocation.
  int failed_before = __syncthreads_or(*a.status != 0);
  if constexpr (PAIRED) {
    const uint32_t flag = bars + BAR_BYTES - 8;
    volatile uint32_t* flag_ptr = reinterpret_cast<volatile uint32_t*>(smem_raw + (flag - raw));
    if (threadIdx.x == 0) flag_ptr[0] = (uint32_t)failed_before;
    cluster_sync();
    if (threadIdx.x == 0) flag_ptr[1] = ld_shared_cluster(mapa_shared(flag, cluster_ctarank() ^ 1u));
    cluster_sync();  // the peer has read this CTA's flag before either may leave
    failed_before = (int)(flag_ptr[0] | flag_ptr[1]);
  }
  if (failed_before) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = (PAIRED && TR::WGRAD)
                        ? a.hdr[HDR_WG_CHUNKS + a.wg_kind] * ((a.m_tiles_w + 1) / 2) * a.n_tiles_n
                    : (PAIRED && TR::FUSED) ? a.hdr[HDR_NUM_MPAIRS] * (a.n_tiles_n + a.n2)
                    : PAIRED                ? a.hdr[HDR_NUM_MPAIRS] * a.n_tiles_n
                    : TR::WGRAD ? a.hdr[HDR_WG_CHUNKS + a.wg_kind] * a.m_tiles_w * a.n_tiles_n
                    : TR::FUSED ? a.hdr[HDR_NUM_MTILES] * (a.n_tiles_n + a.n2)
                                : a.hdr[HDR_NUM_MTILES] * a.n_tiles_n;
  // work units of this CTA: tile (or pair) first, first + step, ...
  const uint32_t rank = PAIRED ? cluster_ctarank() : 0u;
  const int first = PAIRED ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int step = PAIRED ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  auto tile_at = [&](int unit, bool& valid) -> Tile {
    if constexpr (PAIRED) {
      return decode_pair<KIND>(a, unit, rank, valid);
    } else {
      valid = true;
      return decode_tile<KIND>(a, unit);
    }
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      // one arrival per epilogue warp (a pair MMA's even CTA: per epilogue warp of both CTAs)
      mbar_init(acce_bar(b), MMA2 ? 2 * NUM_EPI_WARPS : NUM_EPI_WARPS);
    }
    if constexpr (TR::GU_STAGING)
      for (int i = 0; i < GU_BUFS * NUM_EPI_WARPS; ++i) mbar_init(gu_bar(0) + 8u * i, 1);
    mbar_fence_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if constexpr (TR::A_SPLIT || TR::GU_STAGING) tma_prefetch_desc(&tmL);
    if constexpr (TR::OUT_STAGING) tma_prefetch_desc(&em.out);
    if constexpr (TR::WGRAD) tma_prefetch_desc(&em.part);
    if constexpr (TR::FUSED) {
      tma_prefetch_desc(&em.a2);
      tma_prefetch_desc(&em.b2);
    }
    if constexpr (TR::GU_STAGING) {
      tma_prefetch_desc(&em.dgu_hi);
      tma_prefetch_desc(&em.dgu_lo);
    }
  }
  if (warp == 1) {
    if constexpr (MMA2) {
      tmem_alloc_pair(tmem_holder, TR::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_holder, TR::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // paired: both CTAs' barriers are initialised before either signals the other's
  if constexpr (PAIRED) cluster_sync();
  const uint32_t tmem_base = *tmem_holder_ptr;
  const uint64_t tmo = a.timeout_ns;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int tile = first; tile < total && ok; tile += step) {
        bool tile_ok;
        const Tile t = tile_at(tile, tile_ok);
        if constexpr (TR::FUSED) {
          // a GEMM2 tile waits until every GEMM1 tile of its row block has stored its w*h rows
          // (each of their epilogue warps counts once), then orders those generic-proxy writes
          // before its TMA reads (a pair's half past the expert computes rows nobody stores)
          if (t.part == 1 && tile_ok) {
            if (!wait_counter(a.ready + t.m0 / BM, a.ready_target, tmo)) {
              set_status(a.status, MM_ERR_TIMEOUT);
              ok = false;
              break;
            }
            fence_proxy_async_global();
          }
        }
        for (int kb = 0; kb < t.kiters; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, tmo)) {
            set_status(a.status, MM_ERR_TIMEOUT);
            ok = false;
            break;
          }
          const uint32_t sa = sbase + s * STAGE_BYTES, sb = sa + TR::B_OFF;
          const int k0 = kb * BK;
          if constexpr (MMA2) {
            // both CTAs' bytes complete on the even CTA's barrier; only it posts their count
            // (an M = 128 unit: each CTA loads 64 rows of A)
            if (rank == 0)
              mbar_arrive_expect_tx(full_bar(s), 2 * (STAGE_BYTES - (t.half ? A_BYTES / 2 : 0)));
            const uint32_t fb = mapa_shared(full_bar(s), 0);
            if constexpr (TR::WGRAD) {  // this CTA's 128 rows of A (MN-major), hi and lo
              tma_load_2d_pair(sa, &tmA, fb, t.m0, t.row0 + k0);
              tma_load_2d_pair(sa + MN_BLOCK_BYTES, &tmA, fb, t.m0 + 64, t.row0 + k0);
              tma_load_2d_pair(sa + TR::A_LO_OFF, &tmL, fb, t.m0, t.row0 + k0);
              tma_load_2d_pair(sa + TR::A_LO_OFF + MN_BLOCK_BYTES, &tmL, fb, t.m0 + 64,
                               t.row0 + k0);
            } else if constexpr (TR::FUSED) {  // this CTA's 128 rows of A: x or w*h rows
              tma_load_2d_pair(sa, t.part ? &em.a2 : &tmA, fb, k0, t.m0);
            } else if (t.half) {  // this CTA's 64 rows of A (tmL: the same rows, 64-row boxes)
              tma_load_2d_pair(sa, &tmL, fb, k0, t.m0);
            } else {
              tma_load_2d_pair(sa, &tmA, fb, k0, t.m0);  // this CTA's 128 rows of A
            }
            // this CTA's half of B's columns (its MMA share), in its own shared memory
            if constexpr (TR::FUSED) {  // GEMM1: gate (rank 0) or up blocks; GEMM2: blocks 2r, 2r+1
              const int c0 = t.part ? t.n0 + 128 * (int)rank : (rank ? a.I : 0) + t.n0;
              const CUtensorMap* mb = t.part ? &em.b2 : &tmB;
              tma_load_3d_pair(sb, mb, fb, c0, k0, t.e);
              tma_load_3d_pair(sb + MN_BLOCK_BYTES, mb, fb, c0 + 64, k0, t.e);
            } else if constexpr (KIND == GK_GEMM1_SWIGLU) {
              if (t.half) {  // rank r: gate and up columns n0 + 64 r .. n0 + 64 r + 63
                tma_load_3d_pair(sb, &tmB, fb, t.n0 + 64 * (int)rank, k0, t.e);
                tma_load_3d_pair(sb + MN_BLOCK_BYTES, &tmB, fb, a.I + t.n0 + 64 * (int)rank, k0,
                                 t.e);
              } else {  // rank 0: the gate blocks, rank 1: up
                const int c0 = (rank ? a.I : 0) + t.n0;
                tma_load_3d_pair(sb, &tmB, fb, c0, k0, t.e);
                tma_load_3d_pair(sb + MN_BLOCK_BYTES, &tmB, fb, c0 + 64, k0, t.e);
              }
            } else if constexpr (KIND == GK_GEMM2) {  // rank r: column blocks 2r and 2r + 1
              const int c0 = t.n0 + 128 * (int)rank;
              tma_load_3d_pair(sb, &tmB, fb, c0, k0, t.e);
              tma_load_3d_pair(sb + MN_BLOCK_BYTES, &tmB, fb, c0 + 64, k0, t.e);
            } else if constexpr (TR::WGRAD) {  // rank r: column blocks 2r and 2r + 1 of the rows
              const int c0 = t.n0 + 128 * (int)rank;
              tma_load_2d_pair(sb, &tmB, fb, c0, t.row0 + k0);
              tma_load_2d_pair(sb + MN_BLOCK_BYTES, &tmB, fb, c0 + 64, t.row0 + k0);
            } else {  // INPUT_GRAD, ACT_GRAD, K-major B: rank r loads rows 128r..128r+127
              tma_load_3d_pair(sb, &tmB, fb, k0, t.n0 + B_HALF_ROWS * (int)rank, t.e);
            }
            continue;
          }
          mbar_arrive_expect_tx(full_bar(s), STAGE_BYTES);
          if constexpr (TR::A_MN) {
            tma_load_2d(sa, &tmA, full_bar(s), t.m0, t.row0 + k0);
            tma_load_2d(sa + MN_BLOCK_BYTES, &tmA, full_bar(s), t.m0 + 64, t.row0 + k0);
            if constexpr (TR::A_SPLIT) {
              tma_load_2d(sa + TR::A_LO_OFF, &tmL, full_bar(s), t.m0, t.row0 + k0);
              tma_load_2d(sa + TR::A_LO_OFF + MN_BLOCK_BYTES, &tmL, full_bar(s), t.m0 + 64,
                          t.row0 + k0);
            }
          } else if constexpr (TR::FUSED) {
            tma_load_2d(sa, t.part ? &em.a2 : &tmA, full_bar(s), k0, t.m0);
          } else {
            tma_load_2d(sa, &tmA, full_bar(s), k0, t.m0);
          }
          if constexpr (TR::FUSED) {
            if (t.part == 0) {
              tma_load_3d(sb + 0 * MN_BLOCK_BYTES, &tmB, full_bar(s), t.n0, k0, t.e);
              tma_load_3d(sb + 1 * MN_BLOCK_BYTES, &tmB, full_bar(s), t.n0 + 64, k0, t.e);
              tma_load_3d(sb + 2 * MN_BLOCK_BYTES, &tmB, full_bar(s), a.I + t.n0, k0, t.e);
              tma_load_3d(sb + 3 * MN_BLOCK_BYTES, &tmB, full_bar(s), a.I + t.n0 + 64, k0, t.e);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                tma_load_3d(sb + j * MN_BLOCK_BYTES, &em.b2, full_bar(s), t.n0 + 64 * j, k0, t.e);
            }
          } else if constexpr (KIND == GK_GEMM1_SWIGLU) {
            tma_load_3d(sb + 0 * MN_BLOCK_BYTES, &tmB, full_bar(s), t.n0, k0, t.e);
            tma_load_3d(sb + 1 * MN_BLOCK_BYTES, &tmB, full_bar(s), t.n0 + 64, k0, t.e);
            tma_load_3d(sb + 2 * MN_BLOCK_BYTES, &tmB, full_bar(s), a.I + t.n0, k0, t.e);
            tma_load_3d(sb + 3 * MN_BLOCK_BYTES, &tmB, full_bar(s), a.I + t.n0 + 64, k0, t.e);
          } else if constexpr (TR::GEMM2_LIKE) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_load_3d(sb + j * MN_BLOCK_BYTES, &tmB, full_bar(s), t.n0 + 64 * j, k0, t.e);
          } else if constexpr (KIND == GK_ACT_GRAD || KIND == GK_INPUT_GRAD) {
            tma_load_3d(sb, &tmB, full_bar(s), k0, t.n0, t.e);
          } else {
#pragma unroll
            for (int j = 0; j < TR::TN / 64; ++j)
              tma_load_2d(sb + j * MN_BLOCK_BYTES, &tmB, full_bar(s), t.n0 + 64 * j, t.row0 + k0);
          }
        }
      }
      if constexpr (PAIRED) {
        // both CTAs' releases of every stage's last use have landed on this CTA's barriers
        // before it may leave (the peer's MMA commits arrive here asynchronously)
        for (int s = 0; s < STAGES && ok; ++s) {
          if (it <= (uint32_t)s) break;
          const uint32_t last = (it - 1 - s) / STAGES;  // index of stage s's last use
          if (!mbar_wait(empty_bar(s), last & 1u, tmo)) set_status(a.status, MM_ERR_TIMEOUT);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && (!MMA2 || rank == 0)) {  // a pair MMA is issued by the even CTA alone
      uint32_t it = 0, acc_it = 0;
      bool ok = true;
      for (int tile = first; tile < total && ok; tile += step) {
        bool tile_ok;
        const Tile t = tile_at(tile, tile_ok);
        (void)tile_ok;
        if (t.kiters == 0) continue;
        const uint32_t buf = acc_it & 1u, aph = (acc_it >> 1) & 1u;
        if (!mbar_wait(acce_bar(buf), aph ^ 1u, tmo)) {
          set_status(a.status, MM_ERR_TIMEOUT);
          break;
        }
        tc_fence_after();
        const TraceSpan tsp = trace_begin(a.trace);
        const uint32_t d = tmem_base + buf * TR::TN;
        for (int kb = 0; kb < t.kiters; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait(full_bar(s), ph, tmo)) {
            set_status(a.status, MM_ERR_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = sbase + s * STAGE_BYTES, sb = sa + TR::B_OFF;
          const int nk = kb == t.kiters - 1 ? t.klast : BK / 16;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (kk >= nk) break;
            // k-step offsets: 16 elements = 32 B along a K-major row, 16 k-rows = 2 KB MN-major
            const uint32_t ka = TR::A_MN ? kk * 2048 : kk * 32;
            const uint32_t kbo = TR::B_MN ? kk * 2048 : kk * 32;
            const uint32_t lbo_a = TR::A_MN ? MN_BLOCK_BYTES : 16;
            const uint32_t lbo_b = TR::B_MN ? MN_BLOCK_BYTES : 16;
            const uint64_t ad = sdesc_sw128(sa + ka, lbo_a, 1024);
            const uint64_t bd = sdesc_sw128(sb + kbo, lbo_b, 1024);
            if constexpr (MMA2) {
              umma_bf16_pair(d, ad, bd, t.half ? PAIR_IDESC_HALF : PAIR_IDESC,
                             (kb | kk) != 0 ? 1u : 0u);
              if constexpr (TR::A_SPLIT)
                umma_bf16_pair(d, sdesc_sw128(sa + TR::A_LO_OFF + ka, lbo_a, 1024), bd, PAIR_IDESC,
                               1u);
            } else {
              umma_bf16(d, ad, bd, TR::IDESC, (kb | kk) != 0 ? 1u : 0u);
              if constexpr (TR::A_SPLIT)
                umma_bf16(d, sdesc_sw128(sa + TR::A_LO_OFF + ka, lbo_a, 1024), bd, TR::IDESC, 1u);
            }
          }
          if constexpr (MMA2)
            umma_commit_pair_mc(empty_bar(s), 0x3);  // both CTAs' producers refill this stage
          else
            umma_commit(empty_bar(s));
        }
        if (!ok) break;
        // (test hook: CTA 0 withholds its first hand-off, so its epilogue's wait runs out)
        if (!(a.inject_stall && blockIdx.x == 0 && acc_it == 0)) {
          if constexpr (MMA2)
            umma_commit_pair_mc(accf_bar(buf), 0x3);  // both CTAs' epilogues
          else
            umma_commit(accf_bar(buf));
        }
        trace_end(a.trace, tsp, MM_TRACE_MAINLOOP, tile, rank);
        ++acc_it;
      }
    }
  } else if constexpr (TR::GU_STAGING) {
    const int ew = warp - 2;
    const uint32_t gbuf = epi_base + ew * GU_BUFS * GU_CHUNK_BYTES;
    const uint32_t obuf =
        epi_base + NUM_EPI_WARPS * GU_BUFS * GU_CHUNK_BYTES + ew * OUT_CHUNK_BYTES;
    act_grad_epilogue<PAIR, GU_BUFS>(a, &tmL, &em, total, tmem_base, accf_bar(0), accf_bar(1),
                            acce_bar(0), acce_bar(1), gu_bar(ew), gbuf, smem_raw + (gbuf - raw),
                            obuf, smem_raw + (obuf - raw), warp, lane, first, step, rank);
  } else {
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int hf = (warp - 2) >> 2;  // column half of the tile
    const uint32_t sbuf = epi_base + (warp - 2) * 2 * OUT_TILE_BYTES;  // output staging
    uint32_t chunk_no = 0;
    // hands accumulator `b` back to the MMA issuer (for the odd CTA of a pair MMA: the even
    // CTA's barrier; its tensor-memory reads are complete, so the arrive orders nothing else)
    auto release_acc = [&](uint32_t b) {
      if (MMA2 && rank != 0)
        mbar_arrive_remote_relaxed(mapa_shared(acce_bar(b), 0));
      else
        mbar_arrive(acce_bar(b));
    };
    if constexpr (KIND == GK_W2_GRAD) {
      if (a.d_topk != nullptr) epilogue_d_topk(a, (warp - 2) * 32 + lane);
    }
    uint32_t acc_it = 0;
    // the first epilogue warp's span on each accumulator, closed when the warp moves on
    TraceSpan ep_sp{0u, 0ull};
    bool ep_open = false;
    int ep_unit = 0;
    auto ep_close = [&]() {
      if (ep_open && lane == 0) trace_end(a.trace, ep_sp, MM_TRACE_EPILOGUE, ep_unit, rank);
      ep_open = false;
    };
    for (int tile = first; tile < total; tile += step) {
      ep_close();
      bool tile_ok;
      const Tile t = tile_at(tile, tile_ok);
      if (t.kiters == 0) {
        if constexpr (TR::WGRAD) {
          if (!a.accumulate && tile_ok)  // adding zero changes nothing
            staged_store_tile<KIND>(a, t, epi_geom<false>(t, q, hf, TR::TN), 0u, lane, &em.out,
                                    sbuf, smem_raw + (sbuf - raw), chunk_no, true);
        }
        continue;
      }
      const uint32_t buf = acc_it & 1u, aph = (acc_it >> 1) & 1u;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(accf_bar(buf), aph, tmo) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) set_status(a.status, MM_ERR_TIMEOUT);
        break;
      }
      __syncwarp();
      tc_fence_after();
      if (warp == 2 && a.trace.buf != nullptr) {
        if (lane == 0) ep_sp = trace_begin(a.trace);
        ep_open = true;
        ep_unit = tile;
      }
      const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + buf * TR::TN;
      if (!tile_ok) {  // a pair's second tile outside the expert: nothing to store
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release_acc(buf);
        ++acc_it;
        continue;
      }
      if constexpr (TR::FUSED) {
        if (t.part == 0) {
          // the staging buffer may still be read by this warp's TMA stores of a GEMM2 tile
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
          gemm1_epilogue_staged(a, epi_geom<true>(t, q, hf, TR::TN), tacc, lane,
                                smem_raw + (sbuf - raw),
                                (MMA2 && rank != 0) ? mapa_shared(acce_bar(buf), 0) : acce_bar(buf),
                                MMA2 && rank != 0, true);
          // this warp's w*h (and gate|up) stores, ordered before the async proxy's later reads
          // by each lane, are released at GPU scope by one count from lane 0 (a full fence by
          // every lane instead cost this kernel ~3 %)
          fence_proxy_async_global();
          __syncwarp();
          if (lane == 0) red_add_release_gpu(a.ready + t.m0 / BM, 1);
        } else {
          staged_store_tile<GK_GEMM2>(a, t, epi_geom<false>(t, q, hf, TR::TN), tacc, lane,
                                      &em.out, sbuf, smem_raw + (sbuf - raw), chunk_no);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) release_acc(buf);
          if (a.fuse_combine) fused_combine_warp(a, t, q, hf, lane);
        }
        ++acc_it;
        continue;
      }
      if constexpr (TR::ROW_STAGING) {  // releases the accumulator itself
        gemm1_epilogue_staged(a, epi_geom<true>(t, q, hf, TR::TN), tacc, lane,
                              smem_raw + (sbuf - raw),
                              (MMA2 && rank != 0) ? mapa_shared(acce_bar(buf), 0) : acce_bar(buf),
                              MMA2 && rank != 0);
        ++acc_it;
        continue;
      }
      if constexpr (TR::WGRAD) {
        if (t.slot >= 0)  // a split expert's row chunk: its fp32 partial slice
          staged_store_tile<KIND, true>(a, t, epi_geom<false>(t, q, hf, TR::TN), tacc, lane,
                                        &em.part, sbuf, smem_raw + (sbuf - raw), chunk_no);
        else
          staged_store_tile<KIND>(a, t, epi_geom<false>(t, q, hf, TR::TN), tacc, lane, &em.out,
                                  sbuf, smem_raw + (sbuf - raw), chunk_no);
      } else if constexpr (TR::OUT_STAGING) {
        staged_store_tile<KIND>(a, t, epi_geom<false>(t, q, hf, TR::TN), tacc, lane, &em.out,
                                sbuf, smem_raw + (sbuf - raw), chunk_no);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) release_acc(buf);
      if constexpr (KIND == GK_GEMM2_COMBINE) fused_combine_warp(a, t, q, hf, lane);
      ++acc_it;
    }
    ep_close();
    if constexpr (TR::OUT_STAGING) {
      if (lane == 0) bulk_wait_all();  // this warp's output stores are complete
      __syncwarp();
    }
  }

  // this CTA's work is done: the next kernel may take its SM as soon as it leaves
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  // paired: the peer may still commit onto this CTA's barriers until it is done too
  if constexpr (PAIRED) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (MMA2)
      tmem_dealloc_pair(tmem_base, TR::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TR::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor map; dims/box innermost first; strides in bytes (rank-1). bf16 with the 128-byte
// swizzle unless stated.
bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box,
              CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn) {
    note_error("cuTensorMapEncodeTiled unavailable");
    return false;
  }
  cuuint64_t d[3], s[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides[i];
  const CUresult r = fn(m, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    note_error("tensor map encode failed (CUresult %d): rank %d dims %llu %llu %llu box %u %u %u",
               (int)r, rank, (unsigned long long)d[0], (unsigned long long)(rank > 1 ? d[1] : 0),
               (unsigned long long)(rank > 2 ? d[2] : 0), b[0], rank > 1 ? b[1] : 0u,
               rank > 2 ? b[2] : 0u);
  return r == CUDA_SUCCESS;
}

bool map_rows(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, uint32_t box_cols,
              uint32_t box_rows) {
  const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)cols * 2};
  const uint32_t box[2] = {box_cols, box_rows};
  return make_map(m, base, 2, dims, strides, box);
}

bool map_experts(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t E,
                 uint32_t box_cols, uint32_t box_rows) {
  const uint64_t dims[3] = {(uint64_t)cols, (uint64_t)rows, (uint64_t)E};
  const uint64_t strides[2] = {(uint64_t)cols * 2, (uint64_t)cols * rows * 2};
  const uint32_t box[3] = {box_cols, box_rows, 1};
  return make_map(m, base, 3, dims, strides, box);
}

// The per-device values below are cached in atomics: host threads may call concurrently, and
// a value computed twice is the same value.
int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Dynamic shared memory of a launch: the stage ring, the epilogue's buffers, alignment slack
// and the barriers.
template <int KIND, int PAIR>
constexpr size_t smem_bytes() {
  return PAIR == 2 ? Traits<KIND>::PAIR_SMEM : Traits<KIND>::SMEM;
}

template <int KIND, int PAIR>
cudaError_t set_smem_attr() {
  static std::atomic<uint64_t> done_mask{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done_mask.load(std::memory_order_relaxed) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(k_gemm<KIND, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem_bytes<KIND, PAIR>());
  if (e == cudaSuccess) done_mask.fetch_or(bit, std::memory_order_relaxed);
  return e;
}

inline int cdiv(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

template <int KIND, int PAIR = 0>
cudaError_t run(const Workspace& w, char* ws, const GemmCall& c, cudaStream_t st) {
  constexpr bool PAIRED = PAIR == 2;
  cudaError_t err = set_smem_attr<KIND, PAIR>();
  if (err != cudaSuccess) return err;
  const int nsm = sm_count();
  if (nsm <= 0) return cudaErrorNoDevice;
  const int64_t H = w.H, I = w.I, E = w.E, S_pad = w.S_pad;
  auto bf = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(ws + off); };

  Args a{};
  a.trace = trace_ctx();
  a.hdr = reinterpret_cast<const int*>(ws + w.off_hdr);
  a.status = c.status ? c.status : reinterpret_cast<int*>(ws + w.off_hdr) + HDR_STATUS;
  // token rows: the dispatched (expert-sorted) copies, or x / dy themselves for the shared
  // expert (T rows in token order; TMA zero-fills the pad rows past T)
  const void* xrows = c.rows ? c.rows : ws + w.off_x_slot;
  const void* dyrows = c.rows ? c.rows : ws + w.off_dy_slot;
  const int64_t nrows = c.rows ? w.T : S_pad;
  a.tile_expert = reinterpret_cast<const int32_t*>(ws + w.off_tile_expert);
  a.poff = reinterpret_cast<const int32_t*>(ws + w.off_poff);
  a.counts = reinterpret_cast<const int32_t*>(ws + w.off_counts);
  a.E = (int)E;
  a.I = (int)I;
  a.S_pad = S_pad;
  a.timeout_ns = c.timeout_ns;
  a.inject_stall = c.inject_stall;
  a.accumulate = c.accumulate;
  a.skip_gu = c.skip_gu;
  if (c.comb_y != nullptr) {  // GEMM2 (or the fused forward) with the combine in its epilogue
    a.fuse_combine = 1;
    a.cnt = reinterpret_cast<int*>(ws + w.off_cnt);
    a.slot_of_row = reinterpret_cast<const int32_t*>(ws + w.off_slot_of_row);
    a.row_of_slot = reinterpret_cast<const int32_t*>(ws + w.off_row_of_slot);
    a.comb_w = c.comb_w;
    a.comb_o = reinterpret_cast<const __nv_bfloat16*>(ws + w.off_o);
    a.comb_extra = reinterpret_cast<const __nv_bfloat16*>(c.comb_extra);
    a.comb_extra_lo = reinterpret_cast<const __nv_bfloat16*>(c.comb_extra_lo);
    a.comb_y = reinterpret_cast<__nv_bfloat16*>(c.comb_y);
    a.comb_K = (int)w.K;
    a.comb_H = (int)w.H;
    a.comb_nch = (int)((w.H + 127) / 128);
  }

  CUtensorMap ta, tb, tl;
  EpiMaps em;
  bool ok = true, has_lo = false, has_em = false;
  int64_t tiles_max = 0;
  const int64_t m_tiles_max = S_pad / BM;
  switch (KIND) {
    case GK_GEMM1_SWIGLU:
      ok = map_rows(&ta, xrows, H, nrows, 64, BM) &&
           map_experts(&tb, c.w_up, 2 * I, H, E, 64, 64) &&
           (!PAIRED || map_rows(&tl, xrows, H, nrows, 64, BM / 2));  // the M = 128 units' A
      has_lo = PAIRED;
      a.n_tiles_n = cdiv(I, BN / 2);
      a.k_iters = cdiv(H, BK);
      a.N = (int)I;
      a.out0 = ws + w.off_gu;  // fp32
      a.ld0 = 2 * I;
      a.out1 = bf(w.off_h);  // w*h, hi
      a.out3 = bf(w.off_hw_lo);  // w*h, lo
      a.ld1 = I;
      a.w_row = reinterpret_cast<const float*>(ws + w.off_w_row);
      tiles_max = m_tiles_max * a.n_tiles_n;
      break;
    case GK_FWD_FUSED:
      ok = map_rows(&ta, xrows, H, nrows, 64, BM) &&
           map_experts(&tb, c.w_up, 2 * I, H, E, 64, 64) &&
           map_rows(&em.a2, ws + w.off_h, I, S_pad, 64, BM) &&
           map_experts(&em.b2, c.w_down, H, I, E, 64, 64);
      a.n_tiles_n = cdiv(I, BN / 2);
      a.k_iters = cdiv(H, BK);
      a.n2 = cdiv(H, BN);
      a.k2 = cdiv(I, BK);
      // GEMM1 windows of 128 row tiles (~5 waves of GEMM1 tiles; 64 pairs of row tiles for the
      // pair MMAs) between a row block's GEMM1 and GEMM2 tiles: with one CTA per tile, windows of
      // 8 or 32 row tiles, which interleave the two GEMMs more finely, were 27 % and 6 % slower
      // on a GB300; 128 and one window were equal to two launches
      a.win = PAIRED ? 64 : 128;
      a.ready = reinterpret_cast<int*>(ws + w.off_ready);
      a.ready_target = NUM_EPI_WARPS * a.n_tiles_n;
      a.N = (int)I;
      a.out0 = ws + w.off_gu;  // fp32
      a.ld0 = 2 * I;
      a.out1 = bf(w.off_h);  // w*h, hi
      a.out3 = bf(w.off_hw_lo);  // w*h, lo
      a.ld1 = I;
      a.w_row = reinterpret_cast<const float*>(ws + w.off_w_row);
      tiles_max = m_tiles_max * (a.n_tiles_n + a.n2);
      break;
    case GK_GEMM2:
    case GK_GEMM2_COMBINE:
      ok = map_rows(&ta, ws + w.off_h, I, S_pad, 64, BM) &&
           map_experts(&tb, c.w_down, H, I, E, 64, 64);
      a.n_tiles_n = cdiv(H, BN);
      a.k_iters = cdiv(I, BK);
      a.N = (int)H;
      a.out0 = bf(w.off_o);
      a.out1 = bf(w.off_o_lo);
      a.ld0 = H;
      tiles_max = m_tiles_max * a.n_tiles_n;
      break;
    case GK_ACT_GRAD: {
      // fp32 gate|up rows for the epilogue: boxes of 32 rows x 16 columns, 64-byte swizzle
      const uint64_t gdims[2] = {(uint64_t)(2 * I), (uint64_t)S_pad};
      const uint64_t gstr[1] = {(uint64_t)(2 * I) * 4};
      const uint32_t gbox[2] = {16, 32};
      ok = map_rows(&ta, dyrows, H, nrows, 64, BM) &&
           map_experts(&tb, c.w_down, H, I, E, 64, PAIRED ? B_HALF_ROWS : BN) &&
           make_map(&tl, ws + w.off_gu, 2, gdims, gstr, gbox, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                    CU_TENSOR_MAP_SWIZZLE_64B);
      // output planes, stored in boxes of 32 rows x 16 columns with the 32-byte swizzle
      const uint64_t d3[3] = {(uint64_t)I, 2, (uint64_t)S_pad};
      const uint64_t s3[2] = {(uint64_t)I * 2, (uint64_t)(2 * I) * 2};
      const uint32_t b3[3] = {16, 1, 32};
      const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
      const auto SW = CU_TENSOR_MAP_SWIZZLE_32B;
      ok = ok && make_map(&em.dgu_hi, ws + w.off_dgu, 3, d3, s3, b3, BF, SW) &&
           make_map(&em.dgu_lo, ws + w.off_dgu_lo, 3, d3, s3, b3, BF, SW);
      has_lo = true;
      has_em = true;
      a.n_tiles_n = cdiv(I, BN);
      a.k_iters = cdiv(H, BK);
      a.N = (int)I;
      a.out0 = bf(w.off_dgu);
      a.out2 = bf(w.off_dgu_lo);
      a.ld0 = 2 * I;
      a.gu = reinterpret_cast<const float*>(ws + w.off_gu);
      a.ld_gu = 2 * I;
      a.w_row = reinterpret_cast<const float*>(ws + w.off_w_row);
      a.p_part = reinterpret_cast<float*>(ws + w.off_p_part);
      tiles_max = m_tiles_max * a.n_tiles_n;
      break;
    }
    case GK_INPUT_GRAD:  // paired: each CTA loads half of B's rows
      ok = map_rows(&ta, ws + w.off_dgu, 2 * I, S_pad, 64, BM) &&
           map_experts(&tb, c.w_up, 2 * I, H, E, 64, PAIRED ? B_HALF_ROWS : BN);
      a.n_tiles_n = cdiv(H, BN);
      a.k_iters = cdiv(2 * I, BK);
      a.N = (int)H;
      a.out0 = bf(w.off_o);  // dx_slot reuses the forward's o buffer
      a.out1 = bf(w.off_o_lo);
      a.ld0 = H;
      tiles_max = m_tiles_max * a.n_tiles_n;
      break;
    case GK_W2_GRAD:
      ok = map_rows(&ta, ws + w.off_h, I, S_pad, 64, 64) &&
           map_rows(&tl, ws + w.off_hw_lo, I, S_pad, 64, 64) &&
           map_rows(&tb, dyrows, H, nrows, 64, 64);
      has_lo = true;
      a.m_tiles_w = cdiv(I, BM);
      a.n_tiles_n = cdiv(H, Traits<GK_W2_GRAD>::TN);
      a.M = (int)I;
      a.N = (int)H;
      a.out0 = reinterpret_cast<__nv_bfloat16*>(c.d_w);
      a.ld0 = H;
      a.out_expert_stride = I * H;
      a.wg_kind = WG_W2;
      tiles_max = (E + w.wg_slices[WG_W2]) * a.m_tiles_w * a.n_tiles_n;
      break;
    case GK_W1_GRAD:  // accumulates dW_up^T: rows = the 2I columns of dW_up, columns = H
      ok = map_rows(&ta, ws + w.off_dgu, 2 * I, S_pad, 64, 64) &&
           map_rows(&tl, ws + w.off_dgu_lo, 2 * I, S_pad, 64, 64) &&
           map_rows(&tb, xrows, H, nrows, 64, 64);
      has_lo = true;
      a.m_tiles_w = cdiv(2 * I, BM);
      a.n_tiles_n = cdiv(H, Traits<GK_W1_GRAD>::TN);
      a.M = (int)(2 * I);
      a.N = (int)H;
      a.out0 = reinterpret_cast<__nv_bfloat16*>(c.d_w);
      a.ld0 = 2 * I;
      a.out_expert_stride = H * 2 * I;
      a.wg_kind = WG_W1;
      tiles_max = (E + w.wg_slices[WG_W1]) * a.m_tiles_w * a.n_tiles_n;
      break;
  }
  if (!ok) return cudaErrorInvalidValue;
  if (!has_lo) tl = ta;  // unused by the kinds without a lo plane or M = 128 units
  if (!has_em) em.dgu_hi = em.dgu_lo = ta;  // unused but initialised
  if constexpr (!Traits<KIND>::WGRAD) em.part = ta;                      // unused but initialised
  if constexpr (!Traits<KIND>::FUSED) em.a2 = em.b2 = ta;                // unused but initialised
  if constexpr (Traits<KIND>::OUT_STAGING) {
    // bf16 output in boxes of 32 rows x 32 columns, 64-byte swizzle
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto SW = CU_TENSOR_MAP_SWIZZLE_64B;
    if constexpr (Traits<KIND>::FUSED) {  // GEMM2's o rows [S_pad][H]
      const uint64_t d2[2] = {(uint64_t)H, (uint64_t)S_pad};
      const uint64_t s2[1] = {(uint64_t)H * 2};
      const uint32_t b2[2] = {32, 32};
      if (!make_map(&em.out, ws + w.off_o, 2, d2, s2, b2, BF, SW)) return cudaErrorInvalidValue;
      em.out_lo = em.out;  // unused but initialised
    } else if constexpr (Traits<KIND>::WGRAD) {  // [E][M][N] ([E][N][M] transposed), bf16 or fp32
      a.wgrad_f32 = c.wgrad_f32 ? 1 : 0;
      const uint64_t es = a.wgrad_f32 ? 4 : 2;
      const bool tr = Traits<KIND>::TRANSPOSED_OUT;
      const uint64_t d3[3] = {(uint64_t)(tr ? a.M : a.N), (uint64_t)(tr ? a.N : a.M), (uint64_t)E};
      const uint64_t s3[2] = {(uint64_t)a.ld0 * es, (uint64_t)a.out_expert_stride * es};
      const uint32_t b3[3] = {32, 32, 1};
      if (!make_map(&em.out, a.out0, 3, d3, s3, b3,
                    a.wgrad_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : BF,
                    a.wgrad_f32 ? CU_TENSOR_MAP_SWIZZLE_128B : SW))
        return cudaErrorInvalidValue;
      em.out_lo = em.out;  // unused but initialised
      // the row chunks of this kind's plan, and the fp32 partial slices of split experts: the
      // output's layout with the slice as the third coordinate, in the o / dx row buffer
      // (W2Grad) or the dy row buffer (W1Grad), which are free while these kernels run
      const int k = a.wg_kind;
      a.wg_plan = reinterpret_cast<const int4*>(ws + w.off_wg_plan) + k * (E + w.wg_slices_max);
      const size_t part_off = (k == WG_W1 && w.wg_slices[WG_W1] > 0) ? w.off_dy_slot : w.off_o;
      const uint64_t dp[3] = {d3[0], d3[1], (uint64_t)std::max<int64_t>(1, w.wg_slices[k])};
      const uint64_t sp[2] = {(uint64_t)a.ld0 * 4, (uint64_t)a.out_expert_stride * 4};
      if (!make_map(&em.part, ws + part_off, 3, dp, sp, b3, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                    CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    } else {  // [S_pad][N]
      const uint64_t d2[2] = {(uint64_t)a.N, (uint64_t)S_pad};
      const uint64_t s2[1] = {(uint64_t)a.ld0 * 2};
      const uint32_t b2[2] = {32, 32};
      if (!make_map(&em.out, a.out0, 2, d2, s2, b2, BF, SW)) return cudaErrorInvalidValue;
      a.split_out = c.split_out ? 1 : 0;
      if (a.split_out) {
        if (w.off_o_lo == w.total) return cudaErrorInvalidValue;  // layout has no lo rows
        if (!make_map(&em.out_lo, a.out1, 2, d2, s2, b2, BF, SW)) return cudaErrorInvalidValue;
      } else {
        em.out_lo = em.out;  // unused but initialised
      }
    }
  } else {
    em.out = em.out_lo = ta;  // unused but initialised
  }
  // W2Grad takes over d_topk_weights when its grid has the threads for it (at most 8 slots per
  // epilogue thread, a few microseconds of loads before the first accumulator is due); otherwise
  // the caller launches the d_topk kernel
  auto take_d_topk = [&](int ctas) {
    if (KIND != GK_W2_GRAD || c.d_topk == nullptr || c.d_topk_taken == nullptr) return;
    if ((int64_t)ctas * NUM_EPI_WARPS * 32 * 8 < w.S) return;
    a.d_topk = c.d_topk;
    a.row_of_slot_d = reinterpret_cast<const int32_t*>(ws + w.off_row_of_slot);
    a.p_part = reinterpret_cast<float*>(ws + w.off_p_part);
    a.S_pad = S_pad;
    a.d_topk_S = (int)w.S;
    a.d_topk_tiles = (int)w.n_act_tiles;
    *c.d_topk_taken = true;
  };
  if constexpr (PAIRED) {
    // clusters of two CTAs over pairs of row tiles: as many clusters as fit at once (a
    // persistent grid must not wait for SMs), at most one per pair-column unit
    a.pair_tile = reinterpret_cast<const int32_t*>(ws + w.off_pair_tile);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem_bytes<KIND, PAIR>();
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)(nsm & ~1));
    // clusters that fit at once, queried once per device (a launch inside a stream capture then
    // makes no query)
    static std::atomic<int> max_clusters_of[64];
    int dev = 0;
    err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int max_clusters = max_clusters_of[dev].load(std::memory_order_relaxed);
    if (max_clusters == 0) {
      err = cudaOccupancyMaxActiveClusters(&max_clusters, k_gemm<KIND, PAIR>, &cfg);
      if (err != cudaSuccess) return err;
      max_clusters_of[dev].store(max_clusters, std::memory_order_relaxed);
    }
    if (max_clusters < 1) return cudaErrorInvalidConfiguration;
    const int64_t units = Traits<KIND>::WGRAD
                              ? (E + w.wg_slices[a.wg_kind]) * ((a.m_tiles_w + 1) / 2) * a.n_tiles_n
                          : Traits<KIND>::FUSED ? (m_tiles_max + 1) / 2 * (a.n_tiles_n + a.n2)
                              : (tiles_max / std::max(1, a.n_tiles_n) + 1) / 2 * a.n_tiles_n;
    const int clusters = (int)std::max<int64_t>(1, std::min<int64_t>(max_clusters, units));
    cfg.gridDim = dim3((unsigned)(2 * clusters));
    take_d_topk(2 * clusters);
    cfg.numAttrs = 2;  // and programmatic stream serialization (the occupancy query had only the
                       // cluster shape)
    return cudaLaunchKernelEx(&cfg, k_gemm<KIND, PAIR>, ta, tb, tl, em, a);
  } else {
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(nsm, tiles_max));
    take_d_topk(grid);
    return launch_pdl(k_gemm<KIND, 0>, grid, NUM_THREADS, Traits<KIND>::SMEM, st, ta, tb, tl, em,
                      a);
  }
}

}  // namespace

int device_sm_count() { return sm_count(); }

cudaError_t launch_gemm(const Workspace& w, char* ws, const GemmCall& c, cudaStream_t st) {
  const int pair = c.paired;
  switch (c.kind) {
    case GK_GEMM1_SWIGLU:
      return pair == 2 ? run<GK_GEMM1_SWIGLU, 2>(w, ws, c, st) : run<GK_GEMM1_SWIGLU>(w, ws, c, st);
    case GK_GEMM2:
      return pair == 2 ? run<GK_GEMM2, 2>(w, ws, c, st) : run<GK_GEMM2>(w, ws, c, st);
    case GK_GEMM2_COMBINE: return run<GK_GEMM2_COMBINE>(w, ws, c, st);
    case GK_ACT_GRAD:
      return pair == 2 ? run<GK_ACT_GRAD, 2>(w, ws, c, st) : run<GK_ACT_GRAD>(w, ws, c, st);
    case GK_INPUT_GRAD:
      return pair == 2 ? run<GK_INPUT_GRAD, 2>(w, ws, c, st) : run<GK_INPUT_GRAD>(w, ws, c, st);
    case GK_W2_GRAD:
      return pair == 2 ? run<GK_W2_GRAD, 2>(w, ws, c, st) : run<GK_W2_GRAD>(w, ws, c, st);
    case GK_W1_GRAD:
      return pair == 2 ? run<GK_W1_GRAD, 2>(w, ws, c, st) : run<GK_W1_GRAD>(w, ws, c, st);
    case GK_FWD_FUSED:
      return pair == 2 ? run<GK_FWD_FUSED, 2>(w, ws, c, st) : run<GK_FWD_FUSED>(w, ws, c, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace mm
