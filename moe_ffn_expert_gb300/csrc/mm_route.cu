// Routing preprocessing, dispatch (row gather) and combine (fixed-order weighted unpermute).
//
// RFC "HyperParallel Multicore HyperMegaMoE fused forward/backward operator":
//   §3.3 offsets / group list built inside the operator, §4.1 each token expands into K expert
//   slots, dispatch sends a slot to its expert, combine merges expert outputs back with
//   topk_weights; §2.2 Combine(dX) sums the input-gradient rows of a token's slots.
// On one GPU dispatch is a gather of x rows into expert-sorted order and combine is a gather
// back, summed over k in ascending order in fp32 (deterministic: no atomics on data).
//
// Routing is three small kernels, all integer and bit-exact:
//   count: one warp per chunk of ROUTE_CHUNK slots builds that chunk's per-expert histogram
//          (__match_any_sync groups lanes holding the same expert);
//   scan:  one CTA sums the chunk histograms per expert, scans them into the expert offsets
//          (plain and padded to BM rows), turns the histograms into per-chunk running bases
//          and writes the row-tile -> expert table and the pad-row markers;
//   rank:  each warp replays its chunk in slot order, so a slot's row is its expert's base
//          plus the number of earlier slots of that expert: a stable order in s.
#include <algorithm>

#include "mm_device.cuh"
#include "mm_kernels.h"

namespace mm {
namespace {

template <typename T>
T* region(char* ws, size_t off) {
  return reinterpret_cast<T*>(ws + off);
}
template <typename T>
const T* region(const char* ws, size_t off) {
  return reinterpret_cast<const T*>(ws + off);
}

__global__ void __launch_bounds__(128) k_route_count(const int32_t* __restrict__ ids, int* hdr,
                                                     int32_t* __restrict__ chunk_cnt, int S, int E,
                                                     int n_chunks, TraceCtx tc) {
  pdl_wait();
  const TraceCta trace_cta(tc);
  extern __shared__ int32_t cnt_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * 4 + warp;
  if (chunk >= n_chunks) return;  // whole warp leaves; no CTA-wide barrier below
  int32_t* cnt = cnt_smem + warp * E;
  for (int i = lane; i < E; i += 32) cnt[i] = 0;
  __syncwarp();
  const int s0 = chunk * ROUTE_CHUNK;
  const int s1 = min(S, s0 + ROUTE_CHUNK);
  constexpr int PER_LANE = ROUTE_CHUNK / 32;
  int ev[PER_LANE];  // all of the chunk's ids in flight at once
#pragma unroll
  for (int j = 0; j < PER_LANE; ++j) {
    const int s = s0 + j * 32 + lane;
    ev[j] = s < s1 ? __ldg(ids + s) : -1;
  }
#pragma unroll
  for (int j = 0; j < PER_LANE; ++j) {
    const int s = s0 + j * 32 + lane;
    int e = ev[j];
    if (s < s1 && (e < 0 || e >= E)) {
      set_status(hdr + HDR_STATUS, MM_ERR_BAD_EXPERT_ID);
      atomicCAS(hdr + HDR_BAD_SLOT, 0, s + 1);
      e = -1;
    }
    const unsigned m = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(m) - 1) cnt[e] += __popc(m);
    __syncwarp();
  }
  for (int i = lane; i < E; i += 32) chunk_cnt[(size_t)chunk * E + i] = cnt[i];
}

// Sum of v over the warp's lanes.
__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// Exclusive prefix over the lanes of v (and, through `total`, the warp's sum).
__device__ __forceinline__ int warp_excl(int v, int lane, int& total) {
  int inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += y;
  }
  total = __shfl_sync(0xffffffffu, inc, 31);
  return inc - v;
}

// Chunks for an expert of `blocks` 64-row blocks at threshold `thr` blocks: one unless the
// expert has more than twice that, else about blocks / thr chunks of equal whole blocks.
__device__ __forceinline__ int wgrad_chunks(int blocks, long long thr) {
  if (blocks <= 2 * thr) return 1;
  int s = (int)((blocks + thr - 1) / thr);
  const int per = (blocks + s - 1) / s;  // whole blocks per chunk
  return (blocks + per - 1) / per;
}

// The weight-gradient plans (see WgKind), at the end of the routing scan. A kind whose sizes rule
// out any split (slices < 2, decided on the host) gets one chunk per expert from every thread at
// once. Otherwise one warp plans it (a few sums and prefix sums over the experts, 32 at a time):
// the launch's load per CTA pair is the sum over experts of (64-row blocks x units per chunk)
// over the pairs; an expert with more than twice that many blocks (and more than 32) is cut into
// chunks of about that many whole blocks, so that no unit outlasts the average load by much. If
// the slices that needs do not fit, the threshold doubles until they do (or nothing is split).
// The plan depends only on the routing, the sizes and the device's SM count (not on the CTA
// layout of the launches), so every launch form sums the same partials in the same order.
__device__ void wgrad_plan(int* hdr, const WgPlanArgs& wg, const int* tot_s, const int* po_s,
                           int E) {
  const int tid = threadIdx.x;
  for (int k = 0; k < 2; ++k) {
    if (wg.slices[k] >= 2) continue;
    if (tid < E) {
      int32_t* c = wg.plan + ((size_t)k * wg.plan_stride + tid) * 4;
      c[0] = tid;
      c[1] = po_s[tid];
      c[2] = tot_s[tid];
      c[3] = -1;
    }
    if (tid == 0) {
      hdr[HDR_WG_CHUNKS + k] = E;
      hdr[HDR_WG_SPLITS + k] = 0;
    }
  }
  if ((wg.slices[0] < 2 && wg.slices[1] < 2) || tid >= 32) return;
  const int lane = tid;
  auto blocks_of = [&](int e) { return e < E ? (tot_s[e] + BK - 1) / BK : 0; };
  int sum_blocks = 0;
  for (int e0 = 0; e0 < E; e0 += 32) sum_blocks += warp_sum(blocks_of(e0 + lane));
  for (int k = 0; k < 2; ++k) {
    if (wg.slices[k] < 2) continue;
    int32_t* plan = wg.plan + (size_t)k * wg.plan_stride * 4;
    int32_t* red = wg.red + (size_t)k * E * 4;
    long long thr = (long long)wg.units[k] * sum_blocks / (wg.pairs > 0 ? wg.pairs : 1);
    if (thr < 16) thr = 16;
    bool split = true;
    for (int round = 0;; ++round) {  // warp-uniform: the chunk count is a warp sum
      int need = 0;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int s = wgrad_chunks(blocks_of(e0 + lane), thr);
        need += warp_sum(s > 1 ? s : 0);
      }
      if (need <= wg.slices[k]) break;
      if (round == 40) {
        split = false;
        break;
      }
      thr *= 2;
    }
    // totals first (split chunks come first in the table), then the entries
    int n_split = 0, n_splitters = 0;
    if (split)
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int s = wgrad_chunks(blocks_of(e0 + lane), thr);
        n_split += warp_sum(s > 1 ? s : 0);
        n_splitters += warp_sum(s > 1 ? 1 : 0);
      }
    int base_a = 0, base_b = 0, base_c = 0;  // running chunk, unsplit and splitter indices
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int blocks = blocks_of(e);
      const int s = (split && e < E) ? wgrad_chunks(blocks, thr) : 1;
      int ta, tb, tc;
      const int xa = warp_excl(s > 1 ? s : 0, lane, ta);
      const int xb = warp_excl((e < E && s == 1) ? 1 : 0, lane, tb);
      const int xc = warp_excl(s > 1 ? 1 : 0, lane, tc);
      if (e < E) {
        const int rows = tot_s[e], po = po_s[e];
        if (s > 1) {  // chunks base_a + xa .., each with the slice of its own index
          const int per_rows = ((blocks + s - 1) / s) * BK;
          for (int i = 0; i < s; ++i) {
            const int ci = base_a + xa + i;
            int32_t* c = plan + 4 * ci;
            c[0] = e;
            c[1] = po + i * per_rows;
            c[2] = min(per_rows, rows - i * per_rows);
            c[3] = ci;
          }
          int32_t* r = red + 4 * (base_c + xc);
          r[0] = e;
          r[1] = base_a + xa;
          r[2] = s;
          r[3] = 0;
        } else {  // one chunk after every split chunk, in expert order
          int32_t* c = plan + 4 * (n_split + base_b + xb);
          c[0] = e;
          c[1] = po;
          c[2] = rows;
          c[3] = -1;
        }
      }
      base_a += ta;
      base_b += tb;
      base_c += tc;
    }
    if (lane == 0) {
      hdr[HDR_WG_CHUNKS + k] = n_split + base_b;
      hdr[HDR_WG_SPLITS + k] = n_splitters;
    }
  }
}

// One CTA of 1024 threads. Each expert gets P = 1024 / E threads (a power of two, 1 to 32), each
// owning a contiguous range of the chunk histograms; thread tid serves expert tid % E, so a
// warp reads 32 consecutive experts of one chunk (coalesced). The P threads of an expert sum
// their ranges, the expert totals are scanned across experts (plain and padded to BM rows),
// and each thread then turns its range into running padded-row bases. The row-tile, pair and
// pad-row tables are written last, one warp per expert with coalesced stores (per-expert
// threads writing them took most of the kernel's time: their stores were scattered).
__global__ void __launch_bounds__(1024) k_route_scan(int* hdr, int32_t* __restrict__ chunk_cnt,
                                                     int32_t* __restrict__ counts,
                                                     int32_t* __restrict__ offsets,
                                                     int32_t* __restrict__ poff,
                                                     int32_t* __restrict__ tile_expert,
                                                     int32_t* __restrict__ slot_of_row,
                                                     float* __restrict__ w_row,
                                                     int32_t* __restrict__ pair_tile,
                                                     int32_t* __restrict__ ready,
                                                     const int32_t* __restrict__ tpe, int E,
                                                     int n_chunks, WgPlanArgs wg, TraceCtx tc) {
  pdl_wait();
  const TraceCta trace_cta(tc);
  __shared__ int wsum[32], wsum_p[32], wsum_q[32];
  __shared__ int tot_s[1024], po_s[1024], qo_s[1024], seg_s[1024];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (hdr[HDR_STATUS] != 0) {  // bad ids: schedule nothing downstream
    if (tid == 0) hdr[HDR_NUM_MTILES] = 0;
    return;
  }
  int P = 1;  // threads per expert
  while (P < 32 && P * 2 * E <= 1024) P *= 2;
  const int e = tid % E, j = tid / E;
  const bool active = j < P;
  const int L = (n_chunks + P - 1) / P;  // chunks per thread
  const int k0 = min(n_chunks, j * L), k1 = min(n_chunks, k0 + L);
  int seg = 0;
  if (active) {
#pragma unroll 8
    for (int k = k0; k < k1; ++k) seg += chunk_cnt[(size_t)k * E + e];
    seg_s[j * E + e] = seg;
  }
  __syncthreads();
  // this thread's exclusive prefix over the expert's earlier ranges, and the expert's total
  int before = 0, total = 0;
  if (active) {
    for (int i = 0; i < P; ++i) {
      const int v = seg_s[i * E + e];
      before += i < j ? v : 0;
      total += v;
    }
    if (j == 0) tot_s[e] = total;
  }
  __syncthreads();

  // scan of the expert totals (plain and padded), one thread per expert
  const int c = tid < E ? tot_s[tid] : 0;
  // a caller's histogram is only compared, never used for addressing
  if (tpe != nullptr && tid < E && __ldg(tpe + tid) != c)
    set_status(hdr + HDR_STATUS, MM_ERR_TOKENS_PER_EXPERT);
  const int pc = (c + BM - 1) / BM * BM;
  const int pq = (pc / BM + 1) / 2;  // pairs of row tiles
  int a = c, b = pc, q = pq;  // inclusive warp scans
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int ya = __shfl_up_sync(0xffffffffu, a, d);
    const int yb = __shfl_up_sync(0xffffffffu, b, d);
    const int yq = __shfl_up_sync(0xffffffffu, q, d);
    if (lane >= d) {
      a += ya;
      b += yb;
      q += yq;
    }
  }
  if (lane == 31) {
    wsum[warp] = a;
    wsum_p[warp] = b;
    wsum_q[warp] = q;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int u = lane < nw ? wsum[lane] : 0, v = lane < nw ? wsum_p[lane] : 0;
    int z = lane < nw ? wsum_q[lane] : 0;
    const int u0 = u, v0 = v, z0 = z;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int yu = __shfl_up_sync(0xffffffffu, u, d);
      const int yv = __shfl_up_sync(0xffffffffu, v, d);
      const int yz = __shfl_up_sync(0xffffffffu, z, d);
      if (lane >= d) {
        u += yu;
        v += yv;
        z += yz;
      }
    }
    wsum[lane] = u - u0;  // exclusive prefix of warp totals
    wsum_p[lane] = v - v0;
    wsum_q[lane] = z - z0;
  }
  __syncthreads();
  if (tid < E) {
    const int off = a - c + wsum[warp];
    const int po = b - pc + wsum_p[warp];
    const int qo = q - pq + wsum_q[warp];
    counts[tid] = c;
    offsets[tid] = off;
    poff[tid] = po;
    po_s[tid] = po;
    qo_s[tid] = qo;
    if (tid == E - 1) {
      offsets[E] = off + c;
      poff[E] = po + pc;
      hdr[HDR_NUM_MTILES] = (po + pc) / BM;
      hdr[HDR_NUM_MPAIRS] = qo + pq;
    }
  }
  __syncthreads();
  if (active) {
    // chunk histograms -> running padded-row base of each chunk (this thread's range)
    int run = po_s[e] + before;
    int k = k0;
    for (; k + 8 <= k1; k += 8) {  // eight loads in flight, then the running sums
      int v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = chunk_cnt[(size_t)(k + i) * E + e];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        chunk_cnt[(size_t)(k + i) * E + e] = run;
        run += v[i];
      }
    }
    for (; k < k1; ++k) {
      const int v = chunk_cnt[(size_t)k * E + e];
      chunk_cnt[(size_t)k * E + e] = run;
      run += v;
    }
  }
  // each expert's row tiles (and their ready counters for the one-launch forward, zeroed here so
  // that no memset has to run between the launches), row-tile pairs and pad-row markers: one warp
  // per expert at a time, its lanes over consecutive entries, so that every store instruction is
  // coalesced
  for (int ex = warp; ex < E; ex += (int)(blockDim.x >> 5)) {
    const int tot = tot_s[ex], po = po_s[ex], qo = qo_s[ex];
    const int pcount = (tot + BM - 1) / BM * BM, ntile = pcount / BM;
    for (int t = lane; t < ntile; t += 32) {
      tile_expert[po / BM + t] = ex;
      ready[po / BM + t] = 0;
    }
    for (int i = lane; i < (ntile + 1) / 2; i += 32) {
      const int t0 = po / BM + 2 * i;
      pair_tile[qo + i] = 2 * i + 1 < ntile ? t0 : ~t0;
    }
    for (int r = po + tot + lane; r < po + pcount; r += 32) {
      slot_of_row[r] = -1;
      w_row[r] = 0.0f;
    }
  }
  wgrad_plan(hdr, wg, tot_s, po_s, E);
}

__global__ void __launch_bounds__(128) k_route_rank(const int32_t* __restrict__ ids,
                                                    const float* __restrict__ topk_w,
                                                    const int* hdr,
                                                    const int32_t* __restrict__ chunk_base,
                                                    int32_t* __restrict__ row_of_slot,
                                                    int32_t* __restrict__ slot_of_row,
                                                    float* __restrict__ w_row, int S, int E,
                                                    int n_chunks, TraceCtx tc) {
  pdl_wait();
  const TraceCta trace_cta(tc);
  extern __shared__ int32_t cnt_smem[];
  if (hdr[HDR_STATUS] != 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * 4 + warp;
  if (chunk >= n_chunks) return;
  int32_t* cnt = cnt_smem + warp * E;
  for (int i = lane; i < E; i += 32) cnt[i] = chunk_base[(size_t)chunk * E + i];
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
  const int s0 = chunk * ROUTE_CHUNK;
  const int s1 = min(S, s0 + ROUTE_CHUNK);
  constexpr int PER_LANE = ROUTE_CHUNK / 32;
  int ev[PER_LANE];
  float wv[PER_LANE];
#pragma unroll
  for (int j = 0; j < PER_LANE; ++j) {
    const int s = s0 + j * 32 + lane;
    ev[j] = s < s1 ? __ldg(ids + s) : -1;
    wv[j] = s < s1 ? __ldg(topk_w + s) : 0.0f;
  }
#pragma unroll
  for (int j = 0; j < PER_LANE; ++j) {
    const int s = s0 + j * 32 + lane;
    const int e = ev[j];
    const unsigned m = __match_any_sync(0xffffffffu, e);
    int row = 0;
    if (e >= 0) row = cnt[e] + __popc(m & lt);
    __syncwarp();
    if (e >= 0 && lane == __ffs(m) - 1) cnt[e] += __popc(m);
    __syncwarp();
    if (e >= 0) {
      row_of_slot[s] = row;
      slot_of_row[row] = s;
      w_row[row] = wv[j];
    }
  }
}

// One warp per destination row, 16-byte vectors. The rows are written with the streaming
// (evict-first) cache hint: on a GB300 that made the gathers ~6 % faster (qwen, 0.1335 -> 0.126
// ms each) and left the GEMMs that read the rows next unchanged.
__global__ void __launch_bounds__(256) k_gather_rows(const uint4* __restrict__ src,
                                                     uint4* __restrict__ dst,
                                                     const int32_t* __restrict__ slot_of_row,
                                                     const int* hdr, int K, int vpr,
                                                     TraceCtx tc) {
  pdl_wait();
  const TraceCta trace_cta(tc);
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (hdr[HDR_STATUS] != 0 || row >= hdr[HDR_NUM_MTILES] * BM) return;
  const int s = slot_of_row[row];
  uint4* d = dst + (size_t)row * vpr;
  if (s < 0) {
    for (int i = lane; i < vpr; i += 32) __stcs(d + i, make_uint4(0u, 0u, 0u, 0u));
    return;
  }
  const uint4* p = src + (size_t)(s / K) * vpr;
#pragma unroll 4
  for (int i = lane; i < vpr; i += 32) __stcs(d + i, __ldg(p + i));
}

__device__ __forceinline__ void acc8(float (&a)[8], float w, const uint4& v) {
  a[0] += w * bf16_lo(v.x);
  a[1] += w * bf16_hi(v.x);
  a[2] += w * bf16_lo(v.y);
  a[3] += w * bf16_hi(v.y);
  a[4] += w * bf16_lo(v.z);
  a[5] += w * bf16_hi(v.z);
  a[6] += w * bf16_lo(v.w);
  a[7] += w * bf16_hi(v.w);
}

// The extra rows (weight 1), then one rounding to bf16 and the 16-byte store of out[t][i].
__device__ __forceinline__ void combine_tail(float (&a)[8], const uint4* __restrict__ extra,
                                             const uint4* __restrict__ extra_lo,
                                             uint4* __restrict__ out, int t, int vpr, int i) {
  if (extra != nullptr) acc8(a, 1.0f, __ldg(extra + (size_t)t * vpr + i));
  if (extra_lo != nullptr) acc8(a, 1.0f, __ldg(extra_lo + (size_t)t * vpr + i));
  uint4 o;
  o.x = pack_bf16(a[0], a[1]);
  o.y = pack_bf16(a[2], a[3]);
  o.z = pack_bf16(a[4], a[5]);
  o.w = pack_bf16(a[6], a[7]);
  out[(size_t)t * vpr + i] = o;
}

// One warp per token, 8 columns (16 bytes) per lane per step, slots summed in k order.
// ROW_TABLE: the warp first puts its token's row pointers and weights in shared memory and loads
// eight slots' rows at a time (64 registers, more loads in flight: the forward's combine, ~30 %
// faster alone); without it the table stays in registers and the kernel uses no shared memory,
// which lets more of its CTAs sit beside a GEMM's (the backward's combine beside W1Grad).
// `extra` (optional): one more row per token, row t, added with weight 1 after the K slots
// (the shared expert's output, or its input-gradient rows), as a bf16 hi row plus, when
// `extra_lo` is set, its bf16 lo row (hi + lo carries about 16 significant bits).
template <bool ROW_TABLE>
__global__ void __launch_bounds__(256) k_combine(const uint4* __restrict__ rows,
                                                 const int32_t* __restrict__ row_of_slot,
                                                 const float* __restrict__ weights,
                                                 const uint4* __restrict__ extra,
                                                 const uint4* __restrict__ extra_lo,
                                                 uint4* __restrict__ out, const int* hdr, int T,
                                                 int K, int vpr, TraceCtx tc) {
  pdl_wait();
  const TraceCta trace_cta(tc);
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (hdr[HDR_STATUS] != 0 || t >= T) return;
  if constexpr (ROW_TABLE) {
    __shared__ const uint4* rp_s[8][16];
    __shared__ float w_s[8][16];
    const int wi = threadIdx.x >> 5;
    if (lane < K) {
      rp_s[wi][lane] = rows + (size_t)__ldg(row_of_slot + (size_t)t * K + lane) * vpr;
      w_s[wi][lane] = weights != nullptr ? __ldg(weights + (size_t)t * K + lane) : 1.0f;
    }
    __syncwarp();
    for (int i = lane; i < vpr; i += 32) {
      float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k0 = 0; k0 < 16; k0 += 8) {
        if (k0 < K) {
          uint4 v[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (k0 + k < K) v[k] = __ldg(rp_s[wi][k0 + k] + i);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (k0 + k < K) acc8(a, w_s[wi][k0 + k], v[k]);
        }
      }
      combine_tail(a, extra, extra_lo, out, t, vpr, i);
    }
  } else {
    int r[16];
    float w[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      r[k] = k < K ? __ldg(row_of_slot + (size_t)t * K + k) : 0;
      w[k] = (k < K && weights != nullptr) ? __ldg(weights + (size_t)t * K + k) : 1.0f;
    }
    for (int i = lane; i < vpr; i += 32) {
      float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (k < K) acc8(a, w[k], __ldg(rows + (size_t)r[k] * vpr + i));
      combine_tail(a, extra, extra_lo, out, t, vpr, i);
    }
  }
}



__global__ void __launch_bounds__(256) k_d_topk(const float* __restrict__ p_part,
                                                const int32_t* __restrict__ row_of_slot,
                                                float* __restrict__ d_topk, const int* hdr, int S,
                                                int n_tiles, int64_t S_pad, TraceCtx tc) {
  pdl_wait();
  const TraceCta trace_cta(tc);
  const int s = blockIdx.x * 256 + threadIdx.x;
  if (hdr[HDR_STATUS] != 0 || s >= S) return;
  const int r = row_of_slot[s];
  float acc = 0.f;
  for (int j = 0; j < n_tiles; ++j) acc += p_part[(size_t)j * S_pad + r];
  d_topk[s] = acc;
}

__global__ void __launch_bounds__(256) k_export_rows(const int32_t* __restrict__ row_of_slot,
                                                     const int32_t* __restrict__ tile_expert,
                                                     const int32_t* __restrict__ poff,
                                                     const int32_t* __restrict__ offsets,
                                                     int32_t* __restrict__ out, const int* hdr,
                                                     int S) {
  const int s = blockIdx.x * 256 + threadIdx.x;
  if (s >= S) return;
  if (hdr[HDR_STATUS] != 0) {
    out[s] = -1;
    return;
  }
  const int r = row_of_slot[s];
  const int e = tile_expert[r / BM];
  out[s] = r - poff[e] + offsets[e];
}

// Routing tables of the shared expert (one expert, every token, weight 1, identity order):
// padded row r is token r (r < T), the rows up to the next multiple of BM are pad rows.
__global__ void __launch_bounds__(256) k_shared_tables(int* hdr, int32_t* counts, int32_t* offsets,
                                                       int32_t* poff, int32_t* tile_expert,
                                                       int32_t* pair_tile, int32_t* slot_of_row,
                                                       float* w_row, int32_t* row_of_slot, int T,
                                                       int32_t* wg_plan, int wg_plan_stride,
                                                       TraceCtx tc) {
  pdl_wait();
  const TraceCta trace_cta(tc);
  const int Tp = (T + BM - 1) / BM * BM;
  const int nm = Tp / BM;
  const int r = blockIdx.x * 256 + threadIdx.x;
  if (r < HDR_WORDS)  // every header word
    hdr[r] = r == HDR_NUM_MTILES                                       ? nm
             : r == HDR_NUM_MPAIRS                                     ? (nm + 1) / 2
             : (r == HDR_WG_CHUNKS + WG_W2 || r == HDR_WG_CHUNKS + WG_W1) ? 1
                                                                       : 0;
  // weight-gradient plans: one row chunk, all T rows, stored to the output (never split)
  if (r < 2) {
    int32_t* c = wg_plan + 4 * (size_t)r * wg_plan_stride;
    c[0] = 0;
    c[1] = 0;
    c[2] = T;
    c[3] = -1;
  }
  // row tiles 2i and 2i + 1 form pair i (~2i when the second is past the last row tile)
  if (r < (nm + 1) / 2) pair_tile[r] = 2 * r + 1 < nm ? 2 * r : ~(2 * r);
  if (r == 0) {
    counts[0] = T;
    offsets[0] = 0;
    offsets[1] = T;
    poff[0] = 0;
    poff[1] = Tp;
  }
  if (r < Tp) {
    if (r % BM == 0) tile_expert[r / BM] = 0;
    slot_of_row[r] = r < T ? r : -1;
    w_row[r] = r < T ? 1.0f : 0.0f;
    if (r < T) row_of_slot[r] = r;
  }
}

// A backward with no slot to compute (T = 0) still refuses a workspace whose forward kept no
// gate|up (MM_FLAG_FORWARD_ONLY), as the act_grad kernel does when T > 0.
__global__ void k_backward_check(int* hdr) {
  pdl_wait();
  if (hdr[HDR_NO_BACKWARD] != 0) set_status(hdr + HDR_STATUS, MM_ERR_INVALID_ARG);
}

// The sums of split weight gradients (see WgKind). Work item i = (split expert j, group of four
// elements q of its M x N gradient): out[e] = the sum over the expert's chunks, in chunk order,
// of their fp32 partial slices, rounded once to bf16 (or kept in fp32), or added into out the way
// the direct path's reduce-add stores add (bf16: bf16(out + bf16(sum)); fp32: out + sum).
// Grid-stride; with no split expert the launch returns at once.
__global__ void __launch_bounds__(256) k_wgrad_reduce(const int* hdr, int kind,
                                                      const int4* __restrict__ red,
                                                      const float4* __restrict__ part, void* out,
                                                      int64_t slice4, int out_f32, int accumulate,
                                                      TraceCtx tc) {
  pdl_wait();
  const TraceCta trace_cta(tc);
  if (hdr[HDR_STATUS] != 0) return;
  const int64_t total = (int64_t)hdr[HDR_WG_SPLITS + kind] * slice4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(i / slice4);
    const int64_t q = i - (int64_t)j * slice4;
    const int4 r = __ldg(red + j);  // {expert, first slice, slices, 0}
    float4 acc = __ldg(part + (int64_t)r.y * slice4 + q);
    for (int s = 1; s < r.z; ++s) {
      const float4 v = __ldg(part + (int64_t)(r.y + s) * slice4 + q);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const int64_t o = (int64_t)r.x * slice4 + q;
    if (out_f32) {
      float4* op = reinterpret_cast<float4*>(out) + o;
      if (accumulate) {
        const float4 b = *op;
        acc.x = b.x + acc.x;
        acc.y = b.y + acc.y;
        acc.z = b.z + acc.z;
        acc.w = b.w + acc.w;
      }
      *op = acc;
    } else {
      uint2* op = reinterpret_cast<uint2*>(out) + o;
      float f[4] = {acc.x, acc.y, acc.z, acc.w};
      if (accumulate) {
        const uint2 b = *op;
        const float old[4] = {bf16_lo(b.x), bf16_hi(b.x), bf16_lo(b.y), bf16_hi(b.y)};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          f[u] = old[u] + __bfloat162float(__float2bfloat16_rn(f[u]));
      }
      *op = make_uint2(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]));
    }
  }
}

inline unsigned div_up(int64_t a, int64_t b) { return (unsigned)((a + b - 1) / b); }

}  // namespace

cudaError_t launch_route_count(const Workspace& w, char* ws, const int32_t* ids, cudaStream_t st) {
  const unsigned grid = div_up(w.n_chunks, 4);
  return launch_pdl(k_route_count, grid, 128, 4 * w.E * sizeof(int32_t), st, ids,
                    region<int>(ws, w.off_hdr), region<int32_t>(ws, w.off_chunk), (int)w.S,
                    (int)w.E, (int)w.n_chunks, trace_ctx());
}

namespace {

// CTA-pair units per row chunk of a weight-gradient kind (row-tile pairs x 256-column tiles).
int64_t wgrad_units(const Workspace& w, int kind) {
  const int64_t rows_w = kind == WG_W1 ? 2 * w.I : w.I;
  return ((rows_w + BM - 1) / BM + 1) / 2 * ((w.H + BN - 1) / BN);
}

}  // namespace

// Whether the plan of weight-gradient `kind` may split an expert, decided from the sizes alone:
// an expert with distinct experts per token holds at most T rows (ceil(T / 64) blocks), and the
// average load per CTA pair is at least units x floor(S / 64) / pairs blocks; a split needs the
// first to exceed twice the second (and 32 blocks), and at least two partial slices. When it
// cannot happen the scan writes one chunk per expert and no sum is launched. (Duplicate experts
// in a token can make an expert longer than T rows; such an expert is then simply not split.)
bool wgrad_split_possible(const Workspace& w, int kind) {
  if (w.wg_slices[kind] < 2) return false;
  const int64_t pairs = std::max(1, device_sm_count() / 2);
  const int64_t thr = std::max<int64_t>(16, wgrad_units(w, kind) * (w.S / BK) / pairs);
  return (w.T + BK - 1) / BK > 2 * thr;
}

cudaError_t launch_route_scan(const Workspace& w, char* ws, const int32_t* tokens_per_expert,
                              cudaStream_t st) {
  WgPlanArgs wg{};
  wg.plan = region<int32_t>(ws, w.off_wg_plan);
  wg.red = region<int32_t>(ws, w.off_wg_red);
  for (int k = 0; k < 2; ++k) {
    wg.units[k] = (int)wgrad_units(w, k);
    wg.slices[k] = wgrad_split_possible(w, k) ? (int)w.wg_slices[k] : 0;
  }
  wg.plan_stride = (int)(w.E + w.wg_slices_max);
  wg.pairs = device_sm_count() / 2;
  return launch_pdl(k_route_scan, 1, 1024, 0, st, region<int>(ws, w.off_hdr),
                    region<int32_t>(ws, w.off_chunk), region<int32_t>(ws, w.off_counts),
                    region<int32_t>(ws, w.off_offsets), region<int32_t>(ws, w.off_poff),
                    region<int32_t>(ws, w.off_tile_expert), region<int32_t>(ws, w.off_slot_of_row),
                    region<float>(ws, w.off_w_row), region<int32_t>(ws, w.off_pair_tile),
                    region<int32_t>(ws, w.off_ready), tokens_per_expert, (int)w.E,
                    (int)w.n_chunks, wg, trace_ctx());
}

cudaError_t launch_route_rank(const Workspace& w, char* ws, const int32_t* ids, const float* topk_w,
                              cudaStream_t st) {
  const unsigned grid = div_up(w.n_chunks, 4);
  return launch_pdl(k_route_rank, grid, 128, 4 * w.E * sizeof(int32_t), st, ids, topk_w,
                    region<int>(ws, w.off_hdr), region<int32_t>(ws, w.off_chunk),
                    region<int32_t>(ws, w.off_row_of_slot), region<int32_t>(ws, w.off_slot_of_row),
                    region<float>(ws, w.off_w_row), (int)w.S, (int)w.E, (int)w.n_chunks,
                    trace_ctx());
}

cudaError_t launch_gather_rows(const Workspace& w, char* ws, const void* src, void* dst,
                               cudaStream_t st) {
  const unsigned grid = div_up(w.S_pad, 8);
  return launch_pdl(k_gather_rows, grid, 256, 0, st, reinterpret_cast<const uint4*>(src),
                    reinterpret_cast<uint4*>(dst), region<int32_t>(ws, w.off_slot_of_row),
                    region<int>(ws, w.off_hdr), (int)w.K, (int)(w.H / 8), trace_ctx());
}

cudaError_t launch_combine(const Workspace& w, char* ws, const void* rows, const float* weights,
                           void* out, cudaStream_t st, const void* extra,
                           const void* extra_lo, bool row_table) {
  const unsigned grid = div_up(w.T, 8);
  auto kern = row_table ? k_combine<true> : k_combine<false>;
  return launch_pdl(kern, grid, 256, 0, st, reinterpret_cast<const uint4*>(rows),
                    region<int32_t>(ws, w.off_row_of_slot), weights,
                    reinterpret_cast<const uint4*>(extra), reinterpret_cast<const uint4*>(extra_lo),
                    reinterpret_cast<uint4*>(out), region<int>(ws, w.off_hdr), (int)w.T, (int)w.K,
                    (int)(w.H / 8), trace_ctx());
}

cudaError_t launch_d_topk(const Workspace& w, char* ws, float* d_topk, cudaStream_t st) {
  const unsigned grid = div_up(w.S, 256);
  return launch_pdl(k_d_topk, grid, 256, 0, st, region<float>(ws, w.off_p_part),
                    region<int32_t>(ws, w.off_row_of_slot), d_topk, region<int>(ws, w.off_hdr),
                    (int)w.S, (int)w.n_act_tiles, w.S_pad, trace_ctx());
}

cudaError_t launch_shared_tables(const Workspace& ws_shared, char* ws, cudaStream_t st) {
  const Workspace& w = ws_shared;
  return launch_pdl(k_shared_tables, div_up((w.T + BM - 1) / BM * BM, 256), 256, 0, st,
                    region<int>(ws, w.off_hdr), region<int32_t>(ws, w.off_counts),
                    region<int32_t>(ws, w.off_offsets), region<int32_t>(ws, w.off_poff),
                    region<int32_t>(ws, w.off_tile_expert), region<int32_t>(ws, w.off_pair_tile),
                    region<int32_t>(ws, w.off_slot_of_row), region<float>(ws, w.off_w_row),
                    region<int32_t>(ws, w.off_row_of_slot), (int)w.T,
                    region<int32_t>(ws, w.off_wg_plan), (int)(w.E + w.wg_slices_max), trace_ctx());
}

cudaError_t launch_backward_check(const Workspace& w, char* ws, cudaStream_t st) {
  return launch_pdl(k_backward_check, 1, 1, 0, st, region<int>(ws, w.off_hdr));
}

cudaError_t launch_export_rows(const Workspace& w, const char* ws, int32_t* out, cudaStream_t st) {
  const unsigned grid = div_up(w.S, 256);
  k_export_rows<<<grid, 256, 0, st>>>(
      region<int32_t>(ws, w.off_row_of_slot), region<int32_t>(ws, w.off_tile_expert),
      region<int32_t>(ws, w.off_poff), region<int32_t>(ws, w.off_offsets), out,
      region<int>(ws, w.off_hdr), (int)w.S);
  return cudaGetLastError();
}

}  // namespace mm

namespace mm {

cudaError_t launch_wgrad_reduce(const Workspace& w, char* ws, int kind, void* out, bool out_f32,
                                bool accumulate, cudaStream_t st) {
  const int64_t mn = kind == WG_W1 ? 2 * w.I * w.H : w.I * w.H;  // elements of one gradient
  const size_t part_off = (kind == WG_W1 && w.wg_slices[WG_W1] > 0) ? w.off_dy_slot : w.off_o;
  const unsigned grid = (unsigned)std::max(1, device_sm_count() * 2);
  return launch_pdl(k_wgrad_reduce, grid, 256, 0, st, region<int>(ws, w.off_hdr), kind,
                    reinterpret_cast<const int4*>(ws + w.off_wg_red) + (size_t)kind * w.E,
                    reinterpret_cast<const float4*>(ws + part_off), out, mn / 4,
                    out_f32 ? 1 : 0, accumulate ? 1 : 0, trace_ctx());
}

}  // namespace mm
