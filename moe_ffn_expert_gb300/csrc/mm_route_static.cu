// Routing tables without any caller workspace: mm_route_noalloc.
//
// Some callers cannot allocate device memory at the point where they need the routing
// tables: code running inside a framework that owns the device heap and forbids
// allocation during a step, or a runtime that prepares work ahead of time and may only
// pass pointers it already holds. They can still pass their inputs and outputs. For
// them this entry point computes the same per-expert counts, offsets and stable
// expert-sorted slot positions as mm_forward/mm_routing_export, but keeps its scratch
// (a status word and the per-chunk expert histograms) in one file-scope device array.
//
// That array is a static, process-lifetime allocation on every GPU that loads the library
// (NA_SCRATCH_BYTES below); every call shares it, so calls whose kernels overlap on the
// GPU (two streams, or two host threads) race on it. Host code cannot use the array's
// name as a device address: the first call on each device looks the address up with
// cudaGetSymbolAddress (that first call must happen before any stream capture). Every call
// first makes the current device's primary context current on the calling thread, so the
// address it looked up and the kernels it launches belong to the same context.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/mm.h"
#include "mm_kernels.h"

namespace {

constexpr int NA_CHUNK = 1024;                 // slots per warp
constexpr int64_t NA_MAX_SLOTS = 1 << 20;      // T*K limit of this entry point
constexpr int NA_MAX_E = 1024;                 // expert limit (one scan CTA)
constexpr int64_t NA_MAX_CHUNKS = NA_MAX_SLOTS / NA_CHUNK;
constexpr int NA_HDR_WORDS = 64;               // word 0: status
constexpr int64_t NA_WORDS = NA_HDR_WORDS + NA_MAX_CHUNKS * NA_MAX_E;
constexpr size_t NA_SCRATCH_BYTES = NA_WORDS * sizeof(int32_t);  // 4 MiB + 256 B

static_assert(NA_SCRATCH_BYTES == (4u << 20) + 256u, "4 MiB of histograms + a 256-byte header");
static __device__ __align__(256) int32_t g_route_scratch[NA_WORDS];

__global__ void __launch_bounds__(128) k_na_count(const int32_t* __restrict__ ids,
                                                  int32_t* scratch, int S, int E, int n_chunks) {
  extern __shared__ int32_t cnt_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * 4 + warp;
  if (chunk >= n_chunks) return;
  int32_t* cnt = cnt_smem + warp * E;
  int32_t* hist = scratch + NA_HDR_WORDS;
  for (int i = lane; i < E; i += 32) cnt[i] = 0;
  __syncwarp();
  const int s1 = min(S, (chunk + 1) * NA_CHUNK);
  for (int base = chunk * NA_CHUNK; base < s1; base += 32) {
    const int s = base + lane;
    int e = -1;
    if (s < s1) {
      e = __ldg(ids + s);
      if (e < 0 || e >= E) {
        atomicCAS(scratch, 0, (int)MM_ERR_BAD_EXPERT_ID);
        e = -1;
      }
    }
    const unsigned m = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(m) - 1) cnt[e] += __popc(m);
    __syncwarp();
  }
  for (int i = lane; i < E; i += 32) hist[(size_t)chunk * E + i] = cnt[i];
}

// One CTA: per-expert totals, exclusive offsets, per-chunk running bases.
__global__ void __launch_bounds__(1024) k_na_scan(int32_t* scratch, int32_t* __restrict__ counts,
                                                  int32_t* __restrict__ offsets, int E,
                                                  int n_chunks) {
  __shared__ int wsum[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* hist = scratch + NA_HDR_WORDS;
  const bool bad = scratch[0] != 0;
  int c = 0;
  if (!bad && tid < E)
    for (int k = 0; k < n_chunks; ++k) c += hist[(size_t)k * E + tid];
  int a = c;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, a, d);
    if (lane >= d) a += y;
  }
  if (lane == 31) wsum[warp] = a;
  __syncthreads();
  if (warp == 0) {
    int u = wsum[lane];
    const int u0 = u;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, u, d);
      if (lane >= d) u += y;
    }
    wsum[lane] = u - u0;
  }
  __syncthreads();
  if (tid >= E) return;
  if (bad) {
    counts[tid] = -1;
    offsets[tid] = -1;
    if (tid == E - 1) offsets[E] = -1;
    return;
  }
  const int off = a - c + wsum[warp];
  counts[tid] = c;
  offsets[tid] = off;
  if (tid == E - 1) offsets[E] = off + c;
  int run = off;
  for (int k = 0; k < n_chunks; ++k) {
    const int v = hist[(size_t)k * E + tid];
    hist[(size_t)k * E + tid] = run;
    run += v;
  }
}

__global__ void __launch_bounds__(128) k_na_rank(const int32_t* __restrict__ ids,
                                                 const int32_t* scratch,
                                                 int32_t* __restrict__ row_of_slot, int S, int E,
                                                 int n_chunks) {
  extern __shared__ int32_t cnt_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * 4 + warp;
  if (chunk >= n_chunks) return;
  const int s1 = min(S, (chunk + 1) * NA_CHUNK);
  if (scratch[0] != 0) {
    for (int s = chunk * NA_CHUNK + lane; s < s1; s += 32) row_of_slot[s] = -1;
    return;
  }
  int32_t* cnt = cnt_smem + warp * E;
  const int32_t* hist = scratch + NA_HDR_WORDS;
  for (int i = lane; i < E; i += 32) cnt[i] = hist[(size_t)chunk * E + i];
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
  for (int base = chunk * NA_CHUNK; base < s1; base += 32) {
    const int s = base + lane;
    const int e = s < s1 ? __ldg(ids + s) : -1;
    const unsigned m = __match_any_sync(0xffffffffu, e);
    int row = 0;
    if (e >= 0) row = cnt[e] + __popc(m & lt);
    __syncwarp();
    if (e >= 0 && lane == __ffs(m) - 1) cnt[e] += __popc(m);
    __syncwarp();
    if (e >= 0) row_of_slot[s] = row;
  }
}

// Records the failing step and CUDA error for mm_last_error_detail; returns MM_ERR_CUDA.
mm_status fail(const char* step, cudaError_t e) {
  mm::note_error("mm_route_noalloc: %s: %s (%s)", step, cudaGetErrorString(e), cudaGetErrorName(e));
  return MM_ERR_CUDA;
}

// Makes the current device's primary context current on this thread (the one the scratch
// address below belongs to) and returns the device address of g_route_scratch on it, looked up
// once per device. Concurrent first calls may both look it up; they store the same address.
int32_t* scratch_ptr(mm_status* st) {
  static std::atomic<int32_t*> cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess && (dev < 0 || dev >= 64)) e = cudaErrorInvalidDevice;
  if (e == cudaSuccess) e = cudaSetDevice(dev);
  if (e != cudaSuccess) {
    *st = fail("device / context", e);
    return nullptr;
  }
  int32_t* p = cache[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    void* q = nullptr;
    e = cudaGetSymbolAddress(&q, g_route_scratch);
    if (e == cudaSuccess && q == nullptr) e = cudaErrorInvalidSymbol;
    if (e != cudaSuccess) {
      *st = fail("cudaGetSymbolAddress of the scratch array", e);
      return nullptr;
    }
    p = static_cast<int32_t*>(q);
    cache[dev].store(p, std::memory_order_release);
  }
  *st = MM_OK;
  return p;
}

}  // namespace

extern "C" mm_status mm_route_noalloc(mm_dims d, const int32_t* topk_ids, int32_t* counts,
                                      int32_t* offsets, int32_t* row_of_slot, void* stream) {
  if (d.T < 0 || d.K < 1 || d.E < 1) return MM_ERR_INVALID_ARG;
  mm::note_error("");
  if (d.T == 0) {  // no slot: empty tables (row_of_slot has no element and may be null)
    if (!counts || !offsets) return MM_ERR_INVALID_ARG;
    if (d.K > 16 || d.E > NA_MAX_E) return MM_ERR_UNSUPPORTED;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return fail("device / context", e);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((e = cudaMemsetAsync(counts, 0, (size_t)d.E * sizeof(int32_t), s)) != cudaSuccess ||
        (e = cudaMemsetAsync(offsets, 0, (size_t)(d.E + 1) * sizeof(int32_t), s)) != cudaSuccess)
      return fail("clearing the empty tables", e);
    return MM_OK;
  }
  if (!topk_ids || !counts || !offsets || !row_of_slot) return MM_ERR_INVALID_ARG;
  if (d.K > 16 || d.E > NA_MAX_E || d.T > NA_MAX_SLOTS || d.T * d.K > NA_MAX_SLOTS)
    return MM_ERR_UNSUPPORTED;  // beyond the static scratch: use mm_forward with a workspace
  const auto al4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!al4(topk_ids) || !al4(counts) || !al4(offsets) || !al4(row_of_slot))
    return MM_ERR_INVALID_ARG;
  mm_status st = MM_OK;
  int32_t* scratch = scratch_ptr(&st);
  if (st != MM_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int S = (int)(d.T * d.K), E = (int)d.E;
  const int n_chunks = (S + NA_CHUNK - 1) / NA_CHUNK;
  const unsigned grid = (unsigned)((n_chunks + 3) / 4);
  const size_t smem = 4 * (size_t)E * sizeof(int32_t);
  // the status word must start at zero; the histograms are fully rewritten by each call
  cudaError_t e = cudaMemsetAsync(scratch, 0, NA_HDR_WORDS * sizeof(int32_t), s);
  if (e != cudaSuccess) return fail("clearing the status word", e);
  k_na_count<<<grid, 128, smem, s>>>(topk_ids, scratch, S, E, n_chunks);
  if ((e = cudaGetLastError()) != cudaSuccess) return fail("count kernel launch", e);
  k_na_scan<<<1, 1024, 0, s>>>(scratch, counts, offsets, E, n_chunks);
  if ((e = cudaGetLastError()) != cudaSuccess) return fail("scan kernel launch", e);
  k_na_rank<<<grid, 128, smem, s>>>(topk_ids, scratch, row_of_slot, S, E, n_chunks);
  if ((e = cudaGetLastError()) != cudaSuccess) return fail("rank kernel launch", e);
  return MM_OK;
}
