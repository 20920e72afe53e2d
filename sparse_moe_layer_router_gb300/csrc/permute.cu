// permute.cu -- dispatch: group (token, slot) pairs by expert; gather rows.
//
// "Systems engineering playbook: optimizing Qwen 3.5-397B MoE on Ironwood
// (TPU7x)", section 3, "Option B": every device filters and computes the inputs
// routed to its own experts.  On one GPU that is a stable grouping of the
// T*k pairs p = t*k + j by expert id: an expert histogram, an exclusive scan
// and a stable scatter.  All three steps are integer-exact and deterministic.
//
// Work split: pairs are cut into chunks of kChunk; chunk b counts its experts
// (count kernel), one block turns the [chunks][E] table into per-chunk base
// positions plus counts/offsets (scan kernel), and each chunk places its pairs
// in order (scatter kernel: per-warp segments, __match_any_sync for ranks
// within a step of 32).
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// Expert id of pair p.  An id outside [0, E) (a blob that moe_route did not
// write) sets `bad` and is clamped to the nearest valid expert, so that every
// count, offset and position stays in bounds; the caller records the error.
__device__ __forceinline__ int pair_expert(const int32_t* __restrict__ blob, int k, int E, int p,
                                           bool& bad) {
  const int t = p / k, j = p - t * k;
  const int e = blob[static_cast<size_t>(t) * 2 * k + j];
  if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) return e;
  bad = true;
  return e < 0 ? 0 : E - 1;
}

__device__ __forceinline__ void report_invalid(bool bad, int* status) {
  if (bad && status) atomicCAS(status, 0, MOE_ERR_INVALID_ARG);
}

__global__ void __launch_bounds__(256) permute_count_kernel(const int32_t* __restrict__ blob,
                                                            int P, int k, int E,
                                                            int32_t* __restrict__ chunk_cnt,
                                                            int* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kPermuteChunk;
  const int p1 = min(P, p0 + kPermuteChunk);
  bool bad = false;
  for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x)
    atomicAdd(&hist[pair_expert(blob, k, E, p, bad)], 1);
  report_invalid(bad, status);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_cnt[static_cast<size_t>(blockIdx.x) * E + e] = hist[e];
}

// One block of 1024 threads.  On exit chunk_cnt[b][e] holds the first grouped
// row of chunk b's pairs for expert e.
__global__ void __launch_bounds__(1024) permute_scan_kernel(int32_t* __restrict__ chunk_cnt,
                                                            int B, int E,
                                                            int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ offsets) {
  pdl_wait();
  pdl_trigger();
  __shared__ int warp_sums[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int e0 = 0; e0 < E; e0 += 1024) {
    const int e = e0 + threadIdx.x;
    int total = 0;
    if (e < E) {
      for (int b = 0; b < B; ++b) {
        const size_t i = static_cast<size_t>(b) * E + e;
        const int c = chunk_cnt[i];
        chunk_cnt[i] = total;
        total += c;
      }
      counts[e] = total;
    }
    // block-wide exclusive scan of `total` over e
    int incl = total;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      int s = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += n;
      }
      warp_sums[lane] = s;  // inclusive over warps
    }
    __syncthreads();
    const int excl = carry + (wid ? warp_sums[wid - 1] : 0) + incl - total;
    if (e < E) {
      offsets[e] = excl;
      for (int b = 0; b < B; ++b) chunk_cnt[static_cast<size_t>(b) * E + e] += excl;
    }
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_sums[31];
    __syncthreads();
  }
  if (threadIdx.x == 0) offsets[E] = carry;
}

// 256 threads = 8 warps; warp w owns pairs [p0 + w*seg, p0 + (w+1)*seg) of the chunk.
__global__ void __launch_bounds__(256) permute_scatter_kernel(
    const int32_t* __restrict__ blob, int P, int k, int E, const int32_t* __restrict__ chunk_base,
    int32_t* __restrict__ perm_pair, int32_t* __restrict__ inv_row) {
  bool bad = false;  // reported by the count kernel
  pdl_wait();
  pdl_trigger();
  extern __shared__ int wcnt[];  // [8][E]
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 8 * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  constexpr int seg = kPermuteChunk / 8;
  const int p0 = blockIdx.x * kPermuteChunk + wid * seg;
  const int p1 = min(P, p0 + seg);
  for (int p = p0 + lane; p < p1; p += 32)
    atomicAdd(&wcnt[wid * E + pair_expert(blob, k, E, p, bad)], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = chunk_base[static_cast<size_t>(blockIdx.x) * E + e];
    for (int w = 0; w < 8; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  int* my = wcnt + wid * E;
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int pb = p0; pb < p1; pb += 32) {
    const int p = pb + lane;
    const bool valid = p < p1;
    const int e = valid ? pair_expert(blob, k, E, p, bad) : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int pos = 0;
    if (valid) pos = my[e] + __popc(peers & lt_mask);
    __syncwarp();
    if (valid && (peers & lt_mask) == 0) my[e] += __popc(peers);
    __syncwarp();
    if (valid) {
      perm_pair[pos] = p;
      inv_row[p] = pos;
    }
  }
}

// out[r][:] = a[idx[r] / div][:]  (D bf16 per row, 16-byte vectors); with a
// row range (device pointers row_lo, row_hi) only for *row_lo <= r < *row_hi.
// A source row outside [0, src_rows) is clamped into it and recorded in
// `status` (MOE_ERR_INVALID_ARG) when that is non-null.
// One warp per row, kGatherRowsPerBlock rows per block; each lane issues
// eight 16-byte loads before its stores, so a block keeps 32 KB in flight.
constexpr int kGatherRowsPerBlock = 8;
__global__ void __launch_bounds__(32 * kGatherRowsPerBlock) gather_rows_kernel(
    const uint4* __restrict__ a, const int32_t* __restrict__ idx, int rows, int vec_per_row,
    int div, int src_rows, uint4* __restrict__ out, const int32_t* __restrict__ row_lo,
    const int32_t* __restrict__ row_hi, int* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kGatherRowsPerBlock + (threadIdx.x >> 5);
  if (r >= rows) return;
  if (row_lo && (r < __ldg(row_lo) || r >= __ldg(row_hi))) return;
  int src = idx[r] / div;
  if (static_cast<unsigned>(src) >= static_cast<unsigned>(src_rows)) {
    if (lane == 0 && status) atomicCAS(status, 0, MOE_ERR_INVALID_ARG);
    src = src < 0 ? 0 : src_rows - 1;
  }
  const uint4* sr = a + static_cast<size_t>(src) * vec_per_row;
  uint4* dr = out + static_cast<size_t>(r) * vec_per_row;
  for (int i0 = 0; i0 < vec_per_row; i0 += 8 * 32) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + 32 * u + lane;
      if (i < vec_per_row) v[u] = __ldg(sr + i);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + 32 * u + lane;
      if (i < vec_per_row) dr[i] = v[u];
    }
  }
}

// Token-major form of the same copy: one warp per token reads its x row once
// and writes it to the k grouped rows inv_row[t*k + j], so each x row crosses
// HBM once (a row-major gather reads it k times, and at large T the grouped
// rows streaming through L2 evict x between those reads).  Destination rows
// outside [0, rows) are skipped and recorded; with row_lo / row_hi only rows
// in [*row_lo, *row_hi) are written.
constexpr int kScatterTokensPerBlock = 8;
__global__ void __launch_bounds__(32 * kScatterTokensPerBlock) scatter_rows_kernel(
    const uint4* __restrict__ x, const int32_t* __restrict__ inv_row, int T, int k,
    int vec_per_row, int rows, uint4* __restrict__ out, const int32_t* __restrict__ row_lo,
    const int32_t* __restrict__ row_hi, int* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kScatterTokensPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  const int lo = row_lo ? __ldg(row_lo) : 0;
  const int hi = row_hi ? __ldg(row_hi) : rows;
  // lane j < k holds destination j
  int dst = lane < k ? __ldg(inv_row + static_cast<size_t>(t) * k + lane) : -1;
  if (lane < k && static_cast<unsigned>(dst) >= static_cast<unsigned>(rows)) {
    if (status) atomicCAS(status, 0, MOE_ERR_INVALID_ARG);
    dst = -1;
  }
  if (dst < lo || dst >= hi) dst = -1;
  const uint4* sr = x + static_cast<size_t>(t) * vec_per_row;
  for (int i0 = 0; i0 < vec_per_row; i0 += 8 * 32) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + 32 * u + lane;
      if (i < vec_per_row) v[u] = __ldg(sr + i);
    }
    for (int j = 0; j < k; ++j) {
      const int r = __shfl_sync(0xffffffffu, dst, j);
      if (r < 0) continue;
      uint4* dr = out + static_cast<size_t>(r) * vec_per_row;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + 32 * u + lane;
        if (i < vec_per_row) dr[i] = v[u];
      }
    }
  }
}

// Small problems in one block of 1024 threads (one launch instead of three):
// warp w owns pairs [w*seg, (w+1)*seg); per-warp expert counts in shared
// memory, one block-wide scan over experts, then each warp places its pairs
// in order exactly as permute_scatter_kernel does.  Same results.
constexpr int kPermuteOneBlockMaxPairs = 4096;
__global__ void __launch_bounds__(1024) permute_one_block_kernel(
    const int32_t* __restrict__ blob, int P, int k, int E, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ perm_pair, int32_t* __restrict__ inv_row,
    int* __restrict__ status) {
  bool bad = false;
  pdl_wait();
  pdl_trigger();
  extern __shared__ int wc[];  // [32][E], then [32] warp sums
  int* warp_sums = wc + 32 * E;
  __shared__ int carry;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wc[i] = 0;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int seg = (P + 31) / 32;
  const int p0 = wid * seg, p1 = min(P, p0 + seg);
  for (int p = p0 + lane; p < p1; p += 32) atomicAdd(&wc[wid * E + pair_expert(blob, k, E, p, bad)], 1);
  report_invalid(bad, status);
  __syncthreads();
  for (int e0 = 0; e0 < E; e0 += 1024) {
    const int e = e0 + threadIdx.x;
    int total = 0;
    if (e < E)
      for (int w = 0; w < 32; ++w) total += wc[w * E + e];
    int incl = total;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      int v = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
      }
      warp_sums[lane] = v;
    }
    __syncthreads();
    const int excl = carry + (wid ? warp_sums[wid - 1] : 0) + incl - total;
    if (e < E) {
      counts[e] = total;
      offsets[e] = excl;
      int run = excl;
      for (int w = 0; w < 32; ++w) {
        const int c = wc[w * E + e];
        wc[w * E + e] = run;
        run += c;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_sums[31];
    __syncthreads();
  }
  if (threadIdx.x == 0) offsets[E] = carry;
  int* my = wc + wid * E;
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int pb = p0; pb < p1; pb += 32) {
    const int p = pb + lane;
    const bool valid = p < p1;
    const int e = valid ? pair_expert(blob, k, E, p, bad) : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int pos = 0;
    if (valid) pos = my[e] + __popc(peers & lt_mask);
    __syncwarp();
    if (valid && (peers & lt_mask) == 0) my[e] += __popc(peers);
    __syncwarp();
    if (valid) {
      perm_pair[pos] = p;
      inv_row[p] = pos;
    }
  }
}

// Offsets for the grouped GEMM from a caller: one warp; lane i takes a
// contiguous chunk, clamps it into [0, rows] and keeps the running maximum
// (a warp max-scan carries it across chunks), so the copy is monotone.
__global__ void __launch_bounds__(32) sanitize_offsets_kernel(const int32_t* __restrict__ in,
                                                              int n, int rows,
                                                              int32_t* __restrict__ out,
                                                              int* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x;
  const int chunk = (n + 31) / 32;
  const int i0 = lane * chunk, i1 = min(n, i0 + chunk);
  bool bad = false;
  int run = 0;
  for (int i = i0; i < i1; ++i) {
    const int v = in[i];
    const int c = min(max(v, 0), rows);
    bad |= c != v || c < run;
    run = max(run, c);
  }
  int incl = run;  // max over chunks 0..lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int m = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl = max(incl, m);
  }
  int prev = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) prev = 0;
  // a chunk that starts below the previous chunks' maximum is a decrease too
  if (i0 < i1) bad |= min(max(in[i0], 0), rows) < prev;
  run = prev;
  for (int i = i0; i < i1; ++i) {
    run = max(run, min(max(in[i], 0), rows));
    out[i] = run;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0 && status)
    atomicCAS(status, 0, MOE_ERR_INVALID_ARG);
}

// out[i] = in[i] clamped into [0, hi), recording any change.
__global__ void __launch_bounds__(256) clamp_rows_kernel(const int32_t* __restrict__ in, int n,
                                                         int hi, int32_t* __restrict__ out,
                                                         int* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  bool bad = false;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int v = in[i];
    const bool ok = static_cast<unsigned>(v) < static_cast<unsigned>(hi);
    bad |= !ok;
    out[i] = ok ? v : (v < 0 ? 0 : hi - 1);
  }
  report_invalid(bad, status);
}

cudaError_t launch_sanitize_gemm_indices(const int32_t* offsets, int n_offsets, int rows,
                                         int32_t* offsets_out, const int32_t* perm_pair,
                                         int32_t* perm_out, int* status, cudaStream_t st) {
  cudaError_t e = pdl_launch(sanitize_offsets_kernel, dim3(1), dim3(32), 0, st, offsets,
                             n_offsets, rows, offsets_out, status);
  if (e != cudaSuccess || !perm_pair) return e;
  const int blocks = min((rows + 255) / 256, 1024);
  return pdl_launch(clamp_rows_kernel, dim3(blocks), dim3(256), 0, st, perm_pair, rows, rows,
                    perm_out, status);
}

cudaError_t launch_permute(const int32_t* blob, int T, int k, int E, int32_t* chunk_cnt,
                           int32_t* counts, int32_t* offsets, int32_t* perm_pair,
                           int32_t* inv_row, int* status, cudaStream_t st) {
  const int P = T * k;
  const size_t smem_one = (static_cast<size_t>(32) * E + 32) * sizeof(int);
  if (P <= kPermuteOneBlockMaxPairs && smem_one <= 200 * 1024) {
    if (smem_one > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(permute_one_block_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem_one));
      if (e != cudaSuccess) return e;
    }
    return pdl_launch(permute_one_block_kernel, dim3(1), dim3(1024), smem_one, st, blob, P, k, E,
                      counts, offsets, perm_pair, inv_row, status);
  }
  const int B = (P + kPermuteChunk - 1) / kPermuteChunk;
  const size_t smem_count = static_cast<size_t>(E) * sizeof(int);
  const size_t smem_scatter = static_cast<size_t>(8) * E * sizeof(int);
  if (smem_scatter > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(permute_scatter_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_scatter));
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = pdl_launch(permute_count_kernel, dim3(B), dim3(256), smem_count, st, blob, P, k,
                             E, chunk_cnt, status);
  if (e != cudaSuccess) return e;
  e = pdl_launch(permute_scan_kernel, dim3(1), dim3(1024), 0, st, chunk_cnt, B, E, counts, offsets);
  if (e != cudaSuccess) return e;
  return pdl_launch(permute_scatter_kernel, dim3(B), dim3(256), smem_scatter, st, blob, P, k, E,
                    chunk_cnt, perm_pair, inv_row);
}

cudaError_t launch_scatter_rows(const void* x, const int32_t* inv_row, int T, int k, int D,
                                int rows, void* out, const int32_t* row_lo,
                                const int32_t* row_hi, int* status, cudaStream_t st) {
  const int blocks = (T + kScatterTokensPerBlock - 1) / kScatterTokensPerBlock;
  return pdl_launch(scatter_rows_kernel, dim3(blocks), dim3(32 * kScatterTokensPerBlock), 0, st,
                    static_cast<const uint4*>(x), inv_row, T, k, D / 8, rows,
                    static_cast<uint4*>(out), row_lo, row_hi, status);
}

cudaError_t launch_dispatch_rows(const void* x, const int32_t* perm_pair, const int32_t* inv_row,
                                 int T, int k, int D, void* x_perm, const int32_t* row_lo,
                                 const int32_t* row_hi, int* status, cudaStream_t st) {
  if (T >= kScatterMinTokens)
    return launch_scatter_rows(x, inv_row, T, k, D, T * k, x_perm, row_lo, row_hi, status, st);
  return launch_gather_rows(x, perm_pair, T * k, D, k, T, x_perm, row_lo, row_hi, status, st);
}

cudaError_t launch_gather_rows(const void* a, const int32_t* idx, int rows, int D, int div,
                               int src_rows, void* out, const int32_t* row_lo,
                               const int32_t* row_hi, int* status, cudaStream_t st) {
  const int blocks = (rows + kGatherRowsPerBlock - 1) / kGatherRowsPerBlock;
  return pdl_launch(gather_rows_kernel, dim3(blocks), dim3(32 * kGatherRowsPerBlock), 0, st,
                    static_cast<const uint4*>(a), idx, rows, D / 8, div, src_rows,
                    static_cast<uint4*>(out), row_lo, row_hi, status);
}

// ------------------------------------------------------------------
// Fixed scratch for moe_permute_static: the [chunks][E] count table lives in
// this file-scope device array (kStaticPermuteScratchInts int32 = 256 KiB)
// instead of a caller-provided workspace.  Every device (every context) that
// loads the library holds it until the process exits.  Each call overwrites
// the entries it uses before reading them, so nothing needs clearing; calls
// that overlap on the GPU share the array and race.
static __device__ __align__(256) int32_t g_permute_scratch[kStaticPermuteScratchInts];

namespace {
// The device address of g_permute_scratch belongs to a CUDA context, not to a
// device: a reset primary context or another context made current on the same
// device (cuCtxCreate) has its own copy of the array at another address.  The
// address is therefore cached per context, keyed by the context's unique ID
// (cuCtxGetId: never reused within the process, unlike a context handle).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
struct ScratchEntry {
  unsigned long long ctx_id;
  int32_t* addr;
};
constexpr int kScratchCache = 32;
std::mutex g_scratch_mu;
ScratchEntry g_scratch_cache[kScratchCache] = {};
int g_scratch_used = 0, g_scratch_next = 0;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

template <typename Fn>
bool driver_fn(const char* name, Fn* out) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  *out = reinterpret_cast<Fn>(fn);
  return true;
}

// ID of the context current on this thread, binding the runtime's primary
// context first if none is current.  Called with g_scratch_mu held.
cudaError_t current_ctx_id(unsigned long long* id) {
  if (!g_ctx_get_current && (!driver_fn("cuCtxGetCurrent", &g_ctx_get_current) ||
                             !driver_fn("cuCtxGetId", &g_ctx_get_id)))
    return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
  if (!ctx) {
    // no context yet: a runtime call that needs one binds the primary context
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess) return e;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorUnknown;
  }
  return g_ctx_get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}
}  // namespace

cudaError_t current_context_id(unsigned long long* id) {
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  return current_ctx_id(id);
}

// Device address of g_permute_scratch in the current context.  In host code
// the symbol names a host-side stand-in, so the address is looked up with the
// runtime (once per context, with that context current) and cached.
static cudaError_t static_scratch(int32_t** out) {
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  unsigned long long id = 0;
  cudaError_t e = current_ctx_id(&id);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < g_scratch_used; ++i)
    if (g_scratch_cache[i].ctx_id == id) {
      *out = g_scratch_cache[i].addr;
      return cudaSuccess;
    }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_permute_scratch);
  if (e != cudaSuccess) return e;
  int i = 0;
  if (g_scratch_used < kScratchCache) {
    i = g_scratch_used++;
  } else {  // full: replace the oldest entry
    i = g_scratch_next;
    g_scratch_next = (g_scratch_next + 1) % kScratchCache;
  }
  ScratchEntry& slot = g_scratch_cache[i];
  slot.ctx_id = id;
  slot.addr = static_cast<int32_t*>(p);
  *out = slot.addr;
  return cudaSuccess;
}

cudaError_t launch_permute_static(const int32_t* blob, int T, int k, int E, int32_t* counts,
                                  int32_t* offsets, int32_t* perm_pair, int32_t* inv_row,
                                  const void* x, int D, void* x_perm, cudaStream_t st) {
  int32_t* table = nullptr;
  cudaError_t e = static_scratch(&table);
  if (e != cudaSuccess) return e;
  e = launch_permute(blob, T, k, E, table, counts, offsets, perm_pair, inv_row, nullptr, st);
  if (e != cudaSuccess || !x) return e;
  return launch_dispatch_rows(x, perm_pair, inv_row, T, k, D, x_perm, nullptr, nullptr, nullptr,
                              st);
}

}  // namespace moe
