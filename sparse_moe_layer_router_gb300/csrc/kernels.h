// kernels.h -- host-side launch functions of the libmoe_gb300 kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kPermuteChunk = 2048;  // pairs per permute block

// ---- chained launches (the kernels call griddepcontrol.wait / .launch_dependents)
// Whether launches on this host thread are chained (set per call by the entry
// points: on for batches up to 32768 (token, slot) pairs, where launch latency
// is a visible share of the step; at larger batches the early-launched grids
// measured slower).
inline bool& pdl_enabled() {
  static thread_local bool on = true;
  return on;
}
struct PdlScope {
  bool prev;
  explicit PdlScope(bool on) : prev(pdl_enabled()) { pdl_enabled() = on; }
  ~PdlScope() { pdl_enabled() = prev; }
};

template <typename... KArgs, typename... Args>
cudaError_t pdl_launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}


// ---- router (router.cu)
cudaError_t launch_router_logits_tc(const CUtensorMap& tm_w, const CUtensorMap& tm_x,
                                    const void* x, const void* wr, int T, int D, int E, int S,
                                    int kbs, float* z_part, float* xsq, float* wsq, int* status,
                                    cudaStream_t st);
cudaError_t launch_router_select(const float* z_part, int S, int T, int D, int E, int k,
                                 const float* bias, const float* xsq_part, const float* wsq_part,
                                 float gamma, float gamma2, const void* x, const void* wr,
                                 int32_t* blob, int* counters, cudaStream_t st);

// ---- dispatch (permute.cu)
// Expert ids outside [0, E) are clamped into it and, with a non-null status
// word, recorded there as MOE_ERR_INVALID_ARG.
cudaError_t launch_permute(const int32_t* blob, int T, int k, int E, int32_t* chunk_cnt,
                           int32_t* counts, int32_t* offsets, int32_t* perm_pair,
                           int32_t* inv_row, int* status, cudaStream_t st);
// out[r] = a[idx[r] / div] for every row r, or (row_lo, row_hi non-NULL: device
// pointers to two row indices) only for *row_lo <= r < *row_hi.  Source rows
// outside [0, src_rows) are clamped (and recorded as for launch_permute).
cudaError_t launch_gather_rows(const void* a, const int32_t* idx, int rows, int D, int div,
                               int src_rows, void* out, const int32_t* row_lo,
                               const int32_t* row_hi, int* status, cudaStream_t st);
// out[inv_row[t*k + j]] = x[t] for every token t < T and slot j < k (k <= 32):
// the same rows as launch_gather_rows(x, perm_pair, ...) with div = k, each x
// row read once.  Destination rows outside [0, rows) are skipped (recorded in
// status); with row_lo / row_hi only rows in [*row_lo, *row_hi) are written.
cudaError_t launch_scatter_rows(const void* x, const int32_t* inv_row, int T, int k, int D,
                                int rows, void* out, const int32_t* row_lo,
                                const int32_t* row_hi, int* status, cudaStream_t st);
// x rows in grouped order, x_perm[r] = x[perm_pair[r] / k] (with row_lo /
// row_hi only for *row_lo <= r < *row_hi): from T = kScatterMinTokens the
// token-major scatter (each x row read once; at large T the grouped rows
// would evict x from L2 between a gather's k reads of a row), below it the
// row gather (more blocks for small batches).
constexpr int kScatterMinTokens = 2048;
cudaError_t launch_dispatch_rows(const void* x, const int32_t* perm_pair, const int32_t* inv_row,
                                 int T, int k, int D, void* x_perm, const int32_t* row_lo,
                                 const int32_t* row_hi, int* status, cudaStream_t st);
// Caller index arrays made safe for the grouped GEMM: offsets_out[i] = the
// running maximum of offsets[0..i] clamped into [0, rows] (monotone, so every
// group's row range lies inside [0, rows)); perm_out[r] = perm_pair[r] clamped
// into [0, rows) (perm_pair may be NULL).  A value that needed either is
// recorded as MOE_ERR_INVALID_ARG in *status.
cudaError_t launch_sanitize_gemm_indices(const int32_t* offsets, int n_offsets, int rows,
                                         int32_t* offsets_out, const int32_t* perm_pair,
                                         int32_t* perm_out, int* status, cudaStream_t st);
// Unique ID of the CUDA context current on this thread (binding the primary
// context if none is), never reused within the process.
cudaError_t current_context_id(unsigned long long* id);
// Capacity (int32 entries) of the fixed device array behind moe_permute_static.
constexpr long kStaticPermuteScratchInts = 65536;
cudaError_t launch_permute_static(const int32_t* blob, int T, int k, int E, int32_t* counts,
                                  int32_t* offsets, int32_t* perm_pair, int32_t* inv_row,
                                  const void* x, int D, void* x_perm, cudaStream_t st);

// ---- combine (combine.cu)
// Tokens [0, T) of inv_row / o_shared / y (offset pointers give a token
// range); o has P rows (inv_row values are clamped into [0, P)).
cudaError_t launch_combine(const float* o, const float* o_shared, const int32_t* inv_row, int T,
                           int P, int D, int k, void* y, cudaStream_t st);

// Expert-parallel slice: y32[t] = (s0 <= t < s1 ? o_shared[t - s0] : 0)
//   + sum_j (*row_lo <= inv_row[t*k+j] < *row_hi ? o[inv_row[t*k+j]] : 0), fp32 out.
cudaError_t launch_combine_partial(const float* o, const float* o_shared, const int32_t* inv_row,
                                   int T, int D, int k, const int32_t* row_lo,
                                   const int32_t* row_hi, int s0, int s1, float* y32,
                                   cudaStream_t st);

// ---- int4 weight layout conversion (repack.cu)
cudaError_t launch_repack_int4(const uint32_t* src, uint32_t* dst, size_t n_words, bool offset8,
                               cudaStream_t st);

// ---- bounded-wait self-test (combine.cu)
cudaError_t launch_selftest_wait(int* status, unsigned long long limit_ns, cudaStream_t st);

// ---- grouped GEMM (grouped_gemm.cu)
enum GemmOp : int { kOpGateUp = 0, kOpDown = 1 };

// Scalar parameters of one persistent grouped-GEMM launch.  Group order for
// the tile walk: the shared group first (if any), then routed experts 0..E-1.
struct GemmParams {
  int op;
  int E;
  int has_shared;
  int T_shared;             // rows of the shared group
  const int32_t* offsets;   // [E+1] routed group row ranges
  int m_tiles, m_tiles_s;   // weight-row tiles per group (gate/up: I/64, down: D/128)
  int k_blocks, k_blocks_s; // K / 64
  int a_rows_per_expert;    // rows of one expert in the routed weight map (2I or D)
  int ld_out, ld_out_s;     // output row strides (elements)
  void* out;                // gate/up: bf16 [rows][I]; down: fp32 [rows][D]
  void* out_s;
  const int32_t* perm_pair; // down: grouped row -> pair
  const int32_t* blob;      // down: weights
  int k;
  int* status;              // workspace status word
  // W4A16 only
  const int32_t* wq;        // packed routed weights (row-major [rows][K/8])
  const uint16_t* wscale;   // routed scales [rows][K/group]
  const int32_t* wq_s;
  const uint16_t* wscale_s;
  int K, K_s;               // reduction sizes (elements)
  int group;
  int scale_table;          // W4A16: tile scales come from tm_sc / tm_sc_s by TMA
  int channel;              // W4A16: one scale per weight row ([rows]), applied in the epilogue
  int split_role;           // bf16 kernel: 0 = every group; 1 = groups of >= kSplitRows rows on
                            // the first gh CTAs; 2 = smaller groups on the last grid - gh
  const int* split_gh;      // gh, written by launch_split_plan before the split launches
};

// Groups of at least this many rows count as hot (compute-bound) when a bf16
// launch is split into a hot and a cold part.
constexpr int kSplitRows = 64;
// *gh <- the SMs (of ncta) that the hot part of a split launch of p gets.
cudaError_t launch_split_plan(const GemmParams& p, int ncta, int* gh, cudaStream_t st);

struct GemmMaps {
  CUtensorMap a, a_s, b, b_s;  // weights (routed, shared), activations (routed, shared)
  CUtensorMap sc, sc_s;        // W4A16 group scales (routed, shared)
  CUtensorMap b2, b2_s;        // bf16 kernels: activations in 32-row boxes (b, b_s: 16 rows)
  CUtensorMap b4, b4_s;        //               64-row boxes
  CUtensorMap b8, b8_s;        //               128-row boxes
};

// Kernel variants: BN_MAX token rows per tile (64 or 256); quant 0 = bf16, 1 = W4A16.
cudaError_t launch_grouped_gemm(const GemmParams& p, const GemmMaps& maps, int bn_max, int quant,
                                int num_sms, cudaStream_t st);

}  // namespace moe
