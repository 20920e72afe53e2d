// grouped_gemm.cu -- persistent grouped GEMM over ragged expert row groups (sm_103a).
//
// "Systems engineering playbook: optimizing Qwen 3.5-397B MoE on Ironwood
// (TPU7x)", executive summary: grouped GEMM is one of the reusable building
// blocks; section 1 "Sparse Mixture-of-Experts (MoE)": each routed expert and
// the always-on shared expert is a SwiGLU FFN.  "vLLM TPU Inference v0.31.0:
// hierarchical MoE dispatch and W4A16": the expert-parallel grouped-matmul
// (GMM) path, and int4 weights that stay packed in HBM and are restored tile by
// tile on chip.
//
// Design (one CTA per SM, persistent, warp-specialised):
//   * A tile = 128 weight rows x 64 K (bf16, 128-byte swizzle), B tile = up to
//     BN_MAX token rows x 64 K.  The MMA is "swap-AB": weights are the M = 128
//     operand, tokens the N operand (16..BN_MAX, multiple of 16), so a group
//     with few tokens still streams full-width weight tiles.
//   * warp 0: TMA producer (one thread); warp 1: TMEM allocation and
//     tcgen05.mma issue (one thread), fp32 accumulators in TMEM, double
//     buffered; warps 2-5: epilogue (tcgen05.ld; warps 2-9 in the bf16
//     kernel, two per TMEM lane quarter).  The W4A16 kernels add
//     dequant warps that restore the packed int4 tiles (into the shared-memory
//     operand for 256-row token tiles, into tensor memory for tiles of up to 64
//     rows) and a token-row producer warp; the TMEM variant has a second MMA
//     warp.
//   * Tiles: every CTA walks tile indices blockIdx.x, +gridDim.x, ... over the
//     concatenation of groups [shared, expert 0, ..., expert E-1]; a group with
//     R rows has ceil(R / BN_MAX) * m_tiles tiles, token tiles of one weight
//     tile adjacent so repeated weight tiles come from L2.  A split bf16
//     launch runs as two grids, each walking only its own groups (those of
//     at least kSplitRows rows, or the smaller ones) on its share of the SMs.
//   * Gate/up: a tile covers 64 output features; its A rows are four blocks of
//     (16 gate rows, 16 up rows) (one 4-D TMA box for bf16, four 3-D boxes for
//     int4), so each epilogue warp holds gate and up of the same 16 features in
//     its TMEM lanes and forms h = silu(g) * u with one lane exchange (no
//     shared memory, no barrier).
//   * Down: a tile covers 128 output features; the epilogue multiplies by the
//     routing weight of the row's (token, slot) pair and stores fp32.
//   * Every wait is bounded (2 s); on expiry the CTA records MOE_ERR_TIMEOUT,
//     stops issuing, waits for its copies and MMAs in flight and frees TMEM.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kAStage = kBM * kBK * 2;  // 16 KB bf16 operand tile
constexpr int kMaxGroups = 1025;
constexpr int kBaseThreads = 192;       // producer, MMA, 4 epilogue warps
// The bf16 kernel runs 8 epilogue warps (two per TMEM lane quarter, each
// taking every other 16-column chunk): its epilogue writes a tile's outputs
// while the next tile's MMAs run, and with 256 token columns and fp32 outputs
// four warps could not keep up.
constexpr int kBf16EpiWarps = 8;
constexpr int kBf16Threads = 64 + 32 * kBf16EpiWarps;

// W4A16: packed stages of 128 rows x 128 B (256 int4 values = 4 k-blocks).
// Shared-memory variant: two dequant groups of four warps (one tile row per
// thread); group g restores k-blocks 4q + g and 4q + 2 + g of packed stage q
// into its two operand buffers 2g and 2g + 1, so it restores one while the MMA
// reads the other.
constexpr int kPackedK = 256;
constexpr int kPackedStage = kBM * kPackedK / 2;  // 16 KB
constexpr int kKPerPacked = kPackedK / kBK;       // 4 k-blocks per packed stage
constexpr int kABuffers = 4;
constexpr int kDequantGroups = 2;
constexpr int kWarpsPerGroup = 4;
constexpr int kDequantWarps = kDequantGroups * kWarpsPerGroup;
constexpr int kTokenWarp = 6 + kDequantWarps;  // W4A16: separate producer for token tiles
constexpr int kW4Threads = kBaseThreads + 32 * kDequantWarps + 32;
constexpr int kScaleTabElems = kBM * 32;  // one tile's scales for K <= 4096
// W4A16 scale group along K.  The host accepts group 128 or channel-wise
// scales only, so the kernels divide by a constant (a power of two) instead
// of a run-time value.
constexpr int kGroup = 128;

struct TileInfo {
  int shared;
  int e;
  int m;
  int n_valid;
  int bn;
  int b_row;
  int k_blocks;
  int n_tiles;  // token tiles of the group: each weight tile is read this many times
};

// Shared-memory parts common to both kernels.
template <int BN_MAX>
struct GemmCommon {
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int tile_start[kMaxGroups + 1];
  int off[kMaxGroups];
  float row_weight[8][BN_MAX];  // down epilogue: routing weight of each token row, per warp
  int walk_ctas;                // bf16 kernel: CTAs that share the tile walk
};

template <int BN_MAX, int STAGES>
struct Bf16Smem {
  uint8_t a[STAGES][kAStage];       // weights, 128-B swizzle
  uint8_t b[STAGES][BN_MAX * 128];  // token rows, 128-B swizzle
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  GemmCommon<BN_MAX> c;
};

template <int BN_MAX, int PSTAGES, int BSTAGES>
struct W4Smem {
  uint8_t a[kABuffers][kAStage];        // restored bf16 operand, two per dequant group
  uint8_t b[BSTAGES][BN_MAX * 128];     // token rows per k-block
  uint8_t praw[PSTAGES][kPackedStage];  // packed int4 rows, 128-B swizzle
  uint16_t stab[2][kScaleTabElems];     // group scales of the current tiles
  uint64_t pfull[PSTAGES], pempty[PSTAGES];
  uint64_t bfull[BSTAGES], bempty[BSTAGES];
  uint64_t aready[kABuffers], afree[kABuffers];
  uint64_t sfull[2], sempty[2];
  GemmCommon<BN_MAX> c;
};

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void record_error(const GemmParams& p, volatile int* abort_flag,
                                             int code) {
  *abort_flag = 1;
  if (p.status) atomicCAS(p.status, 0, code);
}

template <int BN_MAX>
__device__ __forceinline__ TileInfo decode_tile(const GemmCommon<BN_MAX>& s, const GemmParams& p,
                                                int G, int L) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.tile_start[mid] <= L)
      lo = mid;
    else
      hi = mid;
  }
  TileInfo t;
  const int l = L - s.tile_start[lo];
  t.shared = p.has_shared && lo == 0;
  t.e = lo - p.has_shared;
  const int rows = t.shared ? p.T_shared : s.off[t.e + 1] - s.off[t.e];
  const int row0 = t.shared ? 0 : s.off[t.e];
  const int n_tiles = (rows + BN_MAX - 1) / BN_MAX;
  t.n_tiles = n_tiles;
  t.m = l / n_tiles;
  const int n = l - t.m * n_tiles;
  t.n_valid = min(BN_MAX, rows - n * BN_MAX);
  t.bn = (t.n_valid + 15) & ~15;
  t.b_row = row0 + n * BN_MAX;
  t.k_blocks = t.shared ? p.k_blocks_s : p.k_blocks;
  return t;
}

// First weight row of a tile in its weight map (routed maps stack experts).
__device__ __forceinline__ int tile_a_row(const GemmParams& p, const TileInfo& t) {
  return (t.shared ? 0 : t.e * p.a_rows_per_expert) + t.m * (p.op == kOpGateUp ? 64 : kBM);
}

// Weight row (in the full weight matrix of its group) held by row r of a tile.
// Gate/up tiles hold four blocks of (16 gate rows, 16 up rows) of features
// m*64 .. m*64+63; down tiles hold rows m*128 .. m*128+127.
__device__ __forceinline__ int tile_weight_row(const GemmParams& p, const TileInfo& t, int r) {
  if (p.op == kOpGateUp) {
    const int half = t.shared ? p.ld_out_s : p.ld_out;  // I of the group
    const int b = r >> 5, j = r & 31;
    const int f = t.m * 64 + 16 * b + (j & 15);
    const int base = t.shared ? 0 : t.e * p.a_rows_per_expert;
    return base + (j < 16 ? f : half + f);
  }
  return (t.shared ? 0 : t.e * p.a_rows_per_expert) + t.m * kBM + r;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

// Eight signed 4-bit values in pair order (value 2i in bits 4i..4i+3, value
// 2i+1 in bits 16+4i..19+4i) times a bf16 scale -> eight bf16 in order, each
// bf16_rne(q * s).  One shift and mask put the nibbles of values 2i, 2i+1 in
// the low bits of the two halves; XOR with 8 makes them offset binary (q + 8)
// and 0x4300 | u is the bf16 of 128 + u (exact); subtracting 136 (exact) and
// multiplying by the scale (one rounding) gives the pair, already in order.
// The 0x4300 | u step is the classic magic-number integer-to-float
// conversion (an integer placed in the mantissa of a float whose exponent is
// fixed, the float of the offset then subtracted), the method low-bit
// weight-only kernels use to dequantise, e.g. Kim et al., "Who Says Elephants
// Can't Run: Bringing Large Scale MoE Models into Cloud Scale Production"
// (2022).
// kScale = false (channel-wise scales, applied in the epilogue): the exact q.
template <bool kScale = true>
__device__ __forceinline__ uint4 dequant_word(uint32_t w, __nv_bfloat162 s2) {
  const __nv_bfloat162 k136 = __floats2bfloat162_rn(136.0f, 136.0f);
  uint32_t h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t t = ((w >> (4 * i)) & 0x000F000Fu) ^ 0x43084308u;
    __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&t), k136);
    if (kScale) q = __hmul2(q, s2);
    h[i] = *reinterpret_cast<const uint32_t*>(&q);
  }
  return make_uint4(h[0], h[1], h[2], h[3]);
}

// Eight values of a packed word: scaled (group scales) or exact q (channel).
__device__ __forceinline__ uint4 restore_word(uint32_t w, __nv_bfloat162 s2, bool channel) {
  return channel ? dequant_word<false>(w, s2) : dequant_word<true>(w, s2);
}

// Group table: s.off <- offsets, s.tile_start <- exclusive scan of tiles per
// group; returns the number of tiles.  All threads of the CTA call it.  With
// kFilter, groups whose row count lies outside [min_rows, max_rows] get none.
template <int BN_MAX, bool kFilter = false>
__device__ int build_tile_table(GemmCommon<BN_MAX>& s, const GemmParams& p, int G, int nthreads,
                                int min_rows = 0, int max_rows = 0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i <= p.E; i += nthreads) s.off[i] = p.offsets[i];
  __syncthreads();
  for (int g = threadIdx.x; g < G; g += nthreads) {
    const bool sh = p.has_shared && g == 0;
    const int e = g - p.has_shared;
    int rows = sh ? p.T_shared : s.off[e + 1] - s.off[e];
    if (kFilter && (rows < min_rows || rows > max_rows)) rows = 0;
    s.tile_start[g + 1] = ((rows + BN_MAX - 1) / BN_MAX) * (sh ? p.m_tiles_s : p.m_tiles);
  }
  __syncthreads();
  if (warp == 0) {
    const int chunk = (G + 31) / 32;
    const int g0 = lane * chunk, g1 = min(G, g0 + chunk);
    int sum = 0;
    for (int g = g0; g < g1; ++g) sum += s.tile_start[g + 1];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int run = incl - sum;
    for (int g = g0; g < g1; ++g) {
      run += s.tile_start[g + 1];
      s.tile_start[g + 1] = run;
    }
    if (lane == 0) s.tile_start[0] = 0;
  }
  __syncthreads();
  return s.tile_start[G];
}

template <int BN_MAX>
__device__ __forceinline__ void init_common_barriers(GemmCommon<BN_MAX>& c, int epi_warps = 4) {
  for (int i = 0; i < 2; ++i) {
    mbar_init(&c.tfull[i], 1);
    mbar_init(&c.tempty[i], epi_warps);
  }
  mbar_init(&c.drain, 1);
  c.abort_flag = 0;
}

// Epilogue role (warps 2 .. 1+NE): TMEM accumulators -> h (SwiGLU, bf16) or o
// (routing-weighted, fp32).  With NP = 2 the accumulator is the sum of two
// partial accumulators 2 * BN_MAX columns apart (two MMA issuers).  With
// NE = 8 two warps share each TMEM lane quarter and take alternate 16-column
// chunks.
template <int BN_MAX, int NP = 1, bool kSleep = false, int NE = 4>
__device__ void epilogue_role(GemmCommon<BN_MAX>& s, const GemmParams& p, int G, int ntiles,
                              uint32_t tmem_base, volatile int* abort_flag, int warp, int lane) {
  static_assert(NE == 4 || NE == 8, "one or two warps per TMEM lane quarter");
  const int sp = warp & 3;  // TMEM lanes 32*sp .. 32*sp+31
  const int c_first = 16 * ((warp - 2) / 4);  // first 16-column chunk of this warp
  constexpr int c_step = 16 * (NE / 4);
  float* wts = s.row_weight[warp - 2];
  int acc = 0;
  uint32_t acc_phase = 0;
  // the bf16 kernel's walk may be a share of the grid (split launches)
  const int step = NE == 8 ? s.walk_ctas : static_cast<int>(gridDim.x);
  for (int L = blockIdx.x; L < ntiles; L += step) {
    const TileInfo t = decode_tile<BN_MAX>(s, p, G, L);
    if (p.op == kOpDown) {
      // Routing weight of every token row of the tile, fetched before the
      // accumulator is ready: row r holds pair p = perm_pair[r] (token p / k,
      // slot p % k); the shared group has weight 1.
      __syncwarp();
      if constexpr (NE == 8) {
        // The bf16 kernel: every lane issues all its perm_pair loads, then all
        // its blob loads, so a 256-row tile waits for two memory latencies
        // rather than two per row (with one loop iteration per row this chain
        // outlasted the tile's MMAs at T = 8192).  The W4A16 kernels keep the
        // loop below: the unrolled form cost them 4-6%.
        constexpr int kPer = BN_MAX / 32;
        int prs[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int j = lane + 32 * u;
          prs[u] = (!t.shared && j < t.n_valid) ? __ldg(p.perm_pair + t.b_row + j) : 0;
        }
        float wv[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int j = lane + 32 * u;
          wv[u] = 1.0f;
          if (!t.shared && j < t.n_valid) {
            const int pr = prs[u];
            const int tk = pr / p.k;
            wv[u] = __int_as_float(
                __ldg(p.blob + static_cast<size_t>(tk) * 2 * p.k + p.k + (pr - tk * p.k)));
          }
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int j = lane + 32 * u;
          if (j < t.n_valid) wts[j] = wv[u];
        }
      } else {
        for (int j = lane; j < t.n_valid; j += 32) {
          float wgt = 1.0f;
          if (!t.shared) {
            const int pr = __ldg(p.perm_pair + t.b_row + j);
            const int tk = pr / p.k;
            wgt = __int_as_float(
                __ldg(p.blob + static_cast<size_t>(tk) * 2 * p.k + p.k + (pr - tk * p.k)));
          }
          wts[j] = wgt;
        }
      }
      __syncwarp();
    }
    if (!mbar_wait<kSleep>(&s.tfull[acc], acc_phase, abort_flag)) {
      record_error(p, abort_flag, MOE_ERR_TIMEOUT);
      break;
    }
    tc_fence_after();
    const uint32_t tbase =
        tmem_base + static_cast<uint32_t>(acc * BN_MAX) + (static_cast<uint32_t>(sp * 32) << 16);
    // Channel-wise W4A16 scales: this lane's accumulator row is weight row
    // tile_weight_row(32 * sp + lane); its scale multiplies the exact-q sums.
    float row_scale = 1.0f;
    if (p.channel) {
      const uint16_t* sc = t.shared ? p.wscale_s : p.wscale;
      row_scale = bf16_bits_to_float(__ldg(sc + tile_weight_row(p, t, 32 * sp + lane)));
    }
    for (int c0 = c_first; c0 < t.bn; c0 += c_step) {
      uint32_t r[16];
      tmem_ld_32x32b_x16(tbase + static_cast<uint32_t>(c0), r);
      if (NP == 2) {
        uint32_t r2[16];
        tmem_ld_32x32b_x16(tbase + static_cast<uint32_t>(2 * BN_MAX + c0), r2);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
      } else {
        tmem_wait_ld();
      }
      if (p.channel) {
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * row_scale);
      }
      if (p.op == kOpGateUp) {
        // lanes 0-15 hold gate rows, lanes 16-31 the up rows of the same 16
        // features; lane < 16 finishes columns 0-7 of the chunk, lane >= 16
        // columns 8-15.
        const bool hi = lane >= 16;
        float h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t send = hi ? r[i] : r[i + 8];
          const float other = __uint_as_float(__shfl_xor_sync(0xffffffffu, send, 16));
          const float g = hi ? other : __uint_as_float(r[i]);
          const float u = hi ? __uint_as_float(r[i + 8]) : other;
          h[i] = silu_f(g) * u;
        }
        const int f = t.m * 64 + 16 * sp + (lane & 15);
        const int cbase = c0 + (hi ? 8 : 0);
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(t.shared ? p.out_s : p.out);
        const int ld = t.shared ? p.ld_out_s : p.ld_out;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int col = cbase + i;
          if (col < t.n_valid)
            out[static_cast<size_t>(t.b_row + col) * ld + f] = __float2bfloat16_rn(h[i]);
        }
      } else {
        const int f = t.m * kBM + sp * 32 + lane;
        float* out = static_cast<float*>(t.shared ? p.out_s : p.out);
        const int ld = t.shared ? p.ld_out_s : p.ld_out;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int col = c0 + i;
          if (col < t.n_valid)
            out[static_cast<size_t>(t.b_row + col) * ld + f] = wts[col] * __uint_as_float(r[i]);
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.tempty[acc]);
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
}

// Token tile of k-block kb from maps whose boxes are 16, 32, 64 and 128 rows
// high (mb[0..3]): bn (a multiple of 16) is cut into its binary parts, largest
// first, so a tile takes at most four copies (two for bn = 256).  Issuing a
// copy holds the issuing thread for a few hundred cycles.
__device__ __forceinline__ void load_token_tile_p2(uint8_t* dst, const CUtensorMap* const* mb,
                                                   uint64_t* bar, const TileInfo& t, int kb,
                                                   uint64_t pol) {
  int i = 0;
  while (i + 128 <= t.bn) {
    tma_load_2d(dst + i * 128, mb[3], bar, kb * kBK, t.b_row + i, pol);
    i += 128;
  }
#pragma unroll
  for (int lg = 2; lg >= 0; --lg) {
    const int rows = 16 << lg;
    if (i + rows <= t.bn) {
      tma_load_2d(dst + i * 128, mb[lg], bar, kb * kBK, t.b_row + i, pol);
      i += rows;
    }
  }
}

// ==========================================================================
// bf16 weights
// ==========================================================================
// A split bf16 launch runs the groups of at least kSplitRows rows (tensor-bound
// at 256-row tiles) on the first gh CTAs of one grid and the smaller groups
// (bound by streaming their weights) on the last grid - gh CTAs of another,
// each grid the size of the device, concurrently.  gh shares the SMs in
// proportion to the hot groups' MMA flops and the cold groups' weight bytes,
// the bytes weighted by kSplitFlopPerByte: one SM's MMA rate over its rate of
// streaming weights through the eight-stage ring, measured (~125) and rounded
// toward more streaming SMs, because too few of those costs more.  A one-warp
// kernel computes gh before both launches (kept out of the GEMM kernel, whose
// code generation this floating-point work upset) and both read it.
constexpr double kSplitFlopPerByte = 140.0;

__device__ __forceinline__ int split_hot_ctas(const GemmParams& p, int ncta) {
  const int lane = threadIdx.x & 31;
  double hot_rows = 0.0, cold_groups = 0.0;
  for (int e = lane; e < p.E; e += 32) {
    const int r = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
    if (r >= kSplitRows)
      hot_rows += r;
    else if (r > 0)
      cold_groups += 1.0;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    hot_rows += __shfl_xor_sync(0xffffffffu, hot_rows, o);
    cold_groups += __shfl_xor_sync(0xffffffffu, cold_groups, o);
  }
  const double w_elems = static_cast<double>(p.m_tiles) * kBM * p.k_blocks * kBK;
  double hot = hot_rows * 2.0 * w_elems;      // MMA flops of the hot routed rows
  double cold = cold_groups * 2.0 * w_elems;  // bf16 weight bytes of the cold groups
  if (p.has_shared) {
    const double ws_elems = static_cast<double>(p.m_tiles_s) * kBM * p.k_blocks_s * kBK;
    if (p.T_shared >= kSplitRows)
      hot += p.T_shared * 2.0 * ws_elems;
    else if (p.T_shared > 0)
      cold += 2.0 * ws_elems;
  }
  if (cold == 0.0) return ncta;
  if (hot == 0.0) return 0;
  const int gh = static_cast<int>(ncta * hot / (hot + kSplitFlopPerByte * cold) + 0.5);
  return min(max(gh, 1), ncta - 1);
}

__global__ void __launch_bounds__(32) split_plan_kernel(const GemmParams p, int ncta, int* gh) {
  pdl_wait();
  pdl_trigger();
  const int v = split_hot_ctas(p, ncta);
  if (threadIdx.x == 0) *gh = v;
}

cudaError_t launch_split_plan(const GemmParams& p, int ncta, int* gh, cudaStream_t st) {
  return pdl_launch(split_plan_kernel, dim3(1), dim3(32), 0, st, p, ncta, gh);
}

template <int BN_MAX, int STAGES>
__global__ void __launch_bounds__(kBf16Threads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                        const __grid_constant__ CUtensorMap tm_a_s,
                        const __grid_constant__ CUtensorMap tm_b,
                        const __grid_constant__ CUtensorMap tm_b_s,
                        const __grid_constant__ CUtensorMap tm_b2,
                        const __grid_constant__ CUtensorMap tm_b2_s,
                        const __grid_constant__ CUtensorMap tm_b4,
                        const __grid_constant__ CUtensorMap tm_b4_s,
                        const __grid_constant__ CUtensorMap tm_b8,
                        const __grid_constant__ CUtensorMap tm_b8_s, const GemmParams p) {
  pdl_wait();
  // Split launches: this grid's share of the SMs and of the groups; the CTAs
  // beyond the share leave before taking any resource.
  int ncta = static_cast<int>(gridDim.x);
  int min_rows = 0, max_rows = 0x7fffffff;
  if (p.split_role != 0) {
    const int gh = __ldg(p.split_gh);
    if (p.split_role == 1) {
      ncta = gh;
      min_rows = kSplitRows;
    } else {
      ncta -= gh;
      min_rows = 1;
      max_rows = kSplitRows - 1;
    }
    if (static_cast<int>(blockIdx.x) >= ncta) {
      pdl_trigger();
      return;
    }
  }
  extern __shared__ uint8_t smem_raw[];
  using Smem = Bf16Smem<BN_MAX, STAGES>;
  const uint32_t raw = smem_u32(smem_raw);
  Smem& s = *reinterpret_cast<Smem*>(smem_raw + (((raw + 1023u) & ~1023u) - raw));
  GemmCommon<BN_MAX>& cm = s.c;
  constexpr uint32_t kTmemCols = (2 * BN_MAX < 32) ? 32u : static_cast<uint32_t>(2 * BN_MAX);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.E + p.has_shared;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    init_common_barriers<BN_MAX>(cm, kBf16EpiWarps);
    cm.walk_ctas = ncta;
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    prefetch_tmap(&tm_b2);
    prefetch_tmap(&tm_b4);
    prefetch_tmap(&tm_b8);
    if (p.has_shared) {
      prefetch_tmap(&tm_a_s);
      prefetch_tmap(&tm_b_s);
      prefetch_tmap(&tm_b2_s);
      prefetch_tmap(&tm_b4_s);
      prefetch_tmap(&tm_b8_s);
    }
  }
  const int ntiles =
      build_tile_table<BN_MAX, true>(cm, p, G, kBf16Threads, min_rows, max_rows);
  if (warp == 1) {
    tmem_alloc(&cm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = cm.tmem_base;
  volatile int* abort_flag = &cm.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      // Weight tiles read by one token tile stream through L2 (evict first);
      // those of groups with several token tiles are read again by the
      // neighbouring tiles of the walk and are kept (evict last).
      const uint64_t pol_once = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;  // bit i: stage i had a load issued; its phase in issued_ph
      uint32_t issued_ph = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < ntiles && ok; L += ncta) {
        const TileInfo t = decode_tile<BN_MAX>(cm, p, G, L);
        const CUtensorMap* ma = t.shared ? &tm_a_s : &tm_a;
        const CUtensorMap* const mb[4] = {t.shared ? &tm_b_s : &tm_b, t.shared ? &tm_b2_s : &tm_b2,
                                          t.shared ? &tm_b4_s : &tm_b4,
                                          t.shared ? &tm_b8_s : &tm_b8};
        const uint32_t bytes = kAStage + static_cast<uint32_t>(t.bn) * 128u;
        const int row = tile_a_row(p, t);
        const uint64_t pol_w = t.n_tiles > 1 ? pol_x : pol_once;
        for (int kb = 0; kb < t.k_blocks; ++kb) {
          if (!mbar_wait<true>(&s.empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&s.full[stage], bytes);
          issued |= 1u << stage;
          issued_ph = (issued_ph & ~(1u << stage)) | (phase << stage);
          if (p.op == kOpGateUp)
            tma_load_4d(s.a[stage], ma, &s.full[stage], kb * kBK, 0, 0, row / 16, pol_w);
          else
            tma_load_2d(s.a[stage], ma, &s.full[stage], kb * kBK, row, pol_w);
          load_token_tile_p2(s.b[stage], mb, &s.full[stage], t, kb, pol_x);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        record_error(p, abort_flag, MOE_ERR_TIMEOUT);
        for (int i = 0; i < STAGES; ++i)
          if ((issued >> i) & 1u) mbar_wait_time_only(&s.full[i], (issued_ph >> i) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < ntiles && ok; L += ncta) {
        const TileInfo t = decode_tile<BN_MAX>(cm, p, G, L);
        if (!mbar_wait<true>(&cm.tempty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN_MAX);
        const uint32_t idesc = idesc_bf16_f32(kBM, t.bn);
        for (int kb = 0; kb < t.k_blocks; ++kb) {
          if (!mbar_wait<true>(&s.full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_sw128(smem_u32(s.a[stage]));
          const uint64_t bd = sdesc_sw128(smem_u32(s.b[stage]));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16_ss(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          mma_commit(&s.empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&cm.tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) record_error(p, abort_flag, MOE_ERR_TIMEOUT);
      // No MMA may be in flight when TMEM is released.
      mma_commit(&cm.drain);
      mbar_wait_time_only(&cm.drain, 0);
    }
  } else {
    epilogue_role<BN_MAX, 1, true, kBf16EpiWarps>(cm, p, G, ntiles, tmem_base, abort_flag, warp,
                                                  lane);
  }

  // The successor may launch once every CTA is past its tiles (a persistent
  // grid would otherwise let it occupy the SMs' slots for the whole run).
  pdl_trigger();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ==========================================================================
// W4A16 weights: packed int4 restored to bf16 in shared memory ahead of the MMA
// ==========================================================================
//   producer (warp 0): per tile, the tile's group-scale table (TMA, double
//             buffered, when scale_table is set); per packed stage (4 k-blocks),
//             128 rows x 128 B of packed int4 (128-B swizzle).
//   token producer (warp 14): per k-block, the token tile.  A separate thread,
//             so the weight ring prefetches to its full depth (64 KB) no matter
//             how far the token ring is filled.
//   dequant group g (warps 6+4g .. 9+4g): for every packed stage, restores
//             k-blocks 4q + g and 4q + 2 + g (those that exist) into operand
//             buffers 2g and 2g + 1, then releases the packed stage.  Every
//             group consumes every packed stage and only its own buffers, so
//             all waits stay in phase order, and the MMA of one buffer overlaps
//             the restore of the other.
//   MMA:      per k-block 4q + j, operand buffer 2 (j % 2) + j / 2 and the next
//             token stage.
template <int BN_MAX, int PSTAGES, int BSTAGES>
__global__ void __launch_bounds__(kW4Threads, 1)
    grouped_gemm_w4_kernel(const __grid_constant__ CUtensorMap tm_a,
                           const __grid_constant__ CUtensorMap tm_a_s,
                           const __grid_constant__ CUtensorMap tm_b,
                           const __grid_constant__ CUtensorMap tm_b_s,
                           const __grid_constant__ CUtensorMap tm_b2,
                           const __grid_constant__ CUtensorMap tm_b2_s,
                           const __grid_constant__ CUtensorMap tm_b4,
                           const __grid_constant__ CUtensorMap tm_b4_s,
                           const __grid_constant__ CUtensorMap tm_b8,
                           const __grid_constant__ CUtensorMap tm_b8_s,
                           const __grid_constant__ CUtensorMap tm_sc,
                           const __grid_constant__ CUtensorMap tm_sc_s, const GemmParams p) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  using Smem = W4Smem<BN_MAX, PSTAGES, BSTAGES>;
  const uint32_t raw = smem_u32(smem_raw);
  Smem& s = *reinterpret_cast<Smem*>(smem_raw + (((raw + 1023u) & ~1023u) - raw));
  GemmCommon<BN_MAX>& cm = s.c;
  constexpr uint32_t kTmemCols = (2 * BN_MAX < 32) ? 32u : static_cast<uint32_t>(2 * BN_MAX);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.E + p.has_shared;
  const bool table = p.scale_table != 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < PSTAGES; ++i) {
      mbar_init(&s.pfull[i], 1);
      mbar_init(&s.pempty[i], kDequantWarps);
    }
    for (int i = 0; i < BSTAGES; ++i) {
      mbar_init(&s.bfull[i], 1);
      mbar_init(&s.bempty[i], 1);
    }
    for (int i = 0; i < kABuffers; ++i) {
      mbar_init(&s.aready[i], kWarpsPerGroup);
      mbar_init(&s.afree[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.sfull[i], 1);
      mbar_init(&s.sempty[i], kDequantWarps);
    }
    init_common_barriers<BN_MAX>(cm);
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    prefetch_tmap(&tm_b2);
    prefetch_tmap(&tm_b4);
    prefetch_tmap(&tm_b8);
    if (table) prefetch_tmap(&tm_sc);
    if (p.has_shared) {
      prefetch_tmap(&tm_a_s);
      prefetch_tmap(&tm_b_s);
      prefetch_tmap(&tm_b2_s);
      prefetch_tmap(&tm_b4_s);
      prefetch_tmap(&tm_b8_s);
      if (table) prefetch_tmap(&tm_sc_s);
    }
  }
  const int ntiles = build_tile_table<BN_MAX>(cm, p, G, kW4Threads);
  if (warp == 1) {
    tmem_alloc(&cm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = cm.tmem_base;
  volatile int* abort_flag = &cm.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer: weights
      const uint64_t pol_w = policy_evict_first();
      int ps = 0;
      uint32_t pph = 0;
      uint32_t tile_ctr = 0;
      // loads in flight on abort: packed stages (bit, phase) and the last table
      uint32_t p_iss = 0, p_issph = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < ntiles && ok; L += gridDim.x) {
        const TileInfo t = decode_tile<BN_MAX>(cm, p, G, L);
        const CUtensorMap* ma = t.shared ? &tm_a_s : &tm_a;
        const int row = tile_a_row(p, t);
        if (table) {
          const int sb = tile_ctr & 1;
          if (!mbar_wait(&s.sempty[sb], ((tile_ctr >> 1) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const int ngrp = (t.shared ? p.K_s : p.K) / kGroup;
          const CUtensorMap* msc = t.shared ? &tm_sc_s : &tm_sc;
          mbar_arrive_expect_tx(&s.sfull[sb], static_cast<uint32_t>(kBM * ngrp * 2));
          if (p.op == kOpGateUp) {
#pragma unroll
            for (int b = 0; b < 4; ++b)
              tma_load_3d(s.stab[sb] + b * 32 * ngrp, msc, &s.sfull[sb], 0, row + 16 * b, 0,
                          pol_w);
          } else {
            tma_load_2d(s.stab[sb], msc, &s.sfull[sb], 0, row, pol_w);
          }
          ++tile_ctr;
        }
        for (int kb = 0; kb < t.k_blocks; kb += kKPerPacked) {
          {
            if (!mbar_wait(&s.pempty[ps], pph ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&s.pfull[ps], kPackedStage);
            p_iss |= 1u << ps;
            p_issph = (p_issph & ~(1u << ps)) | (pph << ps);
            const int wc = kb * kBK / 8;  // packed words along K
            if (p.op == kOpGateUp) {
#pragma unroll
              for (int b = 0; b < 4; ++b)
                tma_load_3d(s.praw[ps] + b * 4096, ma, &s.pfull[ps], wc, row + 16 * b, 0, pol_w);
            } else {
              tma_load_2d(s.praw[ps], ma, &s.pfull[ps], wc, row, pol_w);
            }
            if (++ps == PSTAGES) {
              ps = 0;
              pph ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        record_error(p, abort_flag, MOE_ERR_TIMEOUT);
        for (int i = 0; i < PSTAGES; ++i)
          if ((p_iss >> i) & 1u) mbar_wait_time_only(&s.pfull[i], (p_issph >> i) & 1u);
        if (tile_ctr > 0) {
          const uint32_t last = tile_ctr - 1;
          mbar_wait_time_only(&s.sfull[last & 1], (last >> 1) & 1u);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int bs = 0;
      uint32_t bph = 0;
      uint32_t aph = 0;  // bit g: phase of operand buffer g
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < ntiles && ok; L += gridDim.x) {
        const TileInfo t = decode_tile<BN_MAX>(cm, p, G, L);
        if (!mbar_wait(&cm.tempty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN_MAX);
        const uint32_t idesc = idesc_bf16_f32(kBM, t.bn);
        for (int kb = 0; kb < t.k_blocks; ++kb) {
          // k-block 4q + j sits in buffer 2 (j % 2) + j / 2 (group j % 2)
          const int j = kb % kKPerPacked;
          const int g = 2 * (j % 2) + j / 2;
          if (!mbar_wait(&s.aready[g], (aph >> g) & 1u, abort_flag) ||
              !mbar_wait(&s.bfull[bs], bph, abort_flag)) {
            ok = false;
            break;
          }
          aph ^= 1u << g;
          tc_fence_after();
          const uint64_t ad = sdesc_sw128(smem_u32(s.a[g]));
          const uint64_t bd = sdesc_sw128(smem_u32(s.b[bs]));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16_ss(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          mma_commit(&s.bempty[bs]);
          mma_commit(&s.afree[g]);
          if (++bs == BSTAGES) {
            bs = 0;
            bph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&cm.tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) record_error(p, abort_flag, MOE_ERR_TIMEOUT);
      mma_commit(&cm.drain);
      mbar_wait_time_only(&cm.drain, 0);
    }
  } else if (warp < 6) {
    epilogue_role<BN_MAX>(cm, p, G, ntiles, tmem_base, abort_flag, warp, lane);
  } else if (warp == kTokenWarp) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer: token tiles
      // in power-of-two boxes of 16 to 128 rows (two copies for 256 rows).
      const uint64_t pol_x = policy_evict_last();
      int bs = 0;
      uint32_t bph = 0;
      uint32_t b_iss = 0, b_issph = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < ntiles && ok; L += gridDim.x) {
        const TileInfo t = decode_tile<BN_MAX>(cm, p, G, L);
        const CUtensorMap* const mb[4] = {t.shared ? &tm_b_s : &tm_b, t.shared ? &tm_b2_s : &tm_b2,
                                          t.shared ? &tm_b4_s : &tm_b4,
                                          t.shared ? &tm_b8_s : &tm_b8};
        for (int kb = 0; kb < t.k_blocks; ++kb) {
          if (!mbar_wait(&s.bempty[bs], bph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&s.bfull[bs], static_cast<uint32_t>(t.bn) * 128u);
          b_iss |= 1u << bs;
          b_issph = (b_issph & ~(1u << bs)) | (bph << bs);
          load_token_tile_p2(s.b[bs], mb, &s.bfull[bs], t, kb, pol_x);
          if (++bs == BSTAGES) {
            bs = 0;
            bph ^= 1u;
          }
        }
      }
      if (!ok) {
        record_error(p, abort_flag, MOE_ERR_TIMEOUT);
        for (int i = 0; i < BSTAGES; ++i)
          if ((b_iss >> i) & 1u) mbar_wait_time_only(&s.bfull[i], (b_issph >> i) & 1u);
      }
    }
  } else {
    // -------------------------------------------------- dequant groups
    // Thread r of group grp owns tile row r.  In a packed stage (128-B swizzled
    // rows of 256 int4 values) k-block j of the stage is 16-B chunks 2j, 2j + 1
    // of each row; the thread writes eight 16-B bf16 chunks into the
    // 128-B-swizzled operand buffer (chunk c of row r at r*128 + ((c ^ (r & 7)) << 4)).
    const int dw = warp - 6;
    const int grp = dw / kWarpsPerGroup;
    const int r = (dw % kWarpsPerGroup) * 32 + lane;
    int ps = 0;
    uint32_t pph = 0;
    uint32_t aphase = 0;  // bit h: phase of this group's buffer 2 grp + h
    uint32_t tile_ctr = 0;
    bool ok = true;
    for (int L = blockIdx.x; L < ntiles && ok; L += gridDim.x) {
      const TileInfo t = decode_tile<BN_MAX>(cm, p, G, L);
      const int K = t.shared ? p.K_s : p.K;
      const int ngrp = K / kGroup;
      const uint16_t* srow = (t.shared ? p.wscale_s : p.wscale) +
                             static_cast<size_t>(tile_weight_row(p, t, r)) * ngrp;
      const int sb = tile_ctr & 1;
      if (table && !mbar_wait(&s.sfull[sb], (tile_ctr >> 1) & 1u, abort_flag)) {
        ok = false;
        break;
      }
      for (int kb0 = 0; kb0 < t.k_blocks && ok; kb0 += kKPerPacked) {
        if (!mbar_wait(&s.pfull[ps], pph, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* prow = s.praw[ps] + r * 128;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = 2 * h + grp;  // k-block within the packed stage
          const int kb = kb0 + j;
          if (kb >= t.k_blocks) continue;
          const int buf = 2 * grp + h;
          const int g = (kb * kBK) / kGroup;
          const uint16_t sbits = p.channel ? uint16_t{0x3F80} : table ? s.stab[sb][r * ngrp + g] : __ldg(srow + g);
          __nv_bfloat162 s2;
          s2.x = __ushort_as_bfloat16(sbits);
          s2.y = s2.x;
          const uint4 p0 = *reinterpret_cast<const uint4*>(prow + (((2 * j) ^ (r & 7)) << 4));
          const uint4 p1 = *reinterpret_cast<const uint4*>(prow + (((2 * j + 1) ^ (r & 7)) << 4));
          const uint32_t words[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
          if (!mbar_wait(&s.afree[buf], ((aphase >> h) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* arow = s.a[buf] + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) << 4)) = restore_word(words[c], s2, p.channel != 0);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.aready[buf]);
          aphase ^= 1u << h;
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.pempty[ps]);
        if (++ps == PSTAGES) {
          ps = 0;
          pph ^= 1u;
        }
      }
      if (!ok) break;
      if (table) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.sempty[sb]);
        ++tile_ctr;
      }
    }
    if (!ok) record_error(p, abort_flag, MOE_ERR_TIMEOUT);
  }

  // The successor may launch once every CTA is past its tiles (a persistent
  // grid would otherwise let it occupy the SMs' slots for the whole run).
  pdl_trigger();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ==========================================================================
// W4A16 weights, restored operand in tensor memory (token tiles up to 64 rows)
// ==========================================================================
// The dequant warps write restored bf16 weight rows straight into TMEM with
// tcgen05.st (thread = tile row = TMEM lane, two K values per 32-bit column),
// and the MMA reads A from TMEM, so shared memory carries only the packed
// weights and the token rows.  Every hand-off is per packed stage (four
// k-blocks): one packed ring slot, one token ring slot (the token rows of the
// same four k-blocks) and one TMEM operand slot of 4 x 32 columns.  A
// tcgen05.mma, a commit and an mbarrier wait each cost tens of cycles on the
// one issuing thread, and one k-block of int4 weights arrives every ~90 ns at
// the HBM rate, so the MMA thread waits twice and commits twice per 16 MMAs.
// Two MMA warps issue in parallel (one issuer alone is bound by its own
// issue latency): issuer i takes k-blocks 2i, 2i+1 of every packed stage
// into its own partial accumulator, and the epilogue adds the two.
// TMEM: 2 issuers x 2 buffers x 64 accumulator columns + kTSlots x 128
// operand columns = 512.  The dequant warps form NG groups that take the
// packed stages in turn, each group into its own operand slot, so two stages
// are restored at once; in a group, warp w serves TMEM lane quarter w % 4
// (the quarter a warp may access) and the k-blocks j of the stage with
// j % kSub == its index within the quarter.  Two groups of four warps (each
// restoring all four k-blocks of its quarter) beat one group of eight by
// 4-6% on the gate/up launch.
constexpr int kTSlots = 2;
constexpr int kTIssuers = 2;
constexpr uint32_t kTmemAccCols = 256;  // 2 issuers x 2 x 64 accumulator columns
constexpr uint32_t kTSlotCols = 32 * kKPerPacked;
constexpr int kTokStage = kKPerPacked * 64 * 128;  // token rows of four k-blocks (32 KB)
static_assert(kTmemAccCols + kTSlotCols * kTSlots <= 512, "TMEM budget");

// Token rows of k-block kb in 32-row boxes (the map's box is 32 rows high):
// ceil(bn / 32) copies; rows past the group (or past the matrix, zero-filled)
// land in columns the MMA does not read or the epilogue drops.
__device__ __forceinline__ int tok_boxes32(const TileInfo& t) { return (t.bn + 31) >> 5; }
__device__ __forceinline__ void load_token_tile32(uint8_t* dst, const CUtensorMap* mb,
                                                  uint64_t* bar, const TileInfo& t, int kb,
                                                  uint64_t pol) {
  for (int i = 0; i < tok_boxes32(t); ++i)
    tma_load_2d(dst + i * 4096, mb, bar, kb * kBK, t.b_row + 32 * i, pol);
}

template <int ND>
__host__ __device__ constexpr int w4t_threads() {
  return kBaseThreads + 32 * ND + 64;  // + token producer + second MMA issuer
}

template <int PSTAGES, int TSTAGES>
struct W4TSmem {
  uint8_t b[TSTAGES][kTokStage];        // token rows, four k-blocks of 64 x 128 B
  uint8_t praw[PSTAGES][kPackedStage];  // packed int4 rows, 128-B swizzle
  uint16_t stab[2][kScaleTabElems];     // group scales of the current tiles
  uint64_t pfull[PSTAGES], pempty[PSTAGES];
  uint64_t bfull[TSTAGES], bempty[TSTAGES];
  uint64_t aready[kTSlots], afree[kTSlots];
  uint64_t sfull[2], sempty[2];
  uint64_t drain2;
  GemmCommon<64> c;
};

// SM: where the restore takes its scale from.  0: the group scales in global
// memory; 1: the group scales from the tile's shared-memory table (TMA);
// 2: channel-wise scales (the restore keeps q exact and the epilogue scales).
template <int PSTAGES, int TSTAGES, int ND, int SM, int NG = 1>
__global__ void __launch_bounds__(w4t_threads<ND>(), 1)
    grouped_gemm_w4t_kernel(const __grid_constant__ CUtensorMap tm_a,
                            const __grid_constant__ CUtensorMap tm_a_s,
                            const __grid_constant__ CUtensorMap tm_b,
                            const __grid_constant__ CUtensorMap tm_b_s,
                            const __grid_constant__ CUtensorMap tm_sc,
                            const __grid_constant__ CUtensorMap tm_sc_s, const GemmParams p) {
  pdl_wait();
  // NG groups of dequant warps take the packed stages in turn (stage q goes
  // to group q % NG), each stage restored by the ND / NG warps of one group.
  constexpr int kGroupWarps = ND / NG;
  static_assert(ND % NG == 0 && kGroupWarps % 4 == 0 && kKPerPacked % (kGroupWarps / 4) == 0,
                "dequant warps per lane quarter");
  static_assert(NG == 1 || (NG == kTSlots && PSTAGES % NG == 0), "one operand slot per group");
  constexpr int BN_MAX = 64;
  constexpr int kThreads = w4t_threads<ND>();
  constexpr int kTokWarp = 6 + ND;
  constexpr int kMma2Warp = 7 + ND;
  constexpr int kSub = kGroupWarps / 4;        // dequant warps per TMEM lane quarter and group
  constexpr int kMyBlocks = kKPerPacked / kSub;  // k-blocks per packed stage and warp
  extern __shared__ uint8_t smem_raw[];
  using Smem = W4TSmem<PSTAGES, TSTAGES>;
  const uint32_t raw = smem_u32(smem_raw);
  Smem& s = *reinterpret_cast<Smem*>(smem_raw + (((raw + 1023u) & ~1023u) - raw));
  GemmCommon<BN_MAX>& cm = s.c;
  constexpr uint32_t kTmemCols = 512;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.E + p.has_shared;
  constexpr bool table = SM == 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < PSTAGES; ++i) {
      mbar_init(&s.pfull[i], 1);
      mbar_init(&s.pempty[i], kGroupWarps);
    }
    for (int i = 0; i < TSTAGES; ++i) {
      mbar_init(&s.bfull[i], 1);
      mbar_init(&s.bempty[i], kTIssuers);
    }
    for (int i = 0; i < kTSlots; ++i) {
      mbar_init(&s.aready[i], kGroupWarps);
      mbar_init(&s.afree[i], kTIssuers);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.sfull[i], 1);
      mbar_init(&s.sempty[i], ND);
    }
    init_common_barriers<BN_MAX>(cm);
    mbar_init(&cm.tfull[0], kTIssuers);
    mbar_init(&cm.tfull[1], kTIssuers);
    mbar_init(&s.drain2, 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    if (table) prefetch_tmap(&tm_sc);
    if (p.has_shared) {
      prefetch_tmap(&tm_a_s);
      prefetch_tmap(&tm_b_s);
      if (table) prefetch_tmap(&tm_sc_s);
    }
  }
  const int ntiles = build_tile_table<BN_MAX>(cm, p, G, kThreads);
  if (warp == 1) {
    tmem_alloc(&cm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = cm.tmem_base;
  volatile int* abort_flag = &cm.abort_flag;

  if (warp == 0) {
    if (lane < 4) {
      // ------------------------------------------------ TMA producer: weights + scales
      // Issuing a tensor copy holds the issuing thread for a few hundred
      // cycles, so lanes 0-3 issue the four boxes of a gate/up stage side by
      // side; lane 0 owns the barriers.
      const uint64_t pol_w = policy_evict_first();
      int ps = 0;
      uint32_t pph = 0;
      uint32_t tile_ctr = 0;
      uint32_t p_iss = 0, p_issph = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < ntiles && ok; L += gridDim.x) {
        const TileInfo t = decode_tile<BN_MAX>(cm, p, G, L);
        const CUtensorMap* ma = t.shared ? &tm_a_s : &tm_a;
        const int row = tile_a_row(p, t);
        if (table) {
          const int sb = tile_ctr & 1;
          bool okw = true;
          if (lane == 0) okw = mbar_wait(&s.sempty[sb], ((tile_ctr >> 1) & 1u) ^ 1u, abort_flag);
          if (!__shfl_sync(0xFu, okw, 0)) {
            ok = false;
            break;
          }
          const int ngrp = (t.shared ? p.K_s : p.K) / kGroup;
          const CUtensorMap* msc = t.shared ? &tm_sc_s : &tm_sc;
          if (lane == 0) {
            mbar_arrive_expect_tx(&s.sfull[sb], static_cast<uint32_t>(kBM * ngrp * 2));
            if (p.op == kOpGateUp) {
#pragma unroll
              for (int b = 0; b < 4; ++b)
                tma_load_3d(s.stab[sb] + b * 32 * ngrp, msc, &s.sfull[sb], 0, row + 16 * b, 0,
                            pol_w);
            } else {
              tma_load_2d(s.stab[sb], msc, &s.sfull[sb], 0, row, pol_w);
            }
          }
          ++tile_ctr;
        }
        for (int kb = 0; kb < t.k_blocks; kb += kKPerPacked) {
          bool okw = true;
          if (lane == 0) okw = mbar_wait(&s.pempty[ps], pph ^ 1u, abort_flag);
          if (!__shfl_sync(0xFu, okw, 0)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&s.pfull[ps], kPackedStage);
            p_iss |= 1u << ps;
            p_issph = (p_issph & ~(1u << ps)) | (pph << ps);
          }
          __syncwarp(0xFu);
          const int wc = kb * kBK / 8;
          if (p.op == kOpGateUp)
            tma_load_3d(s.praw[ps] + lane * 4096, ma, &s.pfull[ps], wc, row + 16 * lane, 0, pol_w);
          else if (lane == 0)
            tma_load_2d(s.praw[ps], ma, &s.pfull[ps], wc, row, pol_w);
          if (++ps == PSTAGES) {
            ps = 0;
            pph ^= 1u;
          }
        }
      }
      if (!ok && lane == 0) {
        record_error(p, abort_flag, MOE_ERR_TIMEOUT);
        for (int i = 0; i < PSTAGES; ++i)
          if ((p_iss >> i) & 1u) mbar_wait_time_only(&s.pfull[i], (p_issph >> i) & 1u);
        if (tile_ctr > 0) {
          const uint32_t last = tile_ctr - 1;
          mbar_wait_time_only(&s.sfull[last & 1], (last >> 1) & 1u);
        }
      }
    }
  } else if (warp == 1 || warp == kMma2Warp) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuers (A from TMEM)
      const int is = warp == 1 ? 0 : 1;
      uint64_t* drain = is == 0 ? &cm.drain : &s.drain2;
      int ts = 0;
      uint32_t tph = 0;
      uint32_t q = 0;  // packed stage counter over the CTA's tiles
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < ntiles && ok; L += gridDim.x) {
        const TileInfo t = decode_tile<BN_MAX>(cm, p, G, L);
        if (!mbar_wait(&cm.tempty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem =
            tmem_base + static_cast<uint32_t>(acc * BN_MAX + is * 2 * BN_MAX);
        const uint32_t idesc = idesc_bf16_f32(kBM, t.bn);
        for (int kb0 = 0; kb0 < t.k_blocks; kb0 += kKPerPacked, ++q) {
          const int slot = static_cast<int>(q % kTSlots);
          if (!mbar_wait(&s.aready[slot], (q / kTSlots) & 1u, abort_flag) ||
              !mbar_wait(&s.bfull[ts], tph, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_slot = tmem_base + kTmemAccCols + kTSlotCols * slot;
#pragma unroll
          for (int jj = 0; jj < kKPerPacked / kTIssuers; ++jj) {
            const int j = is * (kKPerPacked / kTIssuers) + jj;
            const uint64_t bd = sdesc_sw128(smem_u32(s.b[ts] + j * (64 * 128)));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_bf16_ts(d_tmem, a_slot + 32u * j + 8u * kk, bd + 2u * kk, idesc,
                          (kb0 | jj | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&s.afree[slot]);
          mma_commit(&s.bempty[ts]);
          if (++ts == TSTAGES) {
            ts = 0;
            tph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&cm.tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) record_error(p, abort_flag, MOE_ERR_TIMEOUT);
      mma_commit(drain);
      mbar_wait_time_only(drain, 0);
    }
  } else if (warp < 6) {
    epilogue_role<BN_MAX, kTIssuers>(cm, p, G, ntiles, tmem_base, abort_flag, warp, lane);
  } else if (warp == kTokWarp) {
    if (lane < kKPerPacked) {
      // ------------------------------------------------ TMA producer: token tiles
      // Lane j issues the token rows of k-block j of the stage; lane 0 owns
      // the barriers.
      const uint64_t pol_x = policy_evict_last();
      int ts = 0;
      uint32_t tph = 0;
      uint32_t b_iss = 0, b_issph = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < ntiles && ok; L += gridDim.x) {
        const TileInfo t = decode_tile<BN_MAX>(cm, p, G, L);
        const CUtensorMap* mb = t.shared ? &tm_b_s : &tm_b;
        for (int kb0 = 0; kb0 < t.k_blocks; kb0 += kKPerPacked) {
          bool okw = true;
          if (lane == 0) okw = mbar_wait(&s.bempty[ts], tph ^ 1u, abort_flag);
          if (!__shfl_sync(0xFu, okw, 0)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&s.bfull[ts],
                                  static_cast<uint32_t>(tok_boxes32(t)) * 4096u * kKPerPacked);
            b_iss |= 1u << ts;
            b_issph = (b_issph & ~(1u << ts)) | (tph << ts);
          }
          __syncwarp(0xFu);
          load_token_tile32(s.b[ts] + lane * (64 * 128), mb, &s.bfull[ts], t, kb0 + lane, pol_x);
          if (++ts == TSTAGES) {
            ts = 0;
            tph ^= 1u;
          }
        }
      }
      if (!ok && lane == 0) {
        record_error(p, abort_flag, MOE_ERR_TIMEOUT);
        for (int i = 0; i < TSTAGES; ++i)
          if ((b_iss >> i) & 1u) mbar_wait_time_only(&s.bfull[i], (b_issph >> i) & 1u);
      }
    }
  } else if (warp < kTokWarp) {
    // -------------------------------------------------- dequant warps -> TMEM
    const int qd = warp & 3;                 // TMEM lane quarter
    const int grp = (warp - 6) / kGroupWarps;  // packed stages q with q % NG == grp
    const int hd = ((warp - 6) % kGroupWarps) / 4;  // k-blocks j with j % kSub == hd
    const int r = 32 * qd + lane;            // tile row == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(32 * qd) << 16;
    int ps = 0;
    uint32_t pph = 0;
    uint32_t q = 0;
    uint32_t tile_ctr = 0;
    bool ok = true;
    for (int L = blockIdx.x; L < ntiles && ok; L += gridDim.x) {
      const TileInfo t = decode_tile<BN_MAX>(cm, p, G, L);
      const int K = t.shared ? p.K_s : p.K;
      const int ngrp = K / kGroup;
      const uint16_t* srow = (t.shared ? p.wscale_s : p.wscale) +
                             static_cast<size_t>(tile_weight_row(p, t, r)) * ngrp;
      const int sb = tile_ctr & 1;
      if (table && !mbar_wait(&s.sfull[sb], (tile_ctr >> 1) & 1u, abort_flag)) {
        ok = false;
        break;
      }
      for (int kb0 = 0; kb0 < t.k_blocks; kb0 += kKPerPacked, ++q) {
        if (NG > 1 && static_cast<int>(q % NG) != grp) {
          if (++ps == PSTAGES) {
            ps = 0;
            pph ^= 1u;
          }
          continue;
        }
        if (!mbar_wait(&s.pfull[ps], pph, abort_flag)) {
          ok = false;
          break;
        }
        // This warp's packed words leave shared memory first, so the packed
        // slot is released before the (longer) restore.
        const uint8_t* prow = s.praw[ps] + r * 128;
        uint4 pk[kMyBlocks][2];
#pragma unroll
        for (int h = 0; h < kMyBlocks; ++h) {
          const int j = kSub * h + hd;
          pk[h][0] = *reinterpret_cast<const uint4*>(prow + (((2 * j) ^ (r & 7)) << 4));
          pk[h][1] = *reinterpret_cast<const uint4*>(prow + (((2 * j + 1) ^ (r & 7)) << 4));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.pempty[ps]);
        if (++ps == PSTAGES) {
          ps = 0;
          pph ^= 1u;
        }
        const int slot = static_cast<int>(q % kTSlots);
        if (!mbar_wait(&s.afree[slot], ((q / kTSlots) & 1u) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_slot = tmem_base + lane_addr + kTmemAccCols + kTSlotCols * slot;
#pragma unroll
        for (int h = 0; h < kMyBlocks; ++h) {
          const int j = kSub * h + hd;
          const int g = ((kb0 + j) * kBK) / kGroup;
          const uint16_t sbits = SM == 2   ? uint16_t{0x3F80}
                                 : SM == 1 ? s.stab[sb][r * ngrp + g]
                                           : __ldg(srow + g);
          __nv_bfloat162 s2;
          s2.x = __ushort_as_bfloat16(sbits);
          s2.y = s2.x;
          const uint32_t words[8] = {pk[h][0].x, pk[h][0].y, pk[h][0].z, pk[h][0].w,
                                     pk[h][1].x, pk[h][1].y, pk[h][1].z, pk[h][1].w};
          uint32_t v[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 d = restore_word(words[c], s2, SM == 2);
            v[4 * c] = d.x;
            v[4 * c + 1] = d.y;
            v[4 * c + 2] = d.z;
            v[4 * c + 3] = d.w;
          }
          tmem_st_32x32b_x32(a_slot + 32u * j, v);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.aready[slot]);
      }
      if (!ok) break;
      if (table) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.sempty[sb]);
        ++tile_ctr;
      }
    }
    if (!ok) record_error(p, abort_flag, MOE_ERR_TIMEOUT);
  }

  // The successor may launch once every CTA is past its tiles (a persistent
  // grid would otherwise let it occupy the SMs' slots for the whole run).
  pdl_trigger();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int BN_MAX, int STAGES>
static cudaError_t launch_bf16(const GemmParams& p, const GemmMaps& m, int num_sms,
                               cudaStream_t st) {
  const size_t smem = sizeof(Bf16Smem<BN_MAX, STAGES>) + 1024;
  auto kern = grouped_gemm_kernel<BN_MAX, STAGES>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return pdl_launch(kern, dim3(num_sms), dim3(kBf16Threads), smem, st, m.a, m.a_s, m.b, m.b_s,
                    m.b2, m.b2_s, m.b4, m.b4_s, m.b8, m.b8_s, p);
}

template <int BN_MAX, int PSTAGES, int BSTAGES>
static cudaError_t launch_w4(const GemmParams& p, const GemmMaps& m, int num_sms,
                             cudaStream_t st) {
  const size_t smem = sizeof(W4Smem<BN_MAX, PSTAGES, BSTAGES>) + 1024;
  auto kern = grouped_gemm_w4_kernel<BN_MAX, PSTAGES, BSTAGES>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return pdl_launch(kern, dim3(num_sms), dim3(kW4Threads), smem, st, m.a, m.a_s, m.b, m.b_s, m.b2,
                    m.b2_s, m.b4, m.b4_s, m.b8, m.b8_s, m.sc, m.sc_s, p);
}

template <int PSTAGES, int TSTAGES, int ND, int NG = 1>
static cudaError_t launch_w4t(const GemmParams& p, const GemmMaps& m, int num_sms,
                              cudaStream_t st) {
  const size_t smem = sizeof(W4TSmem<PSTAGES, TSTAGES>) + 1024;
  auto kern = p.channel       ? grouped_gemm_w4t_kernel<PSTAGES, TSTAGES, ND, 2, NG>
              : p.scale_table ? grouped_gemm_w4t_kernel<PSTAGES, TSTAGES, ND, 1, NG>
                              : grouped_gemm_w4t_kernel<PSTAGES, TSTAGES, ND, 0, NG>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return pdl_launch(kern, dim3(num_sms), dim3(w4t_threads<ND>()), smem, st, m.a, m.a_s, m.b, m.b_s,
                    m.sc, m.sc_s, p);
}

cudaError_t launch_grouped_gemm(const GemmParams& p, const GemmMaps& maps, int bn_max, int quant,
                                int num_sms, cudaStream_t st) {
  if (quant == 0) {
    if (bn_max == 64) return launch_bf16<64, 8>(p, maps, num_sms, st);
    if (bn_max == 256) return launch_bf16<256, 4>(p, maps, num_sms, st);
  } else if (quant == 1) {
    if (bn_max == 64) return launch_w4t<6, 3, 8, 2>(p, maps, num_sms, st);
    // gate/up (64 k-blocks per tile) gains from a third token stage, which
    // the shared memory holds with two packed stages; down (16 k-blocks per
    // tile) keeps three packed stages.
    if (bn_max == 256)
      return p.op == kOpGateUp ? launch_w4<256, 2, 3>(p, maps, num_sms, st)
                               : launch_w4<256, 3, 2>(p, maps, num_sms, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
