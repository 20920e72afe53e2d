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
//   * warp 0: TMA producer (one thread) into a STAGES-deep shared-memory ring;
//     warp 1: TMEM allocation and tcgen05.mma issue (one thread), fp32
//     accumulators in TMEM, double buffered; warps 2-5: epilogue (tcgen05.ld).
//   * Tiles: every CTA walks tile indices blockIdx.x, +gridDim.x, ... over the
//     concatenation of groups [shared, expert 0, ..., expert E-1]; a group with
//     R rows has ceil(R / BN_MAX) * m_tiles tiles, token tiles of one weight
//     tile adjacent so repeated weight tiles come from L2.
//   * Gate/up: a tile covers 64 output features; its A rows are four blocks of
//     (16 gate rows, 16 up rows) loaded by a 3-D TMA box, so each epilogue warp
//     holds gate and up of the same 16 features in its TMEM lanes and forms
//     h = silu(g) * u with one lane exchange (no shared memory, no barrier).
//   * Down: a tile covers 128 output features; the epilogue multiplies by the
//     routing weight of the row's (token, slot) pair and stores fp32.
//   * Every wait is bounded (2 s); on expiry the CTA records MOE_ERR_TIMEOUT,
//     stops issuing, waits for its copies and MMAs in flight and frees TMEM.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kAStage = kBM * kBK * 2;      // 16 KB bf16 operand tile
constexpr int kARawStage = kBM * kBK / 2;   // 4 KB packed int4 tile
constexpr int kMaxGroups = 1025;
constexpr int kDequantWarps = 8;
constexpr int kDequantGroups = 4;  // groups restore different pipeline stages concurrently
constexpr int kWarpsPerGroup = kDequantWarps / kDequantGroups;

template <int QUANT>
struct GemmRoles {
  static constexpr int kThreads = QUANT ? 192 + 32 * kDequantWarps : 192;
  // a stage is released by the MMA commit and, for W4A16, by the warps of the
  // one dequant group that restored it
  static constexpr int kEmptyArrivals = QUANT ? 1 + kWarpsPerGroup : 1;
};

// W4A16: the raw ring (packed int4 + token tile, STAGES deep, filled by TMA) is
// decoupled from a shallow ring of kABufs restored bf16 operand tiles.
constexpr int kABufs = 4;
static_assert(kABufs % kDequantGroups == 0, "each operand buffer belongs to one group");

// W4A16 group scales of one tile (128 rows x up to 32 groups), double buffered
// across tiles and filled by TMA (used when K is a multiple of 1024 and <= 4096).
constexpr int kScaleTabElems = kBM * 32;

template <int BN_MAX, int STAGES, int QUANT>
struct GemmSmem {
  static constexpr int kA = QUANT ? kABufs : STAGES;
  static constexpr bool kScaleTab = QUANT && BN_MAX == 64;
  uint8_t a[kA][kAStage];                                  // bf16 operand, 128-B swizzle
  uint8_t b[STAGES][BN_MAX * 128];                         // token rows, 128-B swizzle
  uint8_t araw[QUANT ? STAGES : 1][QUANT ? kARawStage : 16];  // packed int4 rows (W4A16)
  uint16_t stab[kScaleTab ? 2 : 1][kScaleTab ? kScaleTabElems : 8];  // W4A16 tile scales
  uint64_t sfull[2];
  uint64_t sempty[2];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t aready[kA];
  uint64_t afree[kA];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int tile_start[kMaxGroups + 1];
  int off[kMaxGroups];
  float row_weight[4][BN_MAX];  // down epilogue: routing weight of each token row, per warp
};

struct TileInfo {
  int shared;
  int e;
  int m;
  int n_valid;
  int bn;
  int b_row;
  int k_blocks;
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

// Waits with only the time bound (used while unwinding after an abort).
__device__ __forceinline__ bool mbar_wait_time_only(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

__device__ __forceinline__ void record_error(const GemmParams& p, volatile int* abort_flag,
                                             int code) {
  *abort_flag = 1;
  if (p.status) atomicCAS(p.status, 0, code);
}

template <typename Smem, int BN_MAX>
__device__ __forceinline__ TileInfo decode_tile(const Smem& s, const GemmParams& p, int G, int L) {
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
  t.m = l / n_tiles;
  const int n = l - t.m * n_tiles;
  t.n_valid = min(BN_MAX, rows - n * BN_MAX);
  t.bn = (t.n_valid + 15) & ~15;
  t.b_row = row0 + n * BN_MAX;
  t.k_blocks = t.shared ? p.k_blocks_s : p.k_blocks;
  return t;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

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

// Eight signed 4-bit values (value j in bits 4j..4j+3) times a bf16 scale ->
// eight bf16 in order, each bf16_rne(q * s).  Nibbles become offset binary
// (q + 8), are placed in the mantissa of 128.0 (0x4300 | u = 128 + u, exact),
// shifted back by 136 (exact) and multiplied by the scale (one rounding).
__device__ __forceinline__ uint4 dequant_word(uint32_t w, __nv_bfloat162 s2) {
  const uint32_t x = w ^ 0x88888888u;
  const __nv_bfloat162 k136 = __floats2bfloat162_rn(136.0f, 136.0f);
  uint32_t h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t t = ((x >> (4 * i)) & 0x000F000Fu) | 0x43004300u;  // (e_i, e_{i+4})
    __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&t), k136);
    __nv_bfloat162 v = __hmul2(q, s2);
    h[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
  uint4 out;
  out.x = __byte_perm(h[0], h[1], 0x5410);  // e0, e1
  out.y = __byte_perm(h[2], h[3], 0x5410);  // e2, e3
  out.z = __byte_perm(h[0], h[1], 0x7632);  // e4, e5
  out.w = __byte_perm(h[2], h[3], 0x7632);  // e6, e7
  return out;
}

template <int BN_MAX, int STAGES, int QUANT>
__global__ void __launch_bounds__(GemmRoles<QUANT>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                        const __grid_constant__ CUtensorMap tm_a_s,
                        const __grid_constant__ CUtensorMap tm_b,
                        const __grid_constant__ CUtensorMap tm_b_s,
                        const __grid_constant__ CUtensorMap tm_sc,
                        const __grid_constant__ CUtensorMap tm_sc_s, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  using Smem = GemmSmem<BN_MAX, STAGES, QUANT>;
  constexpr int kThreads = GemmRoles<QUANT>::kThreads;
  const uint32_t raw = smem_u32(smem_raw);
  Smem& s = *reinterpret_cast<Smem*>(smem_raw + (((raw + 1023u) & ~1023u) - raw));
  constexpr uint32_t kTmemCols = (2 * BN_MAX < 32) ? 32u : static_cast<uint32_t>(2 * BN_MAX);
  constexpr uint32_t kABytes = QUANT ? kARawStage : kAStage;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.E + p.has_shared;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], GemmRoles<QUANT>::kEmptyArrivals);
    }
    for (int i = 0; i < Smem::kA; ++i) {
      mbar_init(&s.aready[i], kWarpsPerGroup);
      mbar_init(&s.afree[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.sfull[i], 1);
      mbar_init(&s.sempty[i], kDequantWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], 4);
    }
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    if (p.has_shared) {
      prefetch_tmap(&tm_a_s);
      prefetch_tmap(&tm_b_s);
    }
  }
  for (int i = threadIdx.x; i <= p.E; i += kThreads) s.off[i] = p.offsets[i];
  __syncthreads();
  // Tiles per group, then an exclusive scan into tile_start.
  for (int g = threadIdx.x; g < G; g += kThreads) {
    const bool sh = p.has_shared && g == 0;
    const int e = g - p.has_shared;
    const int rows = sh ? p.T_shared : s.off[e + 1] - s.off[e];
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
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int ntiles = s.tile_start[G];
  const uint32_t tmem_base = s.tmem_base;
  volatile int* abort_flag = &s.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;  // bit i: stage i had a load issued; its phase in issued_ph
      uint32_t issued_ph = 0;
      uint32_t tile_ctr = 0;  // W4A16 scale tables issued
      uint32_t sissued = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < ntiles && ok; L += gridDim.x) {
        const TileInfo t = decode_tile<Smem, BN_MAX>(s, p, G, L);
        const CUtensorMap* ma = t.shared ? &tm_a_s : &tm_a;
        const CUtensorMap* mb = t.shared ? &tm_b_s : &tm_b;
        const uint32_t bytes = kABytes + static_cast<uint32_t>(t.bn) * 128u;
        const int a_row0 = t.shared ? 0 : t.e * p.a_rows_per_expert;
        if (Smem::kScaleTab && p.scale_table) {
          // this tile's group scales: 128 rows x K/128 groups, same row order as the weights
          const int sb = tile_ctr & 1;
          if (!mbar_wait(&s.sempty[sb], ((tile_ctr >> 1) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const int ngrp = (t.shared ? p.K_s : p.K) / p.group;
          const CUtensorMap* msc = t.shared ? &tm_sc_s : &tm_sc;
          mbar_arrive_expect_tx(&s.sfull[sb], static_cast<uint32_t>(kBM * ngrp * 2));
          if (p.op == kOpGateUp) {
#pragma unroll
            for (int b = 0; b < 4; ++b)
              tma_load_3d(s.stab[sb] + b * 32 * ngrp, msc, &s.sfull[sb], 0,
                          a_row0 + t.m * 64 + 16 * b, 0, pol_w);
          } else {
            tma_load_2d(s.stab[sb], msc, &s.sfull[sb], 0, a_row0 + t.m * kBM, pol_w);
          }
          sissued = 1u << sb;
          ++tile_ctr;
        }
        for (int kb = 0; kb < t.k_blocks; ++kb) {
          if (!mbar_wait(&s.empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&s.full[stage], bytes);
          issued |= 1u << stage;
          issued_ph = (issued_ph & ~(1u << stage)) | (phase << stage);
          const int kc = kb * kBK;
          // weights: bf16 tiles at column kc, or packed int4 at word kc / 8
          void* adst = QUANT ? static_cast<void*>(s.araw[stage]) : static_cast<void*>(s.a[stage]);
          const int ac = QUANT ? kc / 8 : kc;
          constexpr int kRowBytes = QUANT ? kBK / 2 : kBK * 2;
          if (p.op == kOpGateUp) {
            const int row = a_row0 + t.m * 64;
#pragma unroll
            for (int b = 0; b < 4; ++b)
              tma_load_3d(static_cast<uint8_t*>(adst) + b * 32 * kRowBytes, ma, &s.full[stage], ac,
                          row + 16 * b, 0, pol_w);
          } else {
            tma_load_2d(adst, ma, &s.full[stage], ac, a_row0 + t.m * kBM, pol_w);
          }
          for (int i = 0; i < t.bn / 16; ++i)
            tma_load_2d(s.b[stage] + i * 2048, mb, &s.full[stage], kc, t.b_row + 16 * i, pol_x);
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
        if (sissued) {
          const uint32_t last = tile_ctr - 1;
          mbar_wait_time_only(&s.sfull[last & 1], (last >> 1) & 1u);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int abuf = 0;  // W4A16: restored operand buffer and its phase
      uint32_t aphase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < ntiles && ok; L += gridDim.x) {
        const TileInfo t = decode_tile<Smem, BN_MAX>(s, p, G, L);
        if (!mbar_wait(&s.tempty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN_MAX);
        const uint32_t idesc = idesc_bf16_f32(kBM, t.bn);
        for (int kb = 0; kb < t.k_blocks; ++kb) {
          if ((QUANT && !mbar_wait(&s.aready[abuf], aphase, abort_flag)) ||
              !mbar_wait(&s.full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_sw128(smem_u32(s.a[QUANT ? abuf : stage]));
          const uint64_t bd = sdesc_sw128(smem_u32(s.b[stage]));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16_ss(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          mma_commit(&s.empty[stage]);
          if (QUANT) {
            mma_commit(&s.afree[abuf]);
            if (++abuf == Smem::kA) {
              abuf = 0;
              aphase ^= 1u;
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&s.tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) record_error(p, abort_flag, MOE_ERR_TIMEOUT);
      // No MMA may be in flight when TMEM is released.
      mma_commit(&s.drain);
      mbar_wait_time_only(&s.drain, 0);
    }
  } else if (warp < 6) {
    // -------------------------------------------------- epilogue (warps 2-5)
    const int sp = warp & 3;  // TMEM lanes 32*sp .. 32*sp+31
    float* wts = s.row_weight[warp - 2];
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int L = blockIdx.x; L < ntiles; L += gridDim.x) {
      const TileInfo t = decode_tile<Smem, BN_MAX>(s, p, G, L);
      if (p.op == kOpDown) {
        // Routing weight of every token row of the tile, fetched before the
        // accumulator is ready: row r holds pair p = perm_pair[r] (token p / k,
        // slot p % k); the shared group has weight 1.
        __syncwarp();
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
        __syncwarp();
      }
      if (!mbar_wait(&s.tfull[acc], acc_phase, abort_flag)) {
        record_error(p, abort_flag, MOE_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t tbase =
          tmem_base + static_cast<uint32_t>(acc * BN_MAX) + (static_cast<uint32_t>(sp * 32) << 16);
      for (int c0 = 0; c0 < t.bn; c0 += 16) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(tbase + static_cast<uint32_t>(c0), r);
        tmem_wait_ld();
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
  } else if (QUANT) {
    // -------------------------------------------------- dequant (warps 6-13, W4A16)
    // kDequantGroups groups of kWarpsPerGroup warps.  The running k-block index
    // i goes to group i mod kDequantGroups; since the raw ring depth and the
    // operand ring depth are both multiples of the group count, every raw stage
    // and every operand buffer always belongs to the same group, so each group
    // waits on each of its barriers in phase order.  Within a group, thread tg
    // owns tile rows tg + 64 j: it reads the row's 32 B of packed int4 and writes
    // eight 16-B chunks of bf16 into the 128-B-swizzled operand tile (chunk c of
    // row r lives at r*128 + ((c ^ (r & 7)) << 4)).
    constexpr int kGroupThreads = 32 * kWarpsPerGroup;
    constexpr int kRowsPerThread = kBM / kGroupThreads;
    static_assert(STAGES % kDequantGroups == 0, "raw stages must map to fixed groups");
    const int dw = warp - 6;
    const int grp = dw / kWarpsPerGroup;
    const int tg = (dw % kWarpsPerGroup) * 32 + lane;
    uint32_t idx = 0;  // running k-block index (the same sequence every role walks)
    uint32_t tile_ctr = 0;
    const bool table = Smem::kScaleTab && p.scale_table;
    bool ok = true;
    for (int L = blockIdx.x; L < ntiles && ok; L += gridDim.x) {
      const TileInfo t = decode_tile<Smem, BN_MAX>(s, p, G, L);
      const int K = t.shared ? p.K_s : p.K;
      const int ngrp = K / p.group;
      const uint16_t* sbase = t.shared ? p.wscale_s : p.wscale;
      const uint16_t* srow[kRowsPerThread];
#pragma unroll
      for (int j = 0; j < kRowsPerThread; ++j)
        srow[j] = sbase + static_cast<size_t>(tile_weight_row(p, t, tg + j * kGroupThreads)) * ngrp;
      const int sb = tile_ctr & 1;
      if (table && !mbar_wait(&s.sfull[sb], (tile_ctr >> 1) & 1u, abort_flag)) {
        ok = false;
        break;
      }
      for (int kb = 0; kb < t.k_blocks; ++kb, ++idx) {
        if (static_cast<int>(idx % kDequantGroups) != grp) continue;
        const int stage = static_cast<int>(idx % STAGES);
        const uint32_t phase = (idx / STAGES) & 1u;
        const int abuf = static_cast<int>(idx % kABufs);
        const uint32_t aphase = (idx / kABufs) & 1u;
        __nv_bfloat162 s2[kRowsPerThread];
#pragma unroll
        for (int j = 0; j < kRowsPerThread; ++j) {
          const int g = (kb * kBK) / p.group;
          const uint16_t sbits = table ? s.stab[sb][(tg + j * kGroupThreads) * ngrp + g]
                                       : __ldg(srow[j] + g);
          s2[j].x = __ushort_as_bfloat16(sbits);
          s2[j].y = s2[j].x;
        }
        if (!mbar_wait(&s.full[stage], phase, abort_flag) ||
            !mbar_wait(&s.afree[abuf], aphase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int j = 0; j < kRowsPerThread; ++j) {
          const int r = tg + j * kGroupThreads;
          const uint4 p0 = *reinterpret_cast<const uint4*>(s.araw[stage] + r * 32);
          const uint4 p1 = *reinterpret_cast<const uint4*>(s.araw[stage] + r * 32 + 16);
          const uint32_t words[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
          uint8_t* arow = s.a[abuf] + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) << 4)) = dequant_word(words[c], s2[j]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&s.aready[abuf]);
          mbar_arrive(&s.empty[stage]);
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

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int BN_MAX, int STAGES, int QUANT>
static cudaError_t launch_variant(const GemmParams& p, const GemmMaps& m, int num_sms,
                                  cudaStream_t st) {
  const size_t smem = sizeof(GemmSmem<BN_MAX, STAGES, QUANT>) + 1024;
  auto kern = grouped_gemm_kernel<BN_MAX, STAGES, QUANT>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<num_sms, GemmRoles<QUANT>::kThreads, smem, st>>>(m.a, m.a_s, m.b, m.b_s, m.sc, m.sc_s, p);
  return cudaGetLastError();
}

cudaError_t launch_grouped_gemm(const GemmParams& p, const GemmMaps& maps, int bn_max, int quant,
                                int num_sms, cudaStream_t st) {
  if (quant == 0) {
    if (bn_max == 64) return launch_variant<64, 8, 0>(p, maps, num_sms, st);
    if (bn_max == 256) return launch_variant<256, 4, 0>(p, maps, num_sms, st);
  } else if (quant == 1) {
    if (bn_max == 64) return launch_variant<64, 8, 1>(p, maps, num_sms, st);
    if (bn_max == 256) return launch_variant<256, 4, 1>(p, maps, num_sms, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
