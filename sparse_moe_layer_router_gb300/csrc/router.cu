// router.cu -- softmax router with top-k selection (sm_103a).
//
// "Systems engineering playbook: optimizing Qwen 3.5-397B MoE on Ironwood
// (TPU7x)", section 1, "Sparse Mixture-of-Experts (MoE)": the router gate
// projects the token representation, forms a softmax over the experts and
// keeps the top-k routed experts; the selected probabilities are renormalised.
// Section 3, "3-to-2 All-Gather optimisation": ids and weights are packed into
// one int32 blob [T][2][k].
//
// Routing decision.  The deciding logit is defined as the fp64 sum, in index
// order, of the exact products x[t,d]*Wr[e,d] (plus the fp32 bias, added
// last).  The GPU computes fp32 logits v on the tensor cores, one fresh
// accumulator per 64-wide K chunk whose fp32 values are then added in order,
// so |v - z| <= r = gamma * ||x_t|| * ||Wr_e|| + 2^-23 |v| (the Cauchy-Schwarz
// bound on sum |x_d Wr_ed|; gamma covers the chunk accumulation, the chunk and
// split sums and the fp64 definition's own deviation).  A token whose k-th /
// (k+1)-th boundary is separated by these intervals is certified; otherwise
// the experts whose intervals straddle the boundary are recomputed with a
// compensated fp32 dot product whose rigorous radius is ~1e-10 of
// sum |x_d w_d| (level 2), and only if that still cannot separate them with
// the defining fp64 index-order sum itself (level 3: exact ties).  The result
// equals the definition's decision (ties: lower index).
#include "common.cuh"
#include "kernels.h"

namespace moe {

// ---------------------------------------------------------------- logits (tensor cores)
// z_part[split][t][e] = sum over the split's k-blocks of x[t, kb] . Wr[e, kb]
// (64-wide K chunks).  A CTA computes 128 experts (MMA M, TMEM lanes) x 64
// tokens (MMA N) for one split: every k-block is four chained bf16 MMAs into a
// fresh fp32 accumulator (one of two TMEM buffers), which the four epilogue
// warps read and add, in k-block order, to running fp32 sums in registers.
// The tensor core's fp32 accumulation order and rounding are not documented;
// the error radius assumes at most 2^-15 * sum|x w| over each 64-wide chunk
// (about four times the bound of an accumulation that aligns the terms to the
// largest one and truncates to 24 bits), and a GPU test checks the measured
// error against a bound twice as tight.  Warp 0: TMA producer; warp 1:
// TMEM allocation and MMA issue; warps 2-5: epilogue.
constexpr int kRtE = 128, kRtT = 64, kRtStages = 4;

struct RouterTcSmem {
  uint8_t a[kRtStages][kRtE * 128];  // router rows, one k-block (128-B swizzle)
  uint8_t b[kRtStages][kRtT * 128];  // token rows, one k-block
  uint64_t full[kRtStages], empty[kRtStages];
  uint64_t cfull[2], cempty[2], drain;
  uint32_t tmem_base;
  int abort_flag;
};

__global__ void __launch_bounds__(192, 1) router_logits_tc_kernel(
    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x, int T,
    int E, int nkb, int kbs, float* __restrict__ z_part, int* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  RouterTcSmem& s =
      *reinterpret_cast<RouterTcSmem*>(smem_raw + (((raw + 1023u) & ~1023u) - raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.x * kRtE, t0 = blockIdx.y * kRtT, sp = blockIdx.z;
  const int kb_begin = sp * kbs;
  const int nk = max(0, min(nkb, kb_begin + kbs) - kb_begin);
  volatile int* abort_flag = &s.abort_flag;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRtStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.cfull[i], 1);
      mbar_init(&s.cempty[i], 4);
    }
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_x);
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_base;
  auto fail = [&]() {
    *abort_flag = 1;
    if (status) atomicCAS(status, 0, MOE_ERR_TIMEOUT);
  };

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      uint32_t issued = 0, issued_ph = 0;
      bool ok = true;
      for (int c = 0; c < nk; ++c) {
        const int st = c % kRtStages;
        const uint32_t ph = (c / kRtStages) & 1u;
        if (!mbar_wait(&s.empty[st], ph ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&s.full[st], (kRtE + kRtT) * 128);
        issued |= 1u << st;
        issued_ph = (issued_ph & ~(1u << st)) | (ph << st);
        tma_load_2d(s.a[st], &tm_w, &s.full[st], (kb_begin + c) * 64, e0, pol);
        tma_load_2d(s.b[st], &tm_x, &s.full[st], (kb_begin + c) * 64, t0, pol);
      }
      if (!ok) {
        fail();
        for (int i = 0; i < kRtStages; ++i)
          if ((issued >> i) & 1u) mbar_wait_time_only(&s.full[i], (issued_ph >> i) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kRtE, kRtT);
      bool ok = true;
      for (int c = 0; c < nk; ++c) {
        const int st = c % kRtStages, buf = c & 1;
        if (!mbar_wait(&s.cempty[buf], ((c >> 1) & 1u) ^ 1u, abort_flag) ||
            !mbar_wait(&s.full[st], (c / kRtStages) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = sdesc_sw128(smem_u32(s.a[st])), bd = sdesc_sw128(smem_u32(s.b[st]));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ss(tmem_base + static_cast<uint32_t>(buf * kRtT), ad + 2u * kk, bd + 2u * kk,
                      idesc, kk != 0 ? 1u : 0u);
        mma_commit(&s.empty[st]);
        mma_commit(&s.cfull[buf]);
      }
      if (!ok) fail();
      mma_commit(&s.drain);
      mbar_wait_time_only(&s.drain, 0);
    }
  } else {
    // epilogue: lane quarter warp % 4 holds experts e0 + 32 * (warp % 4) + lane
    const int q = warp & 3;
    const int e = e0 + 32 * q + lane;
    float run[kRtT];
#pragma unroll
    for (int j = 0; j < kRtT; ++j) run[j] = 0.f;
    bool ok = true;
    for (int c = 0; c < nk; ++c) {
      const int buf = c & 1;
      if (!mbar_wait(&s.cfull[buf], (c >> 1) & 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tb =
          tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(buf * kRtT);
      uint32_t v[4][16];
#pragma unroll
      for (int g = 0; g < 4; ++g) tmem_ld_32x32b_x16(tb + 16u * g, v[g]);
      tmem_wait_ld();
#pragma unroll
      for (int g = 0; g < 4; ++g) tmem_regs_ready(v[g]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.cempty[buf]);
#pragma unroll
      for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int j = 0; j < 16; ++j) run[16 * g + j] += __uint_as_float(v[g][j]);
    }
    if (!ok) {
      fail();
    } else if (e < E) {
      float* dst = z_part + static_cast<size_t>(sp) * T * E + e;
#pragma unroll
      for (int j = 0; j < kRtT; ++j)
        if (t0 + j < T) dst[static_cast<size_t>(t0 + j) * E] = run[j];
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 128);
  }
}

// Sums of squares of the token rows (xsq[t]) and router rows (wsq[e]), one warp
// per row: each lane adds D/32 squares in order, then a five-step butterfly,
// so every square passes through at most D/32 + 5 fp32 roundings.
__global__ void __launch_bounds__(256) router_sumsq_kernel(const __nv_bfloat16* __restrict__ x,
                                                           const __nv_bfloat16* __restrict__ wr,
                                                           int T, int E, int D,
                                                           float* __restrict__ xsq,
                                                           float* __restrict__ wsq) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= T + E) return;
  const uint4* src = reinterpret_cast<const uint4*>(
      row < T ? x + static_cast<size_t>(row) * D : wr + static_cast<size_t>(row - T) * D);
  float acc = 0.f;
  for (int g = lane; g < D / 8; g += 32) {
    const uint4 v = __ldg(src + g);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
      acc = fmaf(lo, lo, acc);
      acc = fmaf(hi, hi, acc);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) {
    if (row < T)
      xsq[row] = acc;
    else
      wsq[row - T] = acc;
  }
}

// ---------------------------------------------------------------- select
// Upper bound of a Euclidean norm from an fp32 sum of squares: each square
// passes through at most D/32 + 5 roundings (router_sumsq_kernel), relative
// error below 2^-9 for D <= 65536.  A rounding whose result falls below the
// normal range (2^-126) is off by up to 2^-150 in absolute terms instead, and
// there are at most D + 32 of them, below 2^-133 in total for D <= 65536.
// sqrt and the products add 2^-20 of slack.
__device__ __forceinline__ float norm_bound(float sumsq) {
  return sqrtf(fmaf(sumsq, 1.0f + 0x1p-9f, 0x1p-133f)) * (1.0f + 0x1p-20f);
}

// Absolute part of the level-1 radius.  The tensor core may flush to zero an
// input, a product or a partial sum below the fp32 normal range: a lost
// product with a subnormal input is below 2^-126 times the other operand, a
// lost product of normal inputs or a lost partial sum below 2^-126, and there
// are at most D products and D partial sums per logit, so the loss is below
// 2^-126 (2D + sum_d |x_d| + sum_d |w_d|) <= 2^-126 (2D + sqrt(D) (|x| + |w|));
// a factor of 4 of slack on top.
__device__ __forceinline__ float tiny_radius1(int D, float xn, float wn) {
  return 0x1p-124f * (2.0f * static_cast<float>(D) + sqrtf(static_cast<float>(D)) * (xn + wn));
}

// Absolute part of the level-2 radius: level 2 forms every product and sum in
// fp32 on the CUDA cores with subnormals kept, so a result below 2^-126 is off
// by at most 2^-150, and a logit takes at most D + 64 such roundings.
__device__ __forceinline__ float tiny_radius2(int D) {
  return 0x1p-148f * static_cast<float>(D + 64);
}

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bp = s - a;
  e = (a - (s - bp)) + (b - bp);  // a + b == s + e exactly
}

// Level 2: compensated fp32 dot product of a token row and a router row (+ bias),
// warp-cooperative.  Products of two bf16 are exact in fp32 down to the normal
// range (below it, tiny_radius2 covers their rounding); every addition is
// an error-free TwoSum whose error term is collected in `c`; lanes combine
// (sum, error) pairs with TwoSum in a butterfly, so every lane ends with the
// same value.  |(s + c) - exact| <= gamma2 * sum|x_d w_d|, with
// gamma2 set by the host from D (about 1e-10 at D = 4096).  The (sum, error)
// pair (s, c) is returned unevaluated: the value is s + c.
__device__ float2 warp_dot_comp(const __nv_bfloat16* __restrict__ xr,
                               const __nv_bfloat16* __restrict__ wrow, int D,
                               const float* __restrict__ bias, int e, int lane) {
  float s = 0.f, c = 0.f;
  const uint4* xp = reinterpret_cast<const uint4*>(xr);
  const uint4* wp = reinterpret_cast<const uint4*>(wrow);
#pragma unroll 8
  for (int g = lane; g < D / 8; g += 32) {
    const uint4 xv = __ldg(xp + g), wv = __ldg(wp + g);
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float t, err;
      two_sum(s, __uint_as_float(xw[j] << 16) * __uint_as_float(ww[j] << 16), t, err);
      s = t;
      c += err;
      two_sum(s, __uint_as_float(xw[j] & 0xFFFF0000u) * __uint_as_float(ww[j] & 0xFFFF0000u), t,
              err);
      s = t;
      c += err;
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float so = __shfl_xor_sync(0xffffffffu, s, o);
    const float co = __shfl_xor_sync(0xffffffffu, c, o);
    float t, err;
    two_sum(s, so, t, err);
    s = t;
    c = (c + co) + err;
  }
  if (bias) {
    float t, err;
    two_sum(s, bias[e], t, err);
    s = t;
    c += err;
  }
  return make_float2(s, c);
}

// Level 3: the defining logit itself -- fp64 sum in index order d = 0..D-1 of
// the exact products (+ bias last).  The warp stages 256-element chunks of both
// rows in shared memory (`stage`: 2 x 256 bf16 per warp); lane 0 runs the chain.
// Every lane returns the value.
__device__ double warp_exact_logit(const __nv_bfloat16* __restrict__ xr,
                                   const __nv_bfloat16* __restrict__ wrow, int D,
                                   const float* __restrict__ bias, int e, int lane,
                                   uint4* stage) {
  double acc = 0.0;
  const uint4* xp = reinterpret_cast<const uint4*>(xr);
  const uint4* wp = reinterpret_cast<const uint4*>(wrow);
  for (int c = 0; c < D / 8; c += 32) {
    const bool in = c + lane < D / 8;
    const uint4 xv = in ? __ldg(xp + c + lane) : make_uint4(0, 0, 0, 0);
    const uint4 wv = in ? __ldg(wp + c + lane) : make_uint4(0, 0, 0, 0);
    __syncwarp();
    stage[lane] = xv;
    stage[32 + lane] = wv;
    __syncwarp();
    if (lane == 0) {
      const int n = min(32, D / 8 - c);
      for (int g = 0; g < n; ++g) {
        const uint4 a = stage[g], b = stage[32 + g];
        const uint32_t xw[4] = {a.x, a.y, a.z, a.w};
        const uint32_t ww[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // the product of two bf16 widened to fp64 is exact over the whole
          // bf16 range (16 significant bits, exponents within fp64's range),
          // so adding it in fp64 is the definition's step
          acc += static_cast<double>(__uint_as_float(xw[j] << 16)) *
                 static_cast<double>(__uint_as_float(ww[j] << 16));
          acc += static_cast<double>(__uint_as_float(xw[j] & 0xFFFF0000u)) *
                 static_cast<double>(__uint_as_float(ww[j] & 0xFFFF0000u));
        }
      }
    }
  }
  if (lane == 0 && bias) acc += static_cast<double>(bias[e]);
  return __shfl_sync(0xffffffffu, acc, 0);
}

// Order used for selection: larger value first, lower index on an exact tie;
// a NaN logit orders below every number (-inf included), NaNs among
// themselves by index.  Every search starts from the sentinel (NaN, INT_MAX),
// which any expert beats, so each of the k rounds picks an expert whatever
// the logits hold and the blob always gets k distinct ids in [0, E).
__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
  const bool vn = v != v, bn = bv != bv;
  if (vn || bn) return bn && (!vn || e < be);
  return v > bv || (v == bv && e < be);
}
__device__ __forceinline__ bool better_d(double v, int e, double bv, int be) {
  const bool vn = v != v, bn = bv != bv;
  if (vn || bn) return bn && (!vn || e < be);
  return v > bv || (v == bv && e < be);
}
__device__ __forceinline__ float sentinel_f() { return __int_as_float(0x7fc00000); }
__device__ __forceinline__ double sentinel_d() {
  return __longlong_as_double(0x7ff8000000000000ll);
}
// The same order for numbers only (no operand is NaN), from the sentinel
// (-inf, INT_MAX).
__device__ __forceinline__ bool better_num(float v, int e, float bv, int be) {
  return v > bv || (v == bv && e < be);
}

// k rounds of warp arg-max: each takes the best expert not yet in `sel` and
// lowers min_lo to its v - r.  kNan selects the NaN-aware order; without a
// NaN logit the plain comparisons give the same order.
template <bool kNan, int VPL>
__device__ __forceinline__ void topk_rounds(const float (&v)[VPL], const float (&r)[VPL], int E,
                                            int k, int lane, uint32_t& sel, float& min_lo) {
  for (int j = 0; j < k; ++j) {
    float bv = kNan ? sentinel_f() : -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((sel >> i) & 1u) &&
          (kNan ? better(v[i], e, bv, be) : better_num(v[i], e, bv, be))) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (kNan ? better(ov, oe, bv, be) : better_num(ov, oe, bv, be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) {
      const int i = be >> 5;
#pragma unroll
      for (int q = 0; q < VPL; ++q)
        if (q == i) {
          sel |= 1u << q;
          min_lo = fminf(min_lo, v[q] - r[q]);
        }
    }
  }
}

// One 256-thread block per token.  All threads sum the split-K partials
// (phase 1); warp 0 selects and certifies (phase 2); the experts that level 2
// must recompute are shared out over the eight warps (phase 3); warp 0
// finishes the decision, the weights and the blob (phase 4).
template <int VPL>
__global__ void __launch_bounds__(256) router_select_kernel(
    const float* __restrict__ z_part, int S, int T, int D, int E, int k,
    const float* __restrict__ bias, const float* __restrict__ xsq_part,
    const float* __restrict__ wsq_part, float gamma, const __nv_bfloat16* __restrict__ x,
    const __nv_bfloat16* __restrict__ wr, int32_t* __restrict__ blob,
    int* __restrict__ counters, float gamma2) {
  pdl_wait();
  pdl_trigger();
  // shared: zx double[E] (level-3 logits) | sc float2[E] (level-2 pairs) |
  //         vs float[E] | wss float[E] | clist int[E] | stage uint4[64]
  extern __shared__ double sel_smem[];
  double* zx = sel_smem;
  float2* sc = reinterpret_cast<float2*>(zx + E);
  float* vs = reinterpret_cast<float*>(sc + E);
  float* wss = vs + E;
  int* clist = reinterpret_cast<int*>(wss + E);
  uint4* stage = reinterpret_cast<uint4*>(sel_smem + (static_cast<size_t>(E) * 28 + 15) / 16 * 2);
  __shared__ int s_ncand;
  __shared__ float s_xsq;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.x;
  if (t >= T) return;
  const __nv_bfloat16* xr = x + static_cast<size_t>(t) * D;

  // ---- phase 1: split-K partials of the logits, summed in split order (loads
  // of four splits are issued before their additions); sums of squares.
  // Up to 16 splits (the host plan's cap) x 2 experts per thread: every load
  // is issued before the first addition, so one memory latency covers them.
  for (int e0 = 0; e0 < E; e0 += 2 * 256) {
    float z[2][16];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int e = e0 + tid + 256 * j;
#pragma unroll
      for (int sp = 0; sp < 16; ++sp)
        z[j][sp] = (e < E && sp < S) ? __ldg(z_part + (static_cast<size_t>(sp) * T + t) * E + e)
                                     : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int e = e0 + tid + 256 * j;
      if (e >= E) continue;
      float a = 0.f;
#pragma unroll
      for (int sp = 0; sp < 16; ++sp)
        if (sp < S) a += z[j][sp];
      vs[e] = a;
      wss[e] = __ldg(wsq_part + e);
    }
  }
  if (tid == 0) {
    s_xsq = __ldg(xsq_part + t);
    s_ncand = 0;
  }
  __syncthreads();

  // ---- phase 2 (warp 0): top-k and certification
  float v[VPL], r[VPL], wn[VPL];
  uint32_t sel = 0, cand = 0;
  int slots = 0;
  const float xn = norm_bound(s_xsq);
  if (warp == 0) {
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      wn[i] = norm_bound(wss[e]);
      v[i] = vs[e] + (bias ? __ldg(bias + e) : 0.f);
      r[i] = gamma * xn * wn[i] * (1.0f + 0x1p-10f) + 0x1p-23f * fabsf(v[i]) +
             tiny_radius1(D, xn, wn[i]);
    } else {
      wn[i] = 0.f;
      v[i] = -INFINITY;
      r[i] = 0.f;
    }
  }

  // k rounds of warp arg-max under (value desc, index asc); the NaN-aware
  // order only for a token with a NaN logit (one warp vote).
  float min_lo = INFINITY;
  bool nan_here = false;
#pragma unroll
  for (int i = 0; i < VPL; ++i) nan_here |= v[i] != v[i];
  if (__any_sync(0xffffffffu, nan_here))
    topk_rounds<true>(v, r, E, k, lane, sel, min_lo);
  else
    topk_rounds<false>(v, r, E, k, lane, sel, min_lo);
  float max_hi = -INFINITY;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E && !((sel >> i) & 1u)) max_hi = fmaxf(max_hi, v[i] + r[i]);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    min_lo = fminf(min_lo, __shfl_xor_sync(0xffffffffu, min_lo, o));
    max_hi = fmaxf(max_hi, __shfl_xor_sync(0xffffffffu, max_hi, o));
  }

  if (!(min_lo > max_hi)) {
    // Not certified: experts whose interval reaches across the boundary.
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e >= E) continue;
      const bool s_in = (sel >> i) & 1u;
      if ((s_in && v[i] - r[i] <= max_hi) || (!s_in && v[i] + r[i] >= min_lo)) cand |= 1u << i;
    }
    slots = __popc(sel & cand);
#pragma unroll
    for (int o = 16; o; o >>= 1) slots += __shfl_xor_sync(0xffffffffu, slots, o);
    if (lane == 0 && counters) atomicAdd(counters, 1);
    // candidate list for phase 3 (ascending i, then lane)
    int base = 0;
    const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const bool c = (cand >> i) & 1u;
      const uint32_t bal = __ballot_sync(0xffffffffu, c);
      if (c) clist[base + __popc(bal & lt_mask)] = lane + 32 * i;
      base += __popc(bal);
    }
    if (lane == 0) s_ncand = base;
  }
  }  // warp 0
  __syncthreads();

  // ---- phase 3 (all warps): level-2 compensated logits of the candidates
  const int ncand = s_ncand;
  for (int c = warp; c < ncand; c += blockDim.x / 32) {
    const int e = clist[c];
    const float2 z2 = warp_dot_comp(xr, wr + static_cast<size_t>(e) * D, D, bias, e, lane);
    if (lane == 0) sc[e] = z2;
  }
  __syncthreads();
  if (warp != 0) return;

  // ---- phase 4 (warp 0): finish the decision
  if (ncand > 0) {
    float zs[VPL], zc[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      zs[i] = zc[i] = 0.f;
      if ((cand >> i) & 1u) {
        const float2 z2 = sc[e];
        zs[i] = z2.x;
        zc[i] = z2.y;
      }
    }
    // Values relative to a common reference (the largest candidate sum s):
    // rel = (s - ref) + c, with |rel - (z - ref)| <= 2^-23 |rel| (s - ref is
    // exact when s is within a factor of two of ref), all in fp32.
    float ref = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if ((cand >> i) & 1u) ref = fmaxf(ref, zs[i]);
#pragma unroll
    for (int o = 16; o; o >>= 1) ref = fmaxf(ref, __shfl_xor_sync(0xffffffffu, ref, o));
    float rel[VPL], rad[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      rel[i] = -INFINITY;
      rad[i] = 0.f;
      if ((cand >> i) & 1u) {
        rel[i] = (zs[i] - ref) + zc[i];
        const float a = xn * wn[i] + (bias ? fabsf(bias[e]) : 0.f);
        // gamma2 * sum|x w| (level-2 error, plus the fp64 definition's own
        // distance from the exact sum) + rounding of rel and of rel -/+ rad
        rad[i] = gamma2 * a * (1.0f + 0x1p-20f) + 0x1p-21f * fabsf(rel[i]) + tiny_radius2(D);
      }
    }
    uint32_t chosen = 0;
    for (int j = 0; j < slots; ++j) {
      float bv = sentinel_f();
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (((cand >> i) & 1u) && !((chosen >> i) & 1u) && better(rel[i], e, bv, be)) {
          bv = rel[i];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (better(ov, oe, bv, be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) chosen |= 1u << (be >> 5);
    }
    float lo = INFINITY, hi = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      if (!((cand >> i) & 1u)) continue;
      if ((chosen >> i) & 1u)
        lo = fminf(lo, rel[i] - rad[i]);
      else
        hi = fmaxf(hi, rel[i] + rad[i]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    // Refined logits replace the fp32 ones for the weights.
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if ((cand >> i) & 1u) v[i] = zs[i] + zc[i];
    if (!(lo > hi)) {
      // Level 3: the defining index-order fp64 sum (exact ties end here).
      if (lane == 0 && counters) atomicAdd(counters + 1, 1);
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        uint32_t bal = __ballot_sync(0xffffffffu, (cand >> i) & 1u);
        while (bal) {
          const int src = __ffs(bal) - 1;
          bal &= bal - 1;
          const int e = src + 32 * i;
          const double z =
              warp_exact_logit(xr, wr + static_cast<size_t>(e) * D, D, bias, e, lane, stage);
          if (lane == src) zx[e] = z;
        }
      }
      __syncwarp();
      chosen = 0;
      for (int j = 0; j < slots; ++j) {
        double bv = sentinel_d();
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int e = lane + 32 * i;
          if (((cand >> i) & 1u) && !((chosen >> i) & 1u) && better_d(zx[e], e, bv, be)) {
            bv = zx[e];
            be = e;
          }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const double ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oe = __shfl_xor_sync(0xffffffffu, be, o);
          if (better_d(ov, oe, bv, be)) {
            bv = ov;
            be = oe;
          }
        }
        if ((be & 31) == lane) chosen |= 1u << (be >> 5);
      }
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if ((cand >> i) & 1u) v[i] = static_cast<float>(zx[e]);
      }
    }
    sel = (sel & ~cand) | chosen;
  }

  // Softmax over all E, renormalised over the selected k:
  //   w_j = exp(v_j - m) / sum_selected exp(v_i - m)   (the full denominator cancels).
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < VPL; ++i) m = fmaxf(m, v[i]);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float ex[VPL];
  float den = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    ex[i] = ((sel >> i) & 1u) ? expf(v[i] - m) : 0.f;
    den += ex[i];
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);

  // Ascending expert order: e = lane + 32 i, so scan i outer, lanes inner.
  int32_t* out = blob + static_cast<size_t>(t) * 2 * k;
  int base = 0;
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const bool s_in = (sel >> i) & 1u;
    const uint32_t bal = __ballot_sync(0xffffffffu, s_in);
    if (s_in) {
      const int pos = base + __popc(bal & lt_mask);
      out[pos] = lane + 32 * i;
      out[k + pos] = __float_as_int(ex[i] / den);
    }
    base += __popc(bal);
  }
}

// Warp-per-token variant for T >= 512 (eight tokens per block): the same
// decision as router_select_kernel, with the level-2 candidates of a token
// recomputed one after another by its warp.
template <int VPL>
__global__ void __launch_bounds__(256) router_select_warp_kernel(
    const float* __restrict__ z_part, int S, int T, int D, int E, int k,
    const float* __restrict__ bias, const float* __restrict__ xsq_part,
    const float* __restrict__ wsq_part, float gamma, const __nv_bfloat16* __restrict__ x,
    const __nv_bfloat16* __restrict__ wr, int32_t* __restrict__ blob,
    int* __restrict__ counters, float gamma2) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ double zx_smem[];  // [8 warps][E] refined logits, then [8][64] uint4 staging
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + wib;
  if (t >= T) return;
  double* zx = zx_smem + static_cast<size_t>(wib) * E;
  uint4* stage = reinterpret_cast<uint4*>(zx_smem + static_cast<size_t>(8) * E) + wib * 64;

  float v[VPL], r[VPL], wn[VPL];
  uint32_t sel = 0, cand = 0;
  // Split-K partials of the logits summed in split order; the VPL loads of one
  // split are independent and coalesced across the warp.
  const float xsq = __ldg(xsq_part + t);
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = 0.f;
    wn[i] = e < E ? __ldg(wsq_part + e) : 0.f;
  }
  for (int sp = 0; sp < S; ++sp) {
    const float* zp = z_part + (static_cast<size_t>(sp) * T + t) * E;
    float part[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      part[i] = e < E ? __ldg(zp + e) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) v[i] += part[i];
  }
  const float xn = norm_bound(xsq);
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    wn[i] = norm_bound(wn[i]);
    if (e < E) {
      if (bias) v[i] += __ldg(bias + e);
      r[i] = gamma * xn * wn[i] * (1.0f + 0x1p-10f) + 0x1p-23f * fabsf(v[i]) +
             tiny_radius1(D, xn, wn[i]);
    } else {
      v[i] = -INFINITY;
      r[i] = 0.f;
    }
  }

  // k rounds of warp arg-max under (value desc, index asc); the NaN-aware
  // order only for a token with a NaN logit (one warp vote).
  float min_lo = INFINITY;
  bool nan_here = false;
#pragma unroll
  for (int i = 0; i < VPL; ++i) nan_here |= v[i] != v[i];
  if (__any_sync(0xffffffffu, nan_here))
    topk_rounds<true>(v, r, E, k, lane, sel, min_lo);
  else
    topk_rounds<false>(v, r, E, k, lane, sel, min_lo);
  float max_hi = -INFINITY;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E && !((sel >> i) & 1u)) max_hi = fmaxf(max_hi, v[i] + r[i]);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    min_lo = fminf(min_lo, __shfl_xor_sync(0xffffffffu, min_lo, o));
    max_hi = fmaxf(max_hi, __shfl_xor_sync(0xffffffffu, max_hi, o));
  }

  if (!(min_lo > max_hi)) {
    // Not certified: experts whose interval reaches across the boundary.
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e >= E) continue;
      const bool s_in = (sel >> i) & 1u;
      if ((s_in && v[i] - r[i] <= max_hi) || (!s_in && v[i] + r[i] >= min_lo)) cand |= 1u << i;
    }
    int slots = __popc(sel & cand);
#pragma unroll
    for (int o = 16; o; o >>= 1) slots += __shfl_xor_sync(0xffffffffu, slots, o);
    if (lane == 0 && counters) atomicAdd(counters, 1);
    const __nv_bfloat16* xr = x + static_cast<size_t>(t) * D;
    // Level 2: compensated fp32 logits of every candidate, kept as the
    // unevaluated pair (s, c) by the lane that owns the expert.
    float zs[VPL], zc[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      zs[i] = zc[i] = 0.f;
      uint32_t bal = __ballot_sync(0xffffffffu, (cand >> i) & 1u);
      while (bal) {
        const int src = __ffs(bal) - 1;
        bal &= bal - 1;
        const int e = src + 32 * i;
        const float2 sc = warp_dot_comp(xr, wr + static_cast<size_t>(e) * D, D, bias, e, lane);
        if (lane == src) {
          zs[i] = sc.x;
          zc[i] = sc.y;
        }
      }
    }
    // Values relative to a common reference (the largest candidate sum s):
    // rel = (s - ref) + c, with |rel - (z - ref)| <= 2^-23 |rel| (s - ref is
    // exact when s is within a factor of two of ref), all in fp32.
    float ref = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if ((cand >> i) & 1u) ref = fmaxf(ref, zs[i]);
#pragma unroll
    for (int o = 16; o; o >>= 1) ref = fmaxf(ref, __shfl_xor_sync(0xffffffffu, ref, o));
    float rel[VPL], rad[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      rel[i] = -INFINITY;
      rad[i] = 0.f;
      if ((cand >> i) & 1u) {
        rel[i] = (zs[i] - ref) + zc[i];
        const float a = xn * wn[i] + (bias ? fabsf(bias[e]) : 0.f);
        // gamma2 * sum|x w| (level-2 error, plus the fp64 definition's own
        // distance from the exact sum) + rounding of rel and of rel -/+ rad
        rad[i] = gamma2 * a * (1.0f + 0x1p-20f) + 0x1p-21f * fabsf(rel[i]) + tiny_radius2(D);
      }
    }
    uint32_t chosen = 0;
    for (int j = 0; j < slots; ++j) {
      float bv = sentinel_f();
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (((cand >> i) & 1u) && !((chosen >> i) & 1u) && better(rel[i], e, bv, be)) {
          bv = rel[i];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (better(ov, oe, bv, be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) chosen |= 1u << (be >> 5);
    }
    float lo = INFINITY, hi = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      if (!((cand >> i) & 1u)) continue;
      if ((chosen >> i) & 1u)
        lo = fminf(lo, rel[i] - rad[i]);
      else
        hi = fmaxf(hi, rel[i] + rad[i]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    // Refined logits replace the fp32 ones for the weights.
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if ((cand >> i) & 1u) v[i] = zs[i] + zc[i];
    if (!(lo > hi)) {
      // Level 3: the defining index-order fp64 sum (exact ties end here).
      if (lane == 0 && counters) atomicAdd(counters + 1, 1);
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        uint32_t bal = __ballot_sync(0xffffffffu, (cand >> i) & 1u);
        while (bal) {
          const int src = __ffs(bal) - 1;
          bal &= bal - 1;
          const int e = src + 32 * i;
          const double z =
              warp_exact_logit(xr, wr + static_cast<size_t>(e) * D, D, bias, e, lane, stage);
          if (lane == src) zx[e] = z;
        }
      }
      __syncwarp();
      chosen = 0;
      for (int j = 0; j < slots; ++j) {
        double bv = sentinel_d();
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int e = lane + 32 * i;
          if (((cand >> i) & 1u) && !((chosen >> i) & 1u) && better_d(zx[e], e, bv, be)) {
            bv = zx[e];
            be = e;
          }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const double ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oe = __shfl_xor_sync(0xffffffffu, be, o);
          if (better_d(ov, oe, bv, be)) {
            bv = ov;
            be = oe;
          }
        }
        if ((be & 31) == lane) chosen |= 1u << (be >> 5);
      }
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if ((cand >> i) & 1u) v[i] = static_cast<float>(zx[e]);
      }
    }
    sel = (sel & ~cand) | chosen;
  }

  // Softmax over all E, renormalised over the selected k:
  //   w_j = exp(v_j - m) / sum_selected exp(v_i - m)   (the full denominator cancels).
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < VPL; ++i) m = fmaxf(m, v[i]);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float ex[VPL];
  float den = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    ex[i] = ((sel >> i) & 1u) ? expf(v[i] - m) : 0.f;
    den += ex[i];
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);

  // Ascending expert order: e = lane + 32 i, so scan i outer, lanes inner.
  int32_t* out = blob + static_cast<size_t>(t) * 2 * k;
  int base = 0;
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const bool s_in = (sel >> i) & 1u;
    const uint32_t bal = __ballot_sync(0xffffffffu, s_in);
    if (s_in) {
      const int pos = base + __popc(bal & lt_mask);
      out[pos] = lane + 32 * i;
      out[k + pos] = __float_as_int(ex[i] / den);
    }
    base += __popc(bal);
  }
}


// ---------------------------------------------------------------- launchers
cudaError_t launch_router_logits_tc(const CUtensorMap& tm_w, const CUtensorMap& tm_x,
                                    const void* x, const void* wr, int T, int D, int E, int S,
                                    int kbs, float* z_part, float* xsq, float* wsq, int* status,
                                    cudaStream_t st) {
  cudaError_t e = pdl_launch(router_sumsq_kernel, dim3((T + E + 7) / 8), dim3(256), 0, st,
                             static_cast<const __nv_bfloat16*>(x),
                             static_cast<const __nv_bfloat16*>(wr), T, E, D, xsq, wsq);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(RouterTcSmem) + 1024;
  e = cudaFuncSetAttribute(router_logits_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((E + kRtE - 1) / kRtE, (T + kRtT - 1) / kRtT, S);
  return pdl_launch(router_logits_tc_kernel, grid, dim3(192), smem, st, tm_w, tm_x, T, E, D / 64,
                    kbs, z_part, status);
}

cudaError_t launch_router_select(const float* z_part, int S, int T, int D, int E, int k,
                                 const float* bias, const float* xsq_part, const float* wsq_part,
                                 float gamma, float gamma2, const void* x, const void* wr,
                                 int32_t* blob, int* counters, cudaStream_t st) {
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  const auto* wb = static_cast<const __nv_bfloat16*>(wr);
  // Small batches: one block per token keeps every SM busy; from 512 tokens a
  // warp per token is faster (measured 52 vs 64 us for the router at T=1024).
  const bool per_warp = T >= 512;
  const int blocks = per_warp ? (T + 7) / 8 : T;
  const size_t smem =
      per_warp ? static_cast<size_t>(8) * E * sizeof(double) + 8 * 64 * sizeof(uint4)
               : (static_cast<size_t>(E) * 28 + 15) / 16 * 16 + 64 * sizeof(uint4);
#define MOE_SELECT_CASE(V)                                                                    \
  if (E <= 32 * (V)) {                                                                        \
    auto kern = per_warp ? router_select_warp_kernel<V> : router_select_kernel<V>;            \
    if (smem > 48 * 1024) {                                                                   \
      cudaError_t e_ = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                            static_cast<int>(smem));                          \
      if (e_ != cudaSuccess) return e_;                                                       \
    }                                                                                         \
    return pdl_launch(kern, dim3(blocks), dim3(256), smem, st, z_part, S, T, D, E, k, bias,  \
                      xsq_part, wsq_part, gamma, xb, wb, blob, counters, gamma2);             \
  }
  MOE_SELECT_CASE(1)
  MOE_SELECT_CASE(4)
  MOE_SELECT_CASE(16)
  MOE_SELECT_CASE(32)
#undef MOE_SELECT_CASE
  return cudaErrorInvalidValue;
}

}  // namespace moe
