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
// last).  The GPU computes fp32 logits v with a summation tree of bounded
// depth h, so |v - z| <= r = gamma_h * ||x_t|| * ||Wr_e|| + 2^-23 |v| (the
// Cauchy-Schwarz bound on sum |x_d Wr_ed|, plus the fp64 definition's own
// deviation folded into gamma).  A token whose k-th / (k+1)-th boundary is
// separated by these intervals is certified; otherwise the experts whose
// intervals straddle the boundary are recomputed with a compensated fp32 dot
// product whose rigorous radius is ~1e-10 of sum |x_d w_d| (level 2), and only
// if that still cannot separate them with the defining fp64 index-order sum
// itself (level 3: exact ties).  The result equals the definition's decision
// (ties: lower index).
#include "common.cuh"
#include "kernels.h"

namespace moe {

// ---------------------------------------------------------------- logits
// z_part[split][t][e] = sum over the split's K range of x[t,k] * Wr[e,k] (fp32).
// Within the range, products are accumulated in sub-chunks of 64 (a fresh fp32
// accumulator each) and sub-chunk sums are added to the running total, so each
// product passes through at most 64 + sub_per_split roundings.
// The same pass also produces partial sums of squares of the x rows (CTAs with
// blockIdx.x == 0) and of the router rows (blockIdx.y == 0) for the error
// radius; every element is squared once per split.
// Global loads of chunk c+1 are issued before chunk c is multiplied (register
// staging, two shared-memory buffers, one barrier per 32-wide chunk).
constexpr int kRT = 64, kRE = 64, kRK = 32;

__global__ void __launch_bounds__(256) router_logits_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ wr, int T, int D,
    int E, int sub_per_split, float* __restrict__ z_part, float* __restrict__ xsq_part,
    float* __restrict__ wsq_part) {
  __shared__ __align__(16) float xs[2][kRK][kRT + 4];
  __shared__ __align__(16) float ws[2][kRK][kRE + 4];
  const int e0 = blockIdx.x * kRE, t0 = blockIdx.y * kRT, split = blockIdx.z;
  const int nsub = D / 64;
  const int sub_begin = split * sub_per_split;
  const int sub_end = min(nsub, sub_begin + sub_per_split);
  const int nchunks = 2 * max(0, sub_end - sub_begin);
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int lrow = tid >> 2, lk = (tid & 3) * 8;
  const bool xrow_ok = t0 + lrow < T, wrow_ok = e0 + lrow < E;
  const __nv_bfloat16* xsrc = x + static_cast<size_t>(t0 + lrow) * D + lk;
  const __nv_bfloat16* wsrc = wr + static_cast<size_t>(e0 + lrow) * D + lk;
  uint4 xv = make_uint4(0, 0, 0, 0), wv = make_uint4(0, 0, 0, 0);
  float xsq = 0.f, wsq = 0.f;

  auto gload = [&](int c) {
    const int kbase = sub_begin * 64 + c * kRK;
    if (xrow_ok) xv = __ldg(reinterpret_cast<const uint4*>(xsrc + kbase));
    if (wrow_ok) wv = __ldg(reinterpret_cast<const uint4*>(wsrc + kbase));
  };
  auto sstore = [&](int buf) {
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float xl = __uint_as_float(xw[j] << 16), xh = __uint_as_float(xw[j] & 0xFFFF0000u);
      const float wl = __uint_as_float(ww[j] << 16), wh = __uint_as_float(ww[j] & 0xFFFF0000u);
      xs[buf][lk + 2 * j][lrow] = xl;
      xs[buf][lk + 2 * j + 1][lrow] = xh;
      ws[buf][lk + 2 * j][lrow] = wl;
      ws[buf][lk + 2 * j + 1][lrow] = wh;
      xsq = fmaf(xh, xh, fmaf(xl, xl, xsq));
      wsq = fmaf(wh, wh, fmaf(wl, wl, wsq));
    }
  };

  float acc[4][4], part[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = part[i][j] = 0.f;

  if (nchunks > 0) {
    gload(0);
    sstore(0);
  }
  __syncthreads();
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    if (c + 1 < nchunks) gload(c + 1);
#pragma unroll
    for (int kk = 0; kk < kRK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&xs[buf][kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&ws[buf][kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) part[i][j] = fmaf(av[i], bv[j], part[i][j]);
    }
    if (c & 1) {  // end of a 64-wide sub-chunk
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] += part[i][j];
          part[i][j] = 0.f;
        }
    }
    if (c + 1 < nchunks) sstore(buf ^ 1);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
    float* dst = z_part + (static_cast<size_t>(split) * T + t) * E;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) dst[e] = acc[i][j];
    }
  }
  // four threads share each staged row: combine their squares
  xsq += __shfl_xor_sync(0xffffffffu, xsq, 1);
  xsq += __shfl_xor_sync(0xffffffffu, xsq, 2);
  wsq += __shfl_xor_sync(0xffffffffu, wsq, 1);
  wsq += __shfl_xor_sync(0xffffffffu, wsq, 2);
  if ((tid & 3) == 0) {
    if (blockIdx.x == 0 && xrow_ok) xsq_part[static_cast<size_t>(split) * T + t0 + lrow] = xsq;
    if (blockIdx.y == 0 && wrow_ok) wsq_part[static_cast<size_t>(split) * E + e0 + lrow] = wsq;
  }
}

// ---------------------------------------------------------------- select
// Upper bound of a Euclidean norm from split partial sums of squares: the fp32
// sums pass each square through at most D/4 + S + 2 roundings (relative error
// below 2^-9 for D <= 65536); sqrt and the products add 2^-20 of slack.
__device__ __forceinline__ float norm_bound(float sumsq) {
  return sqrtf(sumsq * (1.0f + 0x1p-9f)) * (1.0f + 0x1p-20f);
}

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bp = s - a;
  e = (a - (s - bp)) + (b - bp);  // a + b == s + e exactly
}

// Level 2: compensated fp32 dot product of a token row and a router row (+ bias),
// warp-cooperative.  Products of two bf16 are exact in fp32; every addition is
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
          // the fp32 product of two bf16 is exact, so adding it in fp64 is the
          // definition's step
          acc += static_cast<double>(__uint_as_float(xw[j] << 16) *
                                     __uint_as_float(ww[j] << 16));
          acc += static_cast<double>(__uint_as_float(xw[j] & 0xFFFF0000u) *
                                     __uint_as_float(ww[j] & 0xFFFF0000u));
        }
      }
    }
  }
  if (lane == 0 && bias) acc += static_cast<double>(bias[e]);
  return __shfl_sync(0xffffffffu, acc, 0);
}

// Order used for selection: larger value first, lower index on an exact tie.
__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
  return v > bv || (v == bv && e < be);
}
__device__ __forceinline__ bool better_d(double v, int e, double bv, int be) {
  return v > bv || (v == bv && e < be);
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

  // ---- phase 1: split-K partials of the logits and of the squares, summed in
  // split order; loads of four splits are issued before their additions.
  for (int e = tid; e < E; e += blockDim.x) {
    float a = 0.f, b = 0.f;
    int sp = 0;
    for (; sp + 4 <= S; sp += 4) {
      float z4[4], w4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        z4[q] = __ldg(z_part + (static_cast<size_t>(sp + q) * T + t) * E + e);
        w4[q] = __ldg(wsq_part + static_cast<size_t>(sp + q) * E + e);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a += z4[q];
        b += w4[q];
      }
    }
    for (; sp < S; ++sp) {
      a += __ldg(z_part + (static_cast<size_t>(sp) * T + t) * E + e);
      b += __ldg(wsq_part + static_cast<size_t>(sp) * E + e);
    }
    vs[e] = a;
    wss[e] = b;
  }
  if (tid == 0) {
    float xs = 0.f;
    for (int sp = 0; sp < S; ++sp) xs += __ldg(xsq_part + static_cast<size_t>(sp) * T + t);
    s_xsq = xs;
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
      r[i] = gamma * xn * wn[i] * (1.0f + 0x1p-10f) + 0x1p-23f * fabsf(v[i]);
    } else {
      wn[i] = 0.f;
      v[i] = -INFINITY;
      r[i] = 0.f;
    }
  }

  // k rounds of warp arg-max under (value desc, index asc).
  float min_lo = INFINITY;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((sel >> i) & 1u) && better(v[i], e, bv, be)) {
        bv = v[i];
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
        rad[i] = gamma2 * a * (1.0f + 0x1p-20f) + 0x1p-21f * fabsf(rel[i]);
      }
    }
    uint32_t chosen = 0;
    for (int j = 0; j < slots; ++j) {
      float bv = -INFINITY;
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
        double bv = -INFINITY;
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
void launch_router_logits(const void* x, const void* wr, int T, int D, int E, int S,
                          int sub_per_split, float* z_part, float* xsq_part, float* wsq_part,
                          cudaStream_t st) {
  dim3 grid((E + kRE - 1) / kRE, (T + kRT - 1) / kRT, S);
  router_logits_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x),
                                             static_cast<const __nv_bfloat16*>(wr), T, D, E,
                                             sub_per_split, z_part, xsq_part, wsq_part);
}

cudaError_t launch_router_select(const float* z_part, int S, int T, int D, int E, int k,
                                 const float* bias, const float* xsq_part, const float* wsq_part,
                                 float gamma, float gamma2, const void* x, const void* wr,
                                 int32_t* blob, int* counters, cudaStream_t st) {
  const int blocks = T;
  const size_t smem = (static_cast<size_t>(E) * 28 + 15) / 16 * 16 + 64 * sizeof(uint4);
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  const auto* wb = static_cast<const __nv_bfloat16*>(wr);
#define MOE_SELECT_CASE(V)                                                                   \
  if (E <= 32 * (V)) {                                                                       \
    if (smem > 48 * 1024) {                                                                  \
      cudaError_t e_ = cudaFuncSetAttribute(router_select_kernel<V>,                         \
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,     \
                                            static_cast<int>(smem));                         \
      if (e_ != cudaSuccess) return e_;                                                      \
    }                                                                                        \
    router_select_kernel<V><<<blocks, 256, smem, st>>>(z_part, S, T, D, E, k, bias, xsq_part, \
                                                       wsq_part, gamma, xb, wb, blob,        \
                                                       counters, gamma2);                    \
    return cudaGetLastError();                                                               \
  }
  MOE_SELECT_CASE(1)
  MOE_SELECT_CASE(4)
  MOE_SELECT_CASE(16)
  MOE_SELECT_CASE(32)
#undef MOE_SELECT_CASE
  return cudaErrorInvalidValue;
}

}  // namespace moe
