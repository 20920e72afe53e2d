// combine.cu -- unpermute and sum the weighted expert outputs into token order.
//
// "Systems engineering playbook: optimizing Qwen 3.5-397B MoE on Ironwood
// (TPU7x)": the reusable "SparseCore unpermute" block (executive summary) and
// section 3 "Option B" (expert outputs are reduced back to their tokens);
// section 1 "Sparse Mixture-of-Experts (MoE)": the shared expert is added.
//
//   y[t][d] = bf16_rne( o_shared[t][d] + sum_{j<k} o[inv_row[t*k+j]][d] )
//
// fp32 sum in that fixed order, then one rounding.  HBM-bound: each thread
// moves 4 consecutive fp32 per source row (16-byte loads), 8 bytes of output.
#include "common.cuh"
#include "kernels.h"

namespace moe {

__global__ void __launch_bounds__(256) combine_kernel(const float4* __restrict__ o,
                                                      const float4* __restrict__ o_shared,
                                                      const int32_t* __restrict__ inv_row, int P,
                                                      int D4, int k, uint2* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int c = blockIdx.y * blockDim.x + threadIdx.x;
  if (c >= D4) return;
  float4 acc = o_shared ? __ldg(o_shared + static_cast<size_t>(t) * D4 + c)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
  const int32_t* rows = inv_row + static_cast<size_t>(t) * k;
  for (int j = 0; j < k; ++j) {
    // a row outside [0, P) (an inv_row that moe_permute did not write) is
    // clamped, so the load stays inside o
    const int r = min(max(__ldg(rows + j), 0), P - 1);
    const float4 v = __ldg(o + static_cast<size_t>(r) * D4 + c);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 out;
  out.x = *reinterpret_cast<const uint32_t*>(&lo);
  out.y = *reinterpret_cast<const uint32_t*>(&hi);
  y[static_cast<size_t>(t) * D4 + c] = out;
}

cudaError_t launch_combine(const float* o, const float* o_shared, const int32_t* inv_row, int T,
                           int P, int D, int k, void* y, cudaStream_t st) {
  const int D4 = D / 4;
  dim3 grid(T, (D4 + 255) / 256);
  return pdl_launch(combine_kernel, grid, dim3(256), 0, st, reinterpret_cast<const float4*>(o),
                    reinterpret_cast<const float4*>(o_shared), inv_row, P, D4, k,
                    static_cast<uint2*>(y));
}

// Expert-parallel slice ("Option B": each device sums the outputs of its own
// experts; the devices' fp32 partials are then reduce-scattered):
//   y32[t][d] = (s0 <= t < s1 ? o_shared[t - s0][d] : 0)
//             + sum_{j<k, lo <= inv_row[t*k+j] < hi} o[inv_row[t*k+j]][d]
// with lo, hi read from the device (the local experts' grouped-row range).
__global__ void __launch_bounds__(256) combine_partial_kernel(
    const float4* __restrict__ o, const float4* __restrict__ o_shared,
    const int32_t* __restrict__ inv_row, int T, int D4, int k, const int32_t* __restrict__ row_lo,
    const int32_t* __restrict__ row_hi, int s0, int s1, float4* __restrict__ y32) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int c = blockIdx.y * blockDim.x + threadIdx.x;
  if (c >= D4) return;
  const int lo = __ldg(row_lo), hi = __ldg(row_hi);
  float4 acc = (o_shared && t >= s0 && t < s1)
                   ? __ldg(o_shared + static_cast<size_t>(t - s0) * D4 + c)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
  const int32_t* rows = inv_row + static_cast<size_t>(t) * k;
  for (int j = 0; j < k; ++j) {
    const int r = __ldg(rows + j);
    if (r < lo || r >= hi) continue;
    const float4 v = __ldg(o + static_cast<size_t>(r) * D4 + c);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  y32[static_cast<size_t>(t) * D4 + c] = acc;
}

cudaError_t launch_combine_partial(const float* o, const float* o_shared, const int32_t* inv_row,
                                   int T, int D, int k, const int32_t* row_lo,
                                   const int32_t* row_hi, int s0, int s1, float* y32,
                                   cudaStream_t st) {
  const int D4 = D / 4;
  dim3 grid(T, (D4 + 255) / 256);
  return pdl_launch(combine_partial_kernel, grid, dim3(256), 0, st,
                    reinterpret_cast<const float4*>(o), reinterpret_cast<const float4*>(o_shared),
                    inv_row, T, D4, k, row_lo, row_hi, s0, s1, reinterpret_cast<float4*>(y32));
}

// ------------------------------------------------------------------
// Self-test of the bounded-wait path every pipelined kernel relies on: one CTA
// holds TMEM, waits on an mbarrier that nothing arrives on, gives up after
// `limit_ns`, records MOE_ERR_TIMEOUT in the status word, frees TMEM and exits.
__global__ void __launch_bounds__(32) selftest_wait_kernel(int* status,
                                                           unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  tmem_alloc(&tmem, 32);
  tmem_relinquish();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, &abort_flag, limit_ns)) {
    abort_flag = 1;
    atomicCAS(status, 0, MOE_ERR_TIMEOUT);
  }
  __syncthreads();
  __syncwarp();
  tc_fence_after();
  tmem_dealloc(tmem, 32);
}

cudaError_t launch_selftest_wait(int* status, unsigned long long limit_ns, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
