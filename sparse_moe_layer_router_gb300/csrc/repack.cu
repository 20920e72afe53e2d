// repack.cu -- load-time conversion of packed int4 weights to pair order.
//
// "vLLM TPU Inference v0.31.0: hierarchical MoE dispatch and W4A16", 4-bit
// weight section: symmetric int4 weights in the pack-quantized format, eight
// 4-bit values per int32 in sequential order (value j in bits 4j..4j+3).  The
// grouped GEMM reads pair order instead (value 2i in bits 4i..4i+3, value 2i+1
// in bits 16+4i..19+4i), where one shift and mask place two consecutive values
// in the two 16-bit halves of a register.  In sequential order the even values
// are the low nibbles of the four bytes and the odd values the high nibbles,
// so the conversion packs the low nibbles into the low half and the high
// nibbles into the high half.  An offset-binary source (q + 8) becomes two's
// complement by flipping bit 3 of every nibble.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// Four nibbles at bits 0, 8, 16, 24 of v -> bits 0, 4, 8, 12.
__device__ __forceinline__ uint32_t squeeze_nibbles(uint32_t v) {
  v = (v | (v >> 4)) & 0x00FF00FFu;
  return (v | (v >> 8)) & 0x0000FFFFu;
}

__device__ __forceinline__ uint32_t seq_to_pair(uint32_t w, uint32_t flip) {
  w ^= flip;
  return squeeze_nibbles(w & 0x0F0F0F0Fu) | (squeeze_nibbles((w >> 4) & 0x0F0F0F0Fu) << 16);
}

__global__ void __launch_bounds__(256) repack_int4_kernel(const uint4* __restrict__ src,
                                                          uint4* __restrict__ dst, size_t n_vec,
                                                          uint32_t flip) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n_vec;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 w = src[i];
    dst[i] = make_uint4(seq_to_pair(w.x, flip), seq_to_pair(w.y, flip), seq_to_pair(w.z, flip),
                        seq_to_pair(w.w, flip));
  }
}

__global__ void repack_int4_tail_kernel(const uint32_t* __restrict__ src, uint32_t* __restrict__ dst,
                                        size_t n, uint32_t flip) {
  const size_t i = threadIdx.x;
  if (i < n) dst[i] = seq_to_pair(src[i], flip);
}

cudaError_t launch_repack_int4(const uint32_t* src, uint32_t* dst, size_t n_words, bool offset8,
                               cudaStream_t st) {
  const uint32_t flip = offset8 ? 0x88888888u : 0u;
  const size_t n_vec = n_words / 4;
  if (n_vec > 0) {
    const size_t blocks = (n_vec + 255) / 256;
    const unsigned grid = static_cast<unsigned>(blocks < 152 * 16 ? blocks : 152 * 16);
    repack_int4_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const uint4*>(src),
                                             reinterpret_cast<uint4*>(dst), n_vec, flip);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const size_t tail = n_words - 4 * n_vec;
  if (tail > 0) {
    repack_int4_tail_kernel<<<1, 32, 0, st>>>(src + 4 * n_vec, dst + 4 * n_vec, tail, flip);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace moe
