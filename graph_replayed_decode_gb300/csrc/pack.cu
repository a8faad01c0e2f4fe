// pack.cu -- load-time weight re-layout ("33. Removing overhead", section "Fewer, larger matmuls":
// the fused matrices are built once, when the weights are loaded).
#include "common.cuh"
#include "kernels.h"

namespace grd {
ENG_ELEM_NS_BEGIN

// One thread per packed element: gathers the source value of packed position `o`.
__global__ void k_pack(const bf16* __restrict__ src, bf16* __restrict__ dst, int N, int K, int interleave_half) {
  const size_t total = (size_t)N * K;
  const int KT = K >> 5;
  for (size_t o = blockIdx.x * (size_t)blockDim.x + threadIdx.x; o < total; o += (size_t)gridDim.x * blockDim.x) {
    const size_t tile = o >> 9;
    const int within = (int)(o & 511);
    const int i = (int)(tile / KT), j = (int)(tile % KT);
    const int s = within >> 8, lane = (within >> 3) & 31, e = within & 7;
    const int g = lane >> 2, t = lane & 3;
    const int half = (e >> 1) & 1, hi8 = e >> 2, lo = e & 1;
    const int r = g + 8 * half;
    const int col = 32 * j + 16 * s + 2 * t + 8 * hi8 + lo;
    int row = 16 * i + r;
    if (interleave_half > 0) {
      // packed tile i = [A rows 8i..8i+7 ; B rows 8i..8i+7] of the logical [A; B] matrix
      row = (r < 8) ? (8 * i + r) : (interleave_half + 8 * i + (r - 8));
    }
    dst[o] = src[(size_t)row * K + col];
  }
}

cudaError_t launch_pack(const bf16* src, bf16* dst, int N, int K, int interleave_half, cudaStream_t s) {
  const size_t total = (size_t)N * K;
  const int threads = 256;
  size_t blocks = (total + threads - 1) / threads;
  if (blocks > 65535u * 16u) blocks = 65535u * 16u;
  k_pack<<<(unsigned)blocks, threads, 0, s>>>(src, dst, N, K, interleave_half);
  return cudaGetLastError();
}

__global__ void k_bf16_to_f32(const bf16* __restrict__ src, float* __restrict__ dst, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = elem_to_float(src[i]);
}

cudaError_t launch_bf16_to_f32(const bf16* src, float* dst, int64_t n, cudaStream_t s) {
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  k_bf16_to_f32<<<(unsigned)blocks, 256, 0, s>>>(src, dst, n);
  return cudaGetLastError();
}

ENG_ELEM_NS_END
}  // namespace grd
