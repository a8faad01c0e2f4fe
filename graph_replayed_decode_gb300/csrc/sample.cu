// sample.cu -- standalone launches of the sampler arithmetic of sampling.cuh: the Philox uniforms, the
// Gumbel transform and the greedy / Gumbel-max argmax over caller-provided logits.  The fused LM-head
// epilogue (gemm.cu) uses the same device functions, so these launches let tests compare the GPU's
// noise and log bit for bit with a CPU restatement.
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "sampling.cuh"

namespace grd {

__global__ void k_philox_uniforms(uint32_t s0, uint32_t s1, uint32_t o0, uint32_t o1, int rows, int vocab,
                                  float* out) {
  const int64_t n = (int64_t)rows * vocab;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / vocab), v = (int)(i % vocab);
    out[i] = philox_uniform(s0, s1, o0, o1, (uint32_t)r, (uint32_t)v);
  }
}

cudaError_t launch_philox_uniforms(uint64_t seed, uint64_t offset, int rows, int vocab, float* out, cudaStream_t s) {
  const int64_t n = (int64_t)rows * vocab;
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 8192) blocks = 8192;
  k_philox_uniforms<<<(unsigned)blocks, 256, 0, s>>>((uint32_t)seed, (uint32_t)(seed >> 32), (uint32_t)offset,
                                                      (uint32_t)(offset >> 32), rows, vocab, out);
  return cudaGetLastError();
}

__global__ void k_gumbel(const float* u, float* g, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    g[i] = gumbel_from_uniform(u[i]);
}

cudaError_t launch_gumbel(const float* u, float* g, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 8192) blocks = 8192;
  k_gumbel<<<(unsigned)blocks, 256, 0, s>>>(u, g, n);
  return cudaGetLastError();
}

// One CTA per row: every thread scans a strided share of the vocabulary, then a fixed reduction tree.
__global__ void __launch_bounds__(256) k_sample(const float* logits, int vocab, const float* inv_temp,
                                                const uint32_t* rng_dev, int* out_ids, int* status) {
  const int r = blockIdx.x;
  const float it = inv_temp[r];
  uint32_t rng[4] = {rng_dev[0], rng_dev[1], rng_dev[2], rng_dev[3]};
  unsigned long long best = 0ull;
  const float* z = logits + (size_t)r * vocab;
  for (int v = threadIdx.x; v < vocab; v += blockDim.x) {
    const float key = sample_key(z[v], it, rng, (uint32_t)r, (uint32_t)v);
    if (key != key) {
      set_status(status, ST_NAN);
      continue;
    }
    const unsigned long long pk = pack_key_index(key, (uint32_t)v);
    best = pk > best ? pk : best;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long x = __shfl_xor_sync(0xffffffffu, best, o);
    best = x > best ? x : best;
  }
  __shared__ unsigned long long wb[8];
  if ((threadIdx.x & 31) == 0) wb[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long b = 0ull;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) b = wb[w] > b ? wb[w] : b;
    out_ids[r] = (int)unpack_index(b);
  }
}

cudaError_t launch_sample(const float* logits, int rows, int vocab, const float* inv_temp, const uint32_t* rng,
                          unsigned long long* /*best*/, int* out_ids, int* status, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  k_sample<<<rows, 256, 0, s>>>(logits, vocab, inv_temp, rng, out_ids, status);
  return cudaGetLastError();
}

}  // namespace grd

// ------------------------------------------------------------------ sampler without any allocation
//
// eng_sample copies each call's inverse temperatures and Philox words into a small device block it
// allocates.  The variant below keeps that block in a fixed array linked into this library instead, for
// callers that are not allowed to allocate device memory.  Every GPU that loads the library holds the
// array (kNoAllocMaxRows + 4 words) until the process exits, and every call on that GPU shares it.
// The words reach the array as the parameters of a one-CTA staging kernel (launch parameters are copied
// when the launch is enqueued), so the call never reads host memory after it returns.

namespace grd {

static constexpr int kMaxDevices = 64;
static __device__ __align__(256) uint32_t g_sample_scratch[kNoAllocMaxRows + 4];

struct NoAllocWords {
  uint32_t n;                          // words in use: rows + 4
  uint32_t w[kNoAllocMaxRows + 4];     // inverse temperatures (float bits), then seed_lo, seed_hi, offset_lo, offset_hi
};
static_assert(sizeof(NoAllocWords) < 32000, "kernel parameters are limited to 32 KB");

__global__ void __launch_bounds__(256) k_noalloc_stage(const __grid_constant__ NoAllocWords p, uint32_t* dst) {
  for (uint32_t i = threadIdx.x; i < p.n; i += blockDim.x) dst[i] = p.w[i];
}

// Device address of g_sample_scratch for the current device, looked up once per device.  In host code the
// array's name is only a host-side handle, so the address must come from cudaGetSymbolAddress.  The cached
// address belongs to the device's current context: after cudaDeviceReset it is no longer valid.
cudaError_t noalloc_scratch(uint32_t** out) {
  static std::mutex mu;
  static uint32_t* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t r = cudaGetDevice(&dev);
  if (r != cudaSuccess) return r;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    r = cudaGetSymbolAddress(&p, g_sample_scratch);
    if (r != cudaSuccess) return r;
    addr[dev] = static_cast<uint32_t*>(p);
  }
  *out = addr[dev];
  return cudaSuccess;
}

cudaError_t launch_sample_noalloc(const float* logits, int rows, int vocab, const float* inv_temp_host,
                                  const uint32_t rng_host[4], uint32_t* scratch, int* out_ids, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (rows > kNoAllocMaxRows || !scratch) return cudaErrorInvalidValue;
  NoAllocWords w;
  w.n = (uint32_t)rows + 4;
  memcpy(w.w, inv_temp_host, (size_t)rows * 4);
  for (int i = 0; i < 4; ++i) w.w[rows + i] = rng_host[i];
  k_noalloc_stage<<<1, 256, 0, s>>>(w, scratch);
  cudaError_t r = cudaGetLastError();
  if (r != cudaSuccess) return r;
  return launch_sample(logits, rows, vocab, reinterpret_cast<const float*>(scratch), scratch + rows, nullptr, out_ids,
                       nullptr, s);
}

}  // namespace grd
