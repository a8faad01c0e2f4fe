// norm.cu -- RMSNorm rows of the fp32 residual stream into bf16 GEMM inputs.
//
// "33. Removing overhead", section "Fewer, larger matmuls": add_norm does a layer's residual add and the
// next norm in one memory pass.  Here the residual add is already folded into the epilogue of the GEMM
// that produces it (o_proj, down), so this kernel reads the updated residual once and writes the normed
// bf16 row: y = h / sqrt(mean(h^2) + eps) * w.  In embed mode it first gathers h = E[id] (the embedding
// lookup of layer 0) and stores it as the residual.  With a row index it gathers rows (the final norm
// at each request's last token).  One CTA per row; the reduction order is fixed, so a row's result does
// not depend on how many rows the launch has.
#include "common.cuh"
#include "kernels.h"

namespace grd {

template <bool EMBED>
__global__ void __launch_bounds__(256) k_rmsnorm(NormParams p) {
  pdl_wait();
  const int row = blockIdx.x;
  const int H = p.H;
  __shared__ float red[8];
  extern __shared__ float hs[];  // the row, H floats
  float ss = 0.f;
  if (EMBED) {
    int id = p.ids[row];
    if (id < 0 || id >= p.V) id = 0;
    for (int c = threadIdx.x; c < H; c += blockDim.x) {
      const float v = __bfloat162float(p.embed[packed_offset(id, c, H)]);
      hs[c] = v;
      p.h_out[(size_t)row * H + c] = v;
    }
  } else {
    const int src = p.row_index ? p.row_index[row] : row;
    const float4* h4 = reinterpret_cast<const float4*>(p.h_in + (size_t)src * H);
    for (int c = threadIdx.x; c < H / 4; c += blockDim.x) reinterpret_cast<float4*>(hs)[c] = h4[c];
  }
  __syncthreads();
  // fixed-order partial sums: thread i adds elements i, i + 256, ...
  for (int c = threadIdx.x; c < H; c += blockDim.x) ss += hs[c] * hs[c];
  ss = warp_sum(ss);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
    red[0] = rsqrtf(t / (float)H + p.eps);
  }
  __syncthreads();
  const float rs = red[0];
  bf16* y = p.y + (size_t)row * H;
  for (int c = threadIdx.x * 2; c < H; c += blockDim.x * 2) {
    const float a = hs[c] * rs * p.w[c];
    const float b = hs[c + 1] * rs * p.w[c + 1];
    *reinterpret_cast<uint32_t*>(y + c) = pack_bf16x2(a, b);
  }
  pdl_trigger();
}

cudaError_t launch_rmsnorm(const NormParams& p, bool embed, const LaunchOpts& o, cudaStream_t s) {
  if (p.rows <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.rows);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = (size_t)p.H * sizeof(float);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = o.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (embed) return cudaLaunchKernelEx(&cfg, k_rmsnorm<true>, p);
  return cudaLaunchKernelEx(&cfg, k_rmsnorm<false>, p);
}

}  // namespace grd
