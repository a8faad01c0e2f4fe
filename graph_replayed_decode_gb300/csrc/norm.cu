// norm.cu -- embedding gather of layer 0 into the fp32 residual stream.
//
// h[t] = E[id[t]] (the embedding is stored packed; packed_offset finds each element; id[t] optionally
// gathered from the previous step's sampled ids), the row's sum of
// squares, and the first QKV GEMM's operand planes of h * w_in, which that GEMM turns into its input
// RMSNorm by scaling with 1 / rms(h) ("33. Removing overhead", section "Fewer, larger matmuls": add_norm
// does a residual update and the next norm in one pass; here every norm is folded into the GEMM that
// consumes it).  One CTA per token, fixed reduction order.
#include "common.cuh"
#include "kernels.h"

namespace grd {
ENG_ELEM_NS_BEGIN

__global__ void __launch_bounds__(256) k_embed(EmbedParams p) {
  // The first kernel of a step waits for the previous step to finish (its last kernel updates the step
  // inputs in place) before letting the step's later kernels launch: those read the step inputs before
  // their own wait.
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x;
  const int H = p.H;
  __shared__ float red[8];
  int id = p.ids[row];
  // async scheduling: a token whose id the host did not know yet takes the id the previous step sampled
  // for the given request row ("33. Removing overhead", section on async scheduling)
  const int src = p.prev_row ? p.prev_row[row] : -1;
  if (src >= 0) id = src < p.prev_rows ? p.prev_ids[src] : -1;
  if (id < 0 || id >= p.V) {
    set_status(p.status, ST_NAN);
    id = 0;
  }
  float ss = 0.f;
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    const float v = elem_to_float(p.embed[packed_offset(id, c, H)]);
    p.h_out[(size_t)row * H + c] = v;
    put_split(p.xh_out, p.xl_out, (size_t)row * H + c, v * p.norm_w[c]);
    ss += v * v;
  }
  ss = warp_sum(ss);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
    p.sq_out[(size_t)row * p.sq_stride] = tot;
  }
}

cudaError_t launch_embed(const EmbedParams& p, const LaunchOpts& o, cudaStream_t s) {
  if (p.rows <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.rows);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = o.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_embed, p);
}

ENG_ELEM_NS_END
}  // namespace grd
