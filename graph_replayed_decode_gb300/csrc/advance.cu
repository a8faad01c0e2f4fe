// advance.cu -- the "record, advance" half of a device-resident decode step.
//
// "19. Fast decode", section "Static shapes and a static cache" (the fast decoder's step): after sampling,
// the step stores the new token, copies it into the static input and advances the position in place, so
// that the next replay reads the next step's inputs from the same addresses with no host involvement.
// Here that is done for a whole decode batch: for every real row (sequence length > 0; padding rows are
// left alone) the sampled id is recorded into a step-major ring and becomes the row's next input token,
// and the position and sequence length grow by one; the Philox offset grows by one per step.  A row that
// would pass the last position the block tables can hold is not advanced and is flagged in the status word.
#include "common.cuh"
#include "kernels.h"

namespace grd {

__global__ void k_advance(AdvanceParams p) {
  pdl_wait();
  const int step = *p.step;
  for (int r = threadIdx.x; r < p.rows; r += blockDim.x) {
    const int s = p.seq[r];
    if (s <= 0) continue;
    int id = p.sampled[r];
    if (id < 0 || id >= p.vocab) {
      set_status(p.status, ST_NAN);
      id = 0;
    }
    if (step < p.ring_cap) p.ring[(size_t)step * p.rows + r] = id;
    if (p.prev_row) p.prev_row[r] = -1;  // the next step's input is set here, not gathered
    if (s >= p.max_pos) {
      set_status(p.status, ST_BAD_POSITION);
      continue;
    }
    p.ids[r] = id;
    p.pos[r] = s;
    p.seq[r] = s + 1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    *p.step = step + 1;
    const unsigned long long off = ((unsigned long long)p.rng[3] << 32 | p.rng[2]) + 1ull;
    p.rng[2] = (uint32_t)off;
    p.rng[3] = (uint32_t)(off >> 32);
  }
}

cudaError_t launch_advance(const AdvanceParams& p, const LaunchOpts& o, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = o.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_advance, p);
}

}  // namespace grd

namespace grd {

// Holds the stream for `ns` nanoseconds of device time (bounded by the global timer): put in front of an
// eagerly enqueued step that is timed launch by launch, it lets the host enqueue every launch before the
// first one runs, so that each event pair brackets device work only, not host launch latency.
__global__ void k_hold(unsigned long long ns) {
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  do {
    __nanosleep(1000);
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  } while (t - t0 < ns);
}

cudaError_t launch_hold(unsigned long long ns, cudaStream_t s) {
  k_hold<<<1, 1, 0, s>>>(ns);
  return cudaGetLastError();
}

}  // namespace grd
