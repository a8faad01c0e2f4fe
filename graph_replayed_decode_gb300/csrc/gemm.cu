// gemm.cu -- skinny GEMM Y[T][N] = X[T][K] . W[N][K]^T for the decode-sized projections, with the
// step's elementwise work fused into its epilogue.
//
// Shapes: T is the packed token count of the step (1..64 in decode, larger in prefill, handled in
// 64-token chunks), N the output width, K the reduction width.  "33. Removing overhead", section "Fewer,
// larger matmuls": Q/K/V and gate/up are each one matmul over a concatenated matrix; the same section
// lists fusing SiLU-and-mul, RoPE, and the LM head with sampling into the producing kernels.
//
// Design (HBM-bound at decode sizes):
//   * W is pre-packed in m16n8k16 fragment order (common.cuh), so each lane streams its A fragments
//     with 16-byte loads straight from HBM -- every byte of W is read exactly once per chunk;
//   * X is staged through shared memory in 512-column pieces and read with ldmatrix;
//   * a CTA owns RG 16-row tiles and one of S K-ranges; its 8 warps split the K-range, reduce through
//     shared memory in a fixed order, and when S > 1 the last CTA of a row group (atomic ticket, no
//     waiting) adds the S partials in split order -- so results are deterministic and do not depend
//     on T, which makes graph replay and eager execution bit-identical;
//   * epilogues: fp32 store (+bias), residual add into the fp32 stream, SiLU(gate)*up on row-interleaved
//     gate|up tiles, and the LM head: logits (optional) plus a per-token running (key, index) maximum
//     for greedy / Gumbel-max sampling, finished by the last CTA.
#include "common.cuh"
#include "kernels.h"
#include "sampling.cuh"

namespace grd {

static constexpr int kPieceTiles = 16;  // k-tiles (x32 columns) of X staged per piece

template <int NT, int EPI>
__global__ void __launch_bounds__(256) k_gemm(GemmParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int rgi = blockIdx.x, split = blockIdx.y, chunk = blockIdx.z;
  const int nRG = gridDim.x;
  const int n0 = chunk * 64;
  const int KT = p.K >> 5;
  const int ktn = p.kt_per_split;
  const int kt0 = split * ktn;
  const int RG = p.RG, KG = 8 / RG;
  const int rt = warp % RG, kg = warp / RG;
  const int row_tile = rgi * RG + rt;

  pdl_wait();

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

  bf16* xs = reinterpret_cast<bf16*>(smem);
  const uint4* wp = reinterpret_cast<const uint4*>(p.W) + ((size_t)row_tile * KT + kt0) * 64 + lane;

  for (int pc = 0; pc < ktn; pc += kPieceTiles) {
    const int pn = min(kPieceTiles, ktn - pc);
    const int xstride = pn * 32 + 8;
    const int cpr = pn * 4;  // 16-byte chunks per staged row
    if (pc > 0) __syncthreads();
    for (int i = threadIdx.x; i < NT * 8 * cpr; i += 256) {
      const int r = i / cpr, c = i - r * cpr;
      const int tok = n0 + r;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (tok < p.T)
        v = *reinterpret_cast<const uint4*>(p.X + (size_t)tok * p.ldx + (size_t)(kt0 + pc) * 32 + c * 8);
      *reinterpret_cast<uint4*>(xs + r * xstride + c * 8) = v;
    }
    __syncthreads();

    constexpr int U = 4;
    for (int base = kg; base < pn; base += KG * U) {
      uint4 a[U][2];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int kt = base + u * KG;
        if (kt < pn) {
          a[u][0] = ld_stream16(wp + (size_t)(pc + kt) * 64);
          a[u][1] = ld_stream16(wp + (size_t)(pc + kt) * 64 + 32);
        } else {
          a[u][0] = a[u][1] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int kt = base + u * KG;
        if (kt < pn) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            uint32_t b[4];
            const int m = lane >> 3;
            const bf16* addr = xs + (nt * 8 + (lane & 7)) * xstride + kt * 32 + (m >> 1) * 16 + (m & 1) * 8;
            ldmatrix_x4(b, addr);
            mma_bf16(acc[nt], a[u][0].x, a[u][0].y, a[u][0].z, a[u][0].w, b[0], b[1]);
            mma_bf16(acc[nt], a[u][1].x, a[u][1].y, a[u][1].z, a[u][1].w, b[2], b[3]);
          }
        }
      }
    }
  }
  pdl_trigger();

  // ---- reduce the KG warps of each row tile, in warp order
  __syncthreads();
  float4* red = reinterpret_cast<float4*>(smem);
  if (KG > 1) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      red[(warp * NT + nt) * 32 + lane] = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
    __syncthreads();
    if (kg == 0) {
      for (int j = 1; j < KG; ++j) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float4 v = red[((j * RG + rt) * NT + nt) * 32 + lane];
          acc[nt][0] += v.x;
          acc[nt][1] += v.y;
          acc[nt][2] += v.z;
          acc[nt][3] += v.w;
        }
      }
    }
  }

  // ---- split-K: the last CTA of the row group adds the S partials in split order
  __shared__ int s_flag;
  bool finalize = true;
  if (p.S > 1) {
    const size_t group = (size_t)chunk * nRG + rgi;
    if (kg == 0) {
      float4* dst = reinterpret_cast<float4*>(p.ws) + ((group * p.S + split) * RG + rt) * NT * 32 + lane;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) __stcg(dst + nt * 32, make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]));
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const int old = atomicAdd(p.tickets + group, 1);
      s_flag = (old == p.S - 1);
      if (s_flag) p.tickets[group] = 0;
    }
    __syncthreads();
    finalize = s_flag != 0;
    if (finalize) {
      __threadfence();
      if (kg == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        for (int sp = 0; sp < p.S; ++sp) {
          const float4* src = reinterpret_cast<const float4*>(p.ws) + ((group * p.S + sp) * RG + rt) * NT * 32 + lane;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float4 v = __ldcg(src + nt * 32);
            acc[nt][0] += v.x;
            acc[nt][1] += v.y;
            acc[nt][2] += v.z;
            acc[nt][3] += v.w;
          }
        }
      }
    }
  }

  // ---- epilogue
  if (finalize && kg == 0) {
    const int row0 = row_tile * 16 + g;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int tok0 = n0 + nt * 8 + 2 * t;
      if (EPI == EPI_STORE_F32) {
        const float b0 = p.bias ? p.bias[row0] : 0.f;
        const float b8 = p.bias ? p.bias[row0 + 8] : 0.f;
        if (tok0 < p.T) {
          p.out_f32[(size_t)tok0 * p.ldo + row0] = acc[nt][0] + b0;
          p.out_f32[(size_t)tok0 * p.ldo + row0 + 8] = acc[nt][2] + b8;
        }
        if (tok0 + 1 < p.T) {
          p.out_f32[(size_t)(tok0 + 1) * p.ldo + row0] = acc[nt][1] + b0;
          p.out_f32[(size_t)(tok0 + 1) * p.ldo + row0 + 8] = acc[nt][3] + b8;
        }
      } else if (EPI == EPI_RESID) {
        if (tok0 < p.T) {
          p.resid[(size_t)tok0 * p.N + row0] += acc[nt][0];
          p.resid[(size_t)tok0 * p.N + row0 + 8] += acc[nt][2];
        }
        if (tok0 + 1 < p.T) {
          p.resid[(size_t)(tok0 + 1) * p.N + row0] += acc[nt][1];
          p.resid[(size_t)(tok0 + 1) * p.N + row0 + 8] += acc[nt][3];
        }
      } else if (EPI == EPI_SILU) {
        const int j = row_tile * 8 + g;  // gate row j sits at tile row g, up row j at tile row g + 8
        const int I = p.N >> 1;
        if (tok0 < p.T) {
          const float ga = acc[nt][0], up = acc[nt][2];
          p.out_bf16[(size_t)tok0 * I + j] = __float2bfloat16_rn(ga / (1.f + expf(-ga)) * up);
        }
        if (tok0 + 1 < p.T) {
          const float ga = acc[nt][1], up = acc[nt][3];
          p.out_bf16[(size_t)(tok0 + 1) * I + j] = __float2bfloat16_rn(ga / (1.f + expf(-ga)) * up);
        }
      } else if (EPI == EPI_LMHEAD) {
        const bool wl = *p.write_logits != 0;
        unsigned long long best0 = 0ull, best1 = 0ull;
        uint32_t rng[4] = {p.rng[0], p.rng[1], p.rng[2], p.rng[3]};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int tok = tok0 + c;
          if (tok < p.T) {
            const float it = p.inv_temp[tok];
            unsigned long long bb = 0ull;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int v = row0 + 8 * h;
              const float z = acc[nt][2 * h + c];
              if (wl) p.logits[(size_t)tok * p.N + v] = z;
              const float key = sample_key(z, it, rng, (uint32_t)tok, (uint32_t)v);
              if (key != key) {
                set_status(p.status, ST_NAN);
              } else {
                const unsigned long long pk = pack_key_index(key, (uint32_t)v);
                bb = pk > bb ? pk : bb;
              }
            }
            if (c == 0) best0 = bb; else best1 = bb;
          }
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          const unsigned long long x0 = __shfl_xor_sync(0xffffffffu, best0, o);
          const unsigned long long x1 = __shfl_xor_sync(0xffffffffu, best1, o);
          best0 = x0 > best0 ? x0 : best0;
          best1 = x1 > best1 ? x1 : best1;
        }
        if (g == 0) {
          if (tok0 < p.T && best0) atomicMax(p.best + tok0, best0);
          if (tok0 + 1 < p.T && best1) atomicMax(p.best + tok0 + 1, best1);
        }
      }
    }
  }

  if (EPI == EPI_LMHEAD) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const int total = gridDim.x * gridDim.y * gridDim.z;
      const int old = atomicAdd(p.done_counter, 1);
      s_flag = (old == total - 1);
    }
    __syncthreads();
    if (s_flag) {
      __threadfence();
      for (int r = threadIdx.x; r < p.T; r += blockDim.x) {
        const unsigned long long b = atomicExch(p.best + r, 0ull);
        p.out_ids[r] = (int)unpack_index(b);
      }
      if (threadIdx.x == 0) *p.done_counter = 0;
    }
  }
}

// ------------------------------------------------------------------ host side

void gemm_plan(int N, int K, int* RG, int* S, int* kt_per_split) {
  const int tiles = N / 16, KT = K / 32;
  const int target = 2 * 152;
  int s = 1, rg = 1;
  if (tiles >= target) {
    for (int c = 8; c >= 1; c >>= 1)
      if (tiles % c == 0 && tiles / c >= target) {
        rg = c;
        break;
      }
  } else {
    const int want = (target + tiles - 1) / tiles;
    s = KT;
    for (int c = want; c <= KT; ++c)
      if (KT % c == 0) {
        s = c;
        break;
      }
  }
  *RG = rg;
  *S = s;
  *kt_per_split = KT / s;
}

static int chunks_of(int T) { return (T + 63) / 64; }

size_t gemm_ws_floats(int N, int K, int T) {
  int rg, s, ktn;
  gemm_plan(N, K, &rg, &s, &ktn);
  if (s == 1) return 0;
  return (size_t)chunks_of(T) * (N / 16) * s * 8 * 128;  // NT <= 8 n-tiles of 128 floats per 16-row tile
}

int gemm_tickets(int N, int K, int T) {
  int rg, s, ktn;
  gemm_plan(N, K, &rg, &s, &ktn);
  return chunks_of(T) * (N / 16 / rg);
}

template <int NT, int EPI>
static cudaError_t launch_nt(const GemmParams& p, const LaunchOpts& o, cudaStream_t s, dim3 grid) {
  const int pn = p.kt_per_split < kPieceTiles ? p.kt_per_split : kPieceTiles;
  const size_t xs = (size_t)NT * 8 * (pn * 32 + 8) * 2;
  const size_t red = (size_t)8 * NT * 32 * 16;
  const size_t smem = xs > red ? xs : red;
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(k_gemm<NT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = o.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_gemm<NT, EPI>, p);
}

template <int EPI>
static cudaError_t launch_epi(const GemmParams& p, const LaunchOpts& o, cudaStream_t s) {
  const int nRG = p.N / 16 / p.RG;
  const int chunks = chunks_of(p.T);
  const dim3 grid(nRG, p.S, chunks);
  const int ntiles = p.T >= 64 ? 8 : (p.T + 7) / 8;
  if (ntiles <= 1) return launch_nt<1, EPI>(p, o, s, grid);
  if (ntiles <= 2) return launch_nt<2, EPI>(p, o, s, grid);
  if (ntiles <= 4) return launch_nt<4, EPI>(p, o, s, grid);
  return launch_nt<8, EPI>(p, o, s, grid);
}

cudaError_t launch_gemm(const GemmParams& p, int epi, const LaunchOpts& o, cudaStream_t s) {
  if (p.T <= 0) return cudaSuccess;
  switch (epi) {
    case EPI_STORE_F32: return launch_epi<EPI_STORE_F32>(p, o, s);
    case EPI_RESID: return launch_epi<EPI_RESID>(p, o, s);
    case EPI_SILU: return launch_epi<EPI_SILU>(p, o, s);
    case EPI_LMHEAD: return launch_epi<EPI_LMHEAD>(p, o, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace grd
