// kernels.h -- internal launch interface between the engine (engine.cu) and the kernels.
// Every launcher enqueues on `stream`, returns the launch's cudaError_t and never synchronises.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cuda_bf16.h>

namespace grd {

typedef __nv_bfloat16 bf16;

// SM count of the current device (looked up once per device; 0 when it cannot be read).
int device_sm_count();
// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current device, once per (device, kernel):
// the attribute belongs to the device's context, so each GPU a process uses gets its own call.
cudaError_t ensure_smem_limit(const void* kernel, int bytes);

// Launch options shared by all launchers: programmatic dependent launch on/off.
struct LaunchOpts {
  bool pdl = false;
};

// ------------------------------------------------------------------ weight packing (pack.cu)
// dst (packed, see common.cuh) <- src row-major bf16 [N][K].  interleave_half: when > 0, the logical
// rows are the concatenation [A (interleave_half rows); B (interleave_half rows)] and packed row tile i
// holds A rows 8i..8i+7 then B rows 8i..8i+7 (gate|up for the fused SiLU epilogue).
cudaError_t launch_pack(const bf16* src, bf16* dst, int N, int K, int interleave_half, cudaStream_t s);
cudaError_t launch_bf16_to_f32(const bf16* src, float* dst, int64_t n, cudaStream_t s);

// ------------------------------------------------------------------ embedding gather (norm.cu)
struct EmbedParams {
  const bf16* embed;     // packed embedding [V][H]
  const int* ids;        // token ids [rows]
  float* h_out;          // residual rows [rows][H]
  float* sq_out;         // sum of squares of each row -> sq_out[row * sq_stride]
  int sq_stride;
  const float* norm_w;   // the first layer's input-norm weight [H]
  const int* prev_row;   // [rows]: -1, or the previous step's request row whose sampled id is this token's
  const int* prev_ids;   // the previous step's sampled ids [previous num_reqs]
  int prev_rows;         // capacity of prev_ids (the host checks gathers against the previous step's rows)
  bf16* xh_out;          // operand planes of h * norm_w [rows][H] (see GemmParams)
  bf16* xl_out;
  int rows, H, V;
  int* status;
};
cudaError_t launch_embed(const EmbedParams& p, const LaunchOpts& o, cudaStream_t s);

// ------------------------------------------------------------------ skinny GEMM (gemm.cu)
enum GemmEpi { EPI_STORE_F32 = 0, EPI_RESID = 1, EPI_SILU = 2, EPI_LMHEAD = 3, EPI_QKV_ROPE = 4 };

struct GemmParams {
  const bf16* W;   // packed [N][K]
  // Activation operand: two bf16 planes [rows][ldx], hi = bf16(x) and lo = bf16(x - hi), written by the
  // producing kernel; row x_rows[t] (or t) is token t's.  With a norm (NORM_IN) the planes hold h * norm_w
  // and the kernel scales token t's outputs by 1 / rms(h_t), from the producer's partial sums of squares.
  const bf16* Xh;
  const bf16* Xl;
  const int* x_rows;
  int ldx;
  int T, N, K;
  int RG;           // 16-row tiles per CTA (1, 2, 4, 8)
  int S;            // k splits
  int kt_per_split; // 32-column k tiles per split (the S split CTAs of a row group form a cluster)
  const void* pf_ptr;           // weights of a later kernel to prefetch into L2 (pf_bytes, multiple of 16)
  unsigned long long pf_bytes;
  // norm: 1 / rms of token t from its sq_parts partial sums of squares sq_in[x_rows[t] * sq_stride + j]
  const float* sq_in;
  int sq_parts;
  int sq_stride;
  float eps;
  // epilogues
  float* out_f32;   // EPI_STORE_F32: out[t][n] (+ bias[n]), row stride ldo
  int ldo;
  const float* bias;
  float* resid;     // EPI_RESID: resid[t][n] += v (row stride N); sq_out[t * sq_stride + row group] = sum h^2
  float* sq_out;
  const float* next_norm_w;  //         and the next GEMM's operand planes of h * next_norm_w
  bf16* xh_out;     // EPI_RESID, EPI_SILU: operand planes written for the next GEMM (row stride N, or N / 2)
  bf16* xl_out;     // EPI_SILU: silu(gate_j) * up_j
  // EPI_QKV_ROPE: CTA rows are whole heads of the fused [q | k | v] projection
  const int* positions;
  const int* tok2req;
  const int* seq_lens;
  const int* bt;
  int mbs;
  const float* q_norm;
  const float* k_norm;
  const float* cos_sin;   // [max_pos][d/2][2]
  int max_pos;
  float* q_out;           // [T][Hq][d]
  bf16* k_pool;           // this layer's K plane [NB+1][Hkv][16][d]
  bf16* v_pool;
  int* slots;             // [T]
  int Hq, Hkv, d, NB;
  // EPI_LMHEAD: logits and sampling
  float* logits;                // [T][N] when *write_logits != 0
  const int* write_logits;      // device flag
  float* keys_out;              // or null: [T][N] sampling keys (logit / T + Gumbel noise), when *write_keys
  const int* write_keys;        // device flag (with keys_out)
  unsigned int* row_ext;        // or null: [T][2] order-preserving bits of the row's largest finite logit
                                //   and their complement for the smallest (atomicMax), with the logits
  const float* inv_temp;        // [T]; 0 = greedy
  const uint32_t* rng;          // device [4]: seed_lo, seed_hi, offset_lo, offset_hi
  unsigned long long* best;     // [T] packed (key, ~index), zero between launches
  int* done_counter;            // counts finished CTAs, zero between launches
  int* out_ids;                 // [T]
  int* status;
};
// Tensor maps of the tensor-core (tcgen05) GEMM path: the weight as a row-major [N][K] bf16 matrix in
// 128 x 64 boxes, and the activation planes [rows][K] in 64 x 64 boxes, all with 128-byte swizzle.
struct TcMaps {
  CUtensorMap w, xh, xl;
};
// Encodes a 2D bf16 tensor map over a row-major [rows][cols] matrix with boxes of box_rows x 64 columns
// (128-byte swizzle; rows past the end read as zeros).  False when the driver refuses it.
bool make_tc_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);
// True when a tensor-core launch with S K-splits fits the shared-memory budget (its split-K receive buffer
// grows with S).
bool tc_split_fits(int S);
// True when a warp-MMA plan's weight slice (RG row tiles x kt_per_split k-tiles) is small enough to be
// bulk-copied into shared memory before the kernel waits; larger slices stream through registers.
bool gemm_slice_fits(int RG, int ktn);
// Token classes of the tensor-core path (when a projection's shape allows it): from kTcTokens tokens when
// the warp-MMA large plan's weight slice is too large to stage (with K splits), and always from
// kTcPrefillTokens (prefill chunks, no K split).  The boundaries coincide with the plan classes, so an
// eager step and its padded bucket take the same path.
static constexpr int kTcTokens = 9;
static constexpr int kTcPrefillTokens = 65;

// Picks RG / S / kt_per_split for an [N][K] weight (independent of T, so every token count computes
// each output with the same summation order).  rg_fixed > 0 forces the rows per CTA (whole heads); sms is
// the device's SM count (one wave of CTAs).
void gemm_plan(int N, int K, int rg_fixed, int sms, int* RG, int* S, int* kt_per_split);
// The plan for steps of more than 8 tokens (activation bytes per CTA weigh in; see gemm.cu).
void gemm_plan_large(int N, int K, int rg_fixed, int sms, int* RG, int* S, int* kt_per_split);
// Token count from which a step uses the large plans.
static constexpr int kLargePlanTokens = 9;
// tc: the tensor maps of the tcgen05 path (then RG must be 8, S 1, no x_rows; N % 128 == 0, K % 64 == 0),
// or null for the warp-MMA path.
cudaError_t launch_gemm(const GemmParams& p, int epi, bool norm_in, const LaunchOpts& o, cudaStream_t s,
                        const TcMaps* tc = nullptr);

// ------------------------------------------------------------------ attention (attn_decode.cu, attn_prefill.cu)
// Key splits of one (row, KV head) in decode attention (the block-table width divided into at most this many).
constexpr int kAttnMaxSplits = 8;
struct AttnDecodeParams {
  const float* q;         // [T][Hq][d]
  const bf16* k_pool;     // layer K plane
  const bf16* v_pool;     // layer V plane
  const int* bt;          // [R][mbs]
  int mbs;
  const int* seq_lens;    // [R]
  const int* cu;          // [R+1]: request r's query token is cu[r]
  int r0;                 // first request handled (grid.x = rows)
  int rows;
  bf16* out_h;            // operand planes of the output [T][Hq * d] (hi, lo) for the output projection
  bf16* out_l;
  int Hq, Hkv, d, NB;
  int split_blocks;       // KV blocks per split
  int max_splits;         // splits of the grid (<= kAttnMaxSplits)
  float* ws;              // partials [slots][G][d + 2]: rows * Hkv + 4 * flat_ctas pieces of the flat
                          //   partition, or rows * Hkv * max_splits splits
  int* counters;          // [rows][Hkv] finished pieces, zero between launches
  int flat_ctas;          // grid of the flat partition (more than 4 rows, G <= 2): CTAs resident at once
  float scale_log2;       // log2(e) / sqrt(d)
  const void* pf_ptr;     // weights of a later kernel to prefetch into L2
  unsigned long long pf_bytes;
  int* status;
};
cudaError_t launch_attn_decode(const AttnDecodeParams& p, const LaunchOpts& o, cudaStream_t s);
// CTAs of the flat-partition kernel that are resident at once on a device of `sms` SMs, for launches of up
// to `rows` rows (0 if the occupancy query fails).
int attn_flat_ctas(int d, int rows, int sms);

struct AttnPrefillParams {
  const float* q;         // [T][Hq][d]
  const bf16* k_pool;
  const bf16* v_pool;
  const int* bt;
  int mbs;
  const int* positions;   // [T]
  const int4* items;      // work items: (request, first token, token count <= 64, unused)
  int n_items;
  bf16* out_h;            // operand planes of the output [T][Hq * d]
  bf16* out_l;
  int Hq, Hkv, d, NB;
  float scale_log2;
  int* status;
};
cudaError_t launch_attn_prefill(const AttnPrefillParams& p, const LaunchOpts& o, cudaStream_t s);

// ------------------------------------------------------------------ decode advance (advance.cu)
struct AdvanceParams {
  const int* sampled;  // [rows] ids sampled by this step
  int* ids;            // static inputs, advanced in place
  int* prev_row;       // the token-to-previous-row map of the step inputs: reset to -1 for advanced rows
  int* pos;
  int* seq;
  uint32_t* rng;       // [4]: seed_lo, seed_hi, offset_lo, offset_hi (offset += 1)
  int* step;           // ring write index
  int* ring;           // [ring_cap][rows]
  int ring_cap, rows, vocab, max_pos;
  int* status;
};
cudaError_t launch_advance(const AdvanceParams& p, const LaunchOpts& o, cudaStream_t s);
// One thread sleeping on the global timer for `ns` nanoseconds (front of a launch-by-launch timed step).
cudaError_t launch_hold(unsigned long long ns, cudaStream_t s);

// ------------------------------------------------------------------ sampler pieces (sample.cu)
cudaError_t launch_philox_uniforms(uint64_t seed, uint64_t offset, int rows, int vocab, float* out, cudaStream_t s);
cudaError_t launch_gumbel(const float* u, float* g, int64_t n, cudaStream_t s);
cudaError_t launch_sample(const float* logits, int rows, int vocab, const float* inv_temp, const uint32_t* rng,
                          unsigned long long* best, int* out_ids, int* status, cudaStream_t s);
// Top-k / top-p filtered draw (sample_filter.cu): one CTA per row over float32 logits [rows][vocab].
struct FilterParams {
  const float* logits;
  int vocab;
  const float* inv_temp;  // [rows]; 0 = greedy
  const int* top_k;       // [rows] or null; <= 0 or >= vocab: off
  const int* p_units;     // [rows] or null; top-p in units of 2^-24, 0 (or >= 2^24): off
  const uint32_t* rng;    // seed_lo, seed_hi, offset_lo, offset_hi
  int* out_ids;           // [rows]
  int* out_kept;          // [rows] survivor counts, or null
  int* status;            // or null
  int only_filtered;      // 1: rows with no filter (or temperature 0) are left untouched
  const float* keys;      // or null: the rows' sampling keys, already formed when *keys_valid (else computed)
  const int* keys_valid;  // device flag (with keys)
  unsigned int* row_ext;  // or null: the rows' logit extremes, already formed (else found here); reset to 0
                          //   by this kernel for every row it is launched over
};
cudaError_t launch_sample_filtered(const FilterParams& p, int rows, cudaStream_t s);
// Top-k candidates up to this many are sorted in shared memory and drawn from there (no key needed from the
// producer of the logits); rows past it (and top-p without top-k) draw over a pass of the whole row.
constexpr int kFilterGatherCap = 8192;
cudaError_t launch_exp_rn(const float* d, float* out, int64_t n, cudaStream_t s);
// eng_sample_noalloc: the sampler with its per-call words (the rows' inverse temperatures, then seed_lo,
// seed_hi, offset_lo, offset_hi) in a fixed device array of this library (sample.cu) instead of an
// allocation.  The words reach the array as the parameters of a staging kernel, so the call reads no host
// memory after it returns.  At most kNoAllocMaxRows rows: 16 KiB of inverse temperatures.
constexpr int kNoAllocMaxRows = 4096;
static_assert(kNoAllocMaxRows * sizeof(float) == 16 * 1024, "the array holds 16 KiB of inverse temperatures");
// Device address of the array on the current device (looked up once per device, with that device current).
cudaError_t noalloc_scratch(uint32_t** out);
// Stages inv_temp[rows] and rng[4] into the array at `scratch`, then runs the sampler over the logits.
cudaError_t launch_sample_noalloc(const float* logits, int rows, int vocab, const float* inv_temp_host,
                                  const uint32_t rng_host[4], uint32_t* scratch, int* out_ids, cudaStream_t s);


// moe.cu: a mixture-of-experts MLP with shapes that do not depend on the routing (router, alignment of the
// assignments by expert into blocks of 16 rows, grouped gate|up and down GEMMs, combine).
int moe_padded_rows(int total, int E, int bm);
size_t moe_workspace_bytes(int N, int k, int E, int D, int I);
cudaError_t launch_moe_route(const bf16* x, const bf16* wr, int N, int D, int E, int k, float* w, int* ids,
                             cudaStream_t s);
cudaError_t launch_moe_align(const int* ids, int total, int E, int bm, int* sorted_ids, int* block_expert, int* out,
                             cudaStream_t s);
cudaError_t launch_moe_mlp(const bf16* x, const bf16* gate_up, const bf16* down, const float* rw, const int* ids,
                           int N, int D, int I, int E, int k, float* out, void* ws, size_t ws_bytes, cudaStream_t s);

// ------------------------------------------------------------------ persistent decode step (decode_step.cu)
// Every layer of a decode-only step of at most a few tokens in one cooperative launch: one CTA per SM, a
// static per-CTA list of work items per layer and phase (QKV tiles, attention splits, o_proj tiles,
// gate|up tiles, down tiles), weights and K/V streamed into a shared-memory ring ahead of need, and
// activations handed between phases as tagged 64-bit words (value bits | tag << 32).
struct DsLayer {
  const bf16* qkv;  // packed [(Hq + 2 Hkv) d][H]
  const bf16* o;    // packed [H][Hq d]
  const bf16* gu;   // packed [2I][H], gate/up rows interleaved per 16-row tile
  const bf16* down; // packed [H][I]
  const float* qkv_bias;  // or null
  const float* q_norm;    // or null
  const float* k_norm;
  const float* in_norm;
  const float* post_norm;
};
enum DsPhase { DS_QKV = 0, DS_ATTN = 1, DS_O = 2, DS_GU = 3, DS_DOWN = 4, DS_PHASES = 5 };
struct DecodeStepParams {
  CUtensorMap kv_map;     // the KV pool as rows of head_dim bf16 ([L][2][NB + 1][Hkv][16] rows), 64 x 16 boxes,
                          // 128-byte swizzle: K/V blocks land in shared memory in a bank-conflict-free order
  int L, H, Hq, Hkv, d, I, V, NB, mbs, max_pos;
  float eps, scale_log2;
  const DsLayer* layers;  // device [L]
  const bf16* embed;      // packed [V][H]
  const float* final_norm;
  const float* rope;      // [max_pos][d/2][2]
  bf16* kv;               // [L][2][NB + 1][Hkv][16][d]
  int T;                  // rows of the step (one token each)
  const int* ids;
  const int* prev_row;
  const int* prev_ids;
  int prev_rows;
  const int* pos;
  const int* seq;
  const int* bt;          // [rows][mbs]
  const int* sched_off;   // [gridDim.x][DS_PHASES + 1]: item ranges of each CTA's phases
  const int* sched_items;
  int asplits;            // attention splits per (row, KV head) of this step, at most kDsMaxSplits
  int trows;              // rows of the activation staging planes (>= T)
  int kx;                 // row stride of the staging planes (elements)
  int slots_n;            // ring slots of 32 KB
  unsigned long long* h_ll;    // [trows][H]
  unsigned long long* qkv_ll;  // [trows][(Hq + 2 Hkv) d]
  unsigned long long* act_ll;  // [trows][I]
  unsigned long long* attn_ws;   // [trows][Hkv][kDsMaxSplits][G][d + 2]: each split's (O, max, sum)
  unsigned long long* attn_out;  // [trows][Hq d]: the attention output, merged by each row's last split
  unsigned int* epoch;    // [0]: this step's epoch (tags), [1]: epoch of a step given up after a timeout
  bf16* xn_h;             // outputs for the LM head: planes of h * final_norm [T][H]
  bf16* xn_l;
  float* sq;              //   per-token sum of squares of h (one part)
  int sq_stride;
  float* h_out;           //   the final residual [T][H]
  int* slots;             //   [T] KV slot of each token (-1 padding)
  int* status;
  int* diag;              // [4]: the first wait that gave up -- site (DsWaitSite), block, thread, layer
  const void* pf_ptr;     // the start of the LM head's weights, prefetched into L2 during the last layer
  unsigned long long pf_bytes;
};
// Where a wait of the persistent decode kernel gave up (recorded in DecodeStepParams::diag).
enum DsWaitSite { WAIT_RING_FULL = 1, WAIT_RING_EMPTY = 2, WAIT_STAGE = 3, WAIT_HEAD = 4, WAIT_ATTN_MERGE = 6,
                  WAIT_RESIDUAL = 7 };
// Ring slot size, and the shared memory a launch needs for `trows` staged rows of width kmax.
constexpr int kDsSlotBytes = 32 * 1024;
constexpr int kDsMaxItems = 256;  // work items of one CTA per layer (all phases)
constexpr int kDsMaxSplits = 16;  // attention key splits per (row, KV head)
size_t decode_step_smem(int slots_n, int trows, int kx, int d, int G, int H, int layers);
// The kernel's shared-memory limit is raised on first use; false if the device cannot host the grid.
cudaError_t decode_step_prepare(size_t smem, int* max_ctas_per_sm);
cudaError_t launch_decode_step(const DecodeStepParams& p, int grid, size_t smem, cudaStream_t s);

// The launchers whose kernels depend on the 16-bit element format, built again for IEEE binary16
// weights, K/V and operand planes (the fp16 variant of a model; see common.cuh).  Same arguments and
// behaviour as the bfloat16 launchers above.
namespace f16 {
cudaError_t launch_pack(const bf16* src, bf16* dst, int N, int K, int interleave_half, cudaStream_t s);
cudaError_t launch_bf16_to_f32(const bf16* src, float* dst, int64_t n, cudaStream_t s);
cudaError_t launch_embed(const EmbedParams& p, const LaunchOpts& o, cudaStream_t s);
cudaError_t launch_gemm(const GemmParams& p, int epi, bool norm_in, const LaunchOpts& o, cudaStream_t s,
                        const TcMaps* tc = nullptr);
cudaError_t launch_attn_decode(const AttnDecodeParams& p, const LaunchOpts& o, cudaStream_t s);
int attn_flat_ctas(int d, int rows, int sms);
cudaError_t launch_attn_prefill(const AttnPrefillParams& p, const LaunchOpts& o, cudaStream_t s);
}  // namespace f16

}  // namespace grd
