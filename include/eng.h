/*
 * eng.h -- C ABI of the GB300 fused serving step (libeng.so).
 *
 * One call of eng_step runs one serving step of a Qwen3/Qwen2.5-style dense
 * decoder over one unpadded packed sequence: prefill chunks first, decode
 * tokens last ("One forward per step", section "What changed").  Every step of
 * the forward runs in this library's CUDA kernels (sm_103a): embedding gather,
 * fused residual-add + RMSNorm, one concatenated QKV GEMM, per-head QK-RMSNorm,
 * RoPE applied inside the paged KV-cache write, attention split inside the call
 * (packed causal prefill kernel for chunk positions, one-row-per-request paged
 * decode kernel for decode positions), output projection with residual, one
 * concatenated gate|up GEMM with fused SiLU-and-mul, the down projection with
 * residual, the final norm, the LM head and on-device greedy / Gumbel-max
 * sampling.  The step makes no host synchronisation.  Decode-only steps are
 * padded to the smallest captured batch size and replayed as one CUDA graph
 * over static buffers ("33. Removing overhead: fusion, graphs and async
 * scheduling", section "CUDA graphs for a changing batch").
 *
 * Conventions for every function below:
 *   - returns ENG_OK (0) on success, a negative ENG_E* code otherwise; the
 *     message of the last failure is available from eng_last_error;
 *   - "host" pointers are ordinary CPU memory (pinned memory is faster but not
 *     required); "device" pointers are CUDA global memory of the engine's GPU;
 *   - an engine is bound to one CUDA stream and one GPU and is not thread-safe.
 */
#ifndef ENG_H
#define ENG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ errors */
#define ENG_OK 0
#define ENG_EINVAL (-1)    /* bad argument, shape or request order (the pages raise ValueError) */
#define ENG_ECAPACITY (-2) /* a position at or past max_blocks_per_seq * block_size ("19. Fast decode",
                              StaticKVCache: prompt plus new tokens exceed the capacity) */
#define ENG_ENOMEM (-3)    /* a device or pinned-host allocation failed */
#define ENG_EPOOL (-4)     /* the KV block pool has fewer free blocks than requested */
#define ENG_ECUDA (-5)     /* a CUDA runtime call failed (no device, launch failure, ...) */
#define ENG_EDEVICE (-6)   /* a kernel-side check failed; see eng_status */
#define ENG_ESTATE (-7)    /* call not valid in the engine's current state */

/* bits of the device status word (eng_status) */
#define ENG_STATUS_BAD_BLOCK 1    /* a block-table entry outside [0, num_blocks): write redirected to scratch */
#define ENG_STATUS_BAD_POSITION 2 /* a position outside the block table: write redirected to scratch */
#define ENG_STATUS_NAN 4          /* a non-finite logit met the sampler */
#define ENG_STATUS_TIMEOUT 8      /* a bounded wait inside a kernel gave up */

/* ------------------------------------------------------------------ dtypes */
#define ENG_DTYPE_BF16 0
#define ENG_DTYPE_F16 1 /* IEEE binary16: the fp16 variant of a model */
#define ENG_DTYPE_F32 2

typedef struct eng eng_t;

/*
 * Model and engine shape.  Projection widths must be multiples of 16 (rows)
 * and reduction widths multiples of 32: hidden, q_heads*head_dim and
 * intermediate are multiples of 32, vocab a multiple of 16.  head_dim is 64 or
 * 128; q_heads is a multiple of kv_heads with at most 8 query heads per KV
 * head (a KV head's query heads and the low halves of their operands share one
 * 16-row tensor-core tile in decode attention); block_size must be 16.  max_reqs bounds the requests of one step and
 * the capture sizes; max_tokens bounds the packed tokens of one step;
 * max_blocks_per_seq bounds a block-table row (positions < max_blocks_per_seq * 16).
 */
typedef struct {
  int32_t layers, hidden, q_heads, kv_heads, head_dim, intermediate, vocab;
  float rms_eps;     /* RMSNorm epsilon, also used by the QK-norms */
  double rope_theta; /* RoPE base: inv_freq_i = theta^(-2i/head_dim) */
  int32_t qk_norm;   /* 1: per-head RMSNorm of q and k before RoPE (Qwen3) */
  int32_t qkv_bias;  /* 1: q/k/v projections carry a bias (Qwen2.5) */
  int32_t tie_embeddings; /* 1: the LM head is the embedding matrix */
  int32_t dtype;          /* ENG_DTYPE_BF16 or ENG_DTYPE_F16: the 16-bit format of the weights, the K/V
                             cache and the activation operand planes (hi/lo pairs of that format).  An
                             fp16 engine runs every step on the per-layer kernels (the persistent decode
                             kernel is built for bf16) */
  int32_t block_size, num_blocks, max_reqs, max_tokens, max_blocks_per_seq;
  int32_t sampling_filters; /* 1: steps may ask for top-k / top-p (eng_step_t.top_k, .top_p); every step and
                               every captured graph then also writes the logits and runs the filter kernel */
} eng_config_t;

/*
 * One weight tensor, named as in Hugging Face Qwen checkpoints:
 *   model.embed_tokens.weight [vocab, hidden]
 *   model.layers.{i}.input_layernorm.weight [hidden]
 *   model.layers.{i}.self_attn.{q,k,v}_proj.weight [out, hidden] (+ .bias when qkv_bias)
 *   model.layers.{i}.self_attn.{q,k}_norm.weight [head_dim] (when qk_norm)
 *   model.layers.{i}.self_attn.o_proj.weight [hidden, q_heads*head_dim]
 *   model.layers.{i}.post_attention_layernorm.weight [hidden]
 *   model.layers.{i}.mlp.{gate,up}_proj.weight [intermediate, hidden]
 *   model.layers.{i}.mlp.down_proj.weight [hidden, intermediate]
 *   model.norm.weight [hidden]
 *   lm_head.weight [vocab, hidden] (only when tie_embeddings == 0)
 * Row-major, dtype = the config's dtype (or ENG_DTYPE_F32 for norm weights and
 * biases); ENG_EINVAL for a matrix of the other 16-bit format.  on_device = 1 if `data` is a device pointer of the engine's GPU.
 */
typedef struct {
  const char* name;
  const void* data;
  int64_t numel;
  int32_t dtype;
  int32_t on_device;
} eng_tensor_t;

/*
 * One packed step, all arrays in host memory, read before eng_step returns:
 *   token_ids[num_tokens], positions[num_tokens]: absolute position of each token;
 *   cu_seqlens[num_reqs + 1]: request r owns tokens cu_seqlens[r] .. cu_seqlens[r+1]-1
 *     (cu_seqlens[0] = 0, non-decreasing, cu_seqlens[num_reqs] = num_tokens,
 *     every request at least one token, requests with several tokens first);
 *   block_tables[num_reqs * bt_stride]: row r lists request r's KV blocks in order
 *     (bt_stride <= max_blocks_per_seq columns; unused entries are ignored);
 *   seq_lens[num_reqs]: keys visible to request r's last query = its position + 1;
 *   temperature[num_reqs]: 0 selects greedy argmax, > 0 Gumbel-max at that temperature;
 *   seed, offset: Philox key and counter words of this step's Gumbel noise;
 *   top_k[num_reqs], top_p[num_reqs] (each may be NULL: no such filter): the filters of
 *     eng_sample_filtered ahead of request r's draw (top_k <= 0 or >= vocab, top_p outside (0, 1): off;
 *     top_p finite); an engine created with sampling_filters = 0 rejects any active filter (ENG_EINVAL).
 * A request's positions must be consecutive and end at seq_lens[r] - 1.
 */
typedef struct {
  int32_t num_tokens, num_reqs, bt_stride;
  const int32_t* token_ids;
  const int32_t* positions;
  const int32_t* cu_seqlens;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const float* temperature;
  uint64_t seed, offset;
  const int32_t* top_k;
  const float* top_p;
} eng_step_t;

/* What the last eng_step did (for tests and benchmarks). */
typedef struct {
  int32_t replayed;     /* 1: a captured graph was replayed; 2: the projection pieces of a mixed step were
                           replayed with attention launched between them (eng_capture_mixed); 0: eager */
  int32_t bucket;       /* capture size replayed: requests, or tokens when piecewise (num_reqs when eager) */
  int32_t launches;     /* kernels launched (the graph's kernel count when replayed) */
  int32_t num_prefill;  /* requests routed to the packed prefill attention kernel */
  int64_t h2d_bytes;    /* bytes copied host -> device by the step */
} eng_step_info_t;

/*
 * eng_create -- allocate an engine and load fused weights.
 * ("33. Removing overhead", section "Fewer, larger matmuls": Q/K/V and gate/up
 * are concatenated once at load time.)  The weights are copied and re-laid out
 * into the engine's own device memory, so the caller may free its tensors on
 * return.  Allocates the paged KV pool [layers][2][num_blocks + 1][kv_heads][16][head_dim]
 * bf16 (the extra block is the scratch block; the pool is zero-filled) and all
 * static step buffers.  cuda_stream: the cudaStream_t to run on, or NULL for a
 * stream the engine creates.  Errors: ENG_EINVAL (config, missing/mis-sized
 * weight), ENG_ENOMEM, ENG_ECUDA.  *out is NULL on failure.
 * Decode-only steps of at most a few tokens (the largest power of two <= 8 whose
 * staged activation rows fit the kernel's shared memory) run every layer in one
 * persistent cooperative kernel, one CTA per SM ("19. Fast decode", section
 * "Where the time goes": the step's many small kernels); the environment variable
 * ENG_DECODE_KERNEL=0 at creation keeps them on the per-layer kernels.  Results
 * match the oracle either way and are bit-identical between eager steps and graph
 * replays of the same path.
 */
int eng_create(const eng_config_t* cfg, const eng_tensor_t* weights, int32_t n_weights, void* cuda_stream,
               eng_t** out);

/*
 * eng_capture -- record one CUDA graph per batch size, largest first, all
 * sharing the engine's single set of static buffers ("33. Removing overhead",
 * GraphRunner.capture; "(7) Graph Mode", section 4.1).  Every row of a capture
 * is a padding row (slot redirected to the scratch block, sequence length 0),
 * so capture writes only the scratch block of the KV pool.  sizes[n]: distinct
 * values in [1, max_reqs].  Synchronises the stream.  Errors: ENG_EINVAL, ENG_ECUDA.
 */
int eng_capture(eng_t* e, const int32_t* sizes, int32_t n);

/*
 * eng_capture_mixed -- piecewise graphs for mixed (and prefill) steps ("(7) Graph Mode", section
 * PIECEWISE: split at attention; "33. Removing overhead", section "CUDA graphs for a changing batch",
 * the mixed-batch case).  For each token bucket, the step's projections are recorded as L + 1 graphs:
 * the embedding and layer 0's QKV projection, then per layer the output projection, gate|up, down and the
 * next layer's QKV projection.  A later eng_step that is not decode-only, with num_tokens in
 * [65, bucket] and num_reqs < max_reqs, pads its tokens to the smallest such bucket (padding tokens belong
 * to request num_reqs, of length 0, whose K/V go to the scratch block), replays the pieces and launches
 * attention (packed prefill and split decode kernels, sized by the step's own composition) and the LM head
 * eagerly between and after them.  Results are identical to the eager step's bit for bit: both token
 * counts take the same kernels.  token_buckets: host int32[n], each in [65, max_tokens], distinct.
 * Synchronises the engine's stream.  Errors: ENG_EINVAL, ENG_ECUDA.
 */
int eng_capture_mixed(eng_t* e, const int32_t* token_buckets, int32_t n);

/*
 * eng_step -- run one packed step and write one sampled token id per request.
 * Decode-only steps (every request one token) with num_reqs <= the largest
 * captured size replay the smallest captured graph >= num_reqs, with rows
 * num_reqs.. padded (token 0, position 0, sequence length 0); every other step
 * runs the same kernels eagerly ("33. Removing overhead", GraphRunner.can_run).
 * out_ids_dev: device int32[num_reqs]; out_logits_dev: device float[num_reqs][vocab]
 * or NULL.  Both are written in stream order; eng_step returns without waiting
 * for the GPU, so synchronise the stream before reading them.  The request's
 * sampled id comes from its last packed token.  Errors: ENG_EINVAL (shapes,
 * order, block ids out of range), ENG_ECAPACITY, ENG_ECUDA.
 */
int eng_step(eng_t* e, const eng_step_t* step, int32_t* out_ids_dev, float* out_logits_dev);

/*
 * eng_step_async -- eng_step for a scheduler that prepares step N+1 while step N still runs ("33.
 * Removing overhead", the async-scheduling section: the next step's inputs are staged before the
 * previous step's sampled tokens reach the host).  prev_row: host int32[num_tokens]; -1 takes
 * step->token_ids[t] as usual; r >= 0 takes, on the device, the id the previous step sampled for its
 * request row r (step->token_ids[t] is then ignored).  The previous step is the last eng_step,
 * eng_step_async, eng_decode or eng_profile step of this engine since the last eng_capture.  The ids are
 * gathered inside the step's first kernel, so a decode-only step still replays its graph.  A later
 * eng_decode continues the batch as usual.  Errors: those of eng_step, and ENG_EINVAL when prev_row is
 * NULL or an entry is outside [-1, previous num_reqs).
 */
int eng_step_async(eng_t* e, const eng_step_t* step, const int32_t* prev_row, int32_t* out_ids_dev,
                   float* out_logits_dev);

/* eng_last_step_info -- what the last successful eng_step (or eng_decode) did. */
int eng_last_step_info(const eng_t* e, eng_step_info_t* info);

/*
 * eng_decode -- run n_steps further pure-decode steps entirely on the device, continuing the batch of
 * the last eng_step, which must have been decode-only.  "19. Fast decode", section "Static shapes and a
 * static cache" and the fast decoder's step: run, sample, record, advance -- every step reads only
 * static device buffers, so no host value depends on the GPU's results.  After each step a request's
 * sampled id becomes its next input token, its position and sequence length grow by one, and the
 * Philox offset grows by one.  Each step replays the captured graph of the last step's bucket (or runs
 * eagerly when none applies), so its kernels and results are those of eng_step.
 * out_ids_dev: device int32[n_steps][num_reqs], step-major, written in stream order; the call returns
 * without waiting for the GPU.  The caller must already hold the KV blocks of the new positions in the
 * block tables it passed to eng_step.  Errors: ENG_ESTATE (no decode batch to continue), ENG_ECAPACITY
 * (a sequence would outgrow its block-table row or max_blocks_per_seq * 16), ENG_EINVAL, ENG_ECUDA.
 */
int eng_decode(eng_t* e, int32_t n_steps, int32_t* out_ids_dev);

/*
 * eng_generate -- eng_decode with stop tokens checked once every check_every steps ("19. Fast decode",
 * the section on syncs: one synchronisation per check; tokens generated after a stop are trimmed
 * afterwards, so at most check_every - 1 steps are wasted).  Continues the decode batch of the last
 * eng_step like eng_decode, in groups of min(check_every, steps left) device-resident steps; after each
 * group one copy brings the group's ids to the host, where each request's first stop id is found.  The
 * call ends when every request has met a stop id or max_steps steps have run.  Requests that stopped keep
 * decoding (shapes stay static) until the call ends; their later tokens are trimmed.
 * stop_ids: host int32[n_stop] (may be NULL when n_stop = 0).  out_tokens: host int32[num_reqs][max_steps]:
 * request r's tokens, -1 past out_lengths[r].  out_lengths: host int32[num_reqs]: tokens up to and
 * including the first stop id, or every step run when there is none.  Returns the number of steps run
 * (>= 0; a multiple of check_every unless max_steps cut the last group), or ENG_EINVAL, ENG_ESTATE,
 * ENG_ECAPACITY (checked for all max_steps before any step runs), ENG_ENOMEM, ENG_ECUDA.  The engine's
 * batch continues after the steps that ran.
 */
int eng_generate(eng_t* e, int32_t max_steps, int32_t check_every, const int32_t* stop_ids, int32_t n_stop,
                 int32_t* out_tokens, int32_t* out_lengths);

/* Kernel kinds reported by eng_profile. */
#define ENG_K_EMBED_NORM 0
#define ENG_K_NORM 1
#define ENG_K_GEMM_QKV 2
#define ENG_K_ROPE_KV 3
#define ENG_K_ATTN_DECODE 4
#define ENG_K_ATTN_PREFILL 5
#define ENG_K_GEMM_O 6
#define ENG_K_GEMM_GATE_UP 7
#define ENG_K_GEMM_DOWN 8
#define ENG_K_LM_HEAD 9
#define ENG_K_ADVANCE 10
#define ENG_K_SAMPLE_FILTER 11
#define ENG_K_DECODE_LAYERS 12 /* every layer of a small decode-only step in one persistent kernel */

/*
 * eng_profile -- time every kernel of one further decode step of the current batch (as eng_decode with
 * n_steps = 1, launched eagerly on the engine's stream) with a CUDA event pair around each launch, and
 * report per launch its kind (ENG_K_*), duration in milliseconds and algorithmic HBM bytes (weights
 * read once, activations in and out, K/V read over the rows' current lengths and written at the new
 * position).  A 20 ms device-side hold runs first so that the whole step is enqueued before its first
 * kernel starts: the pairs then time device work only (launches run back to back, without the overlap
 * programmatic dependent launch gives them inside a graph).  kinds/ms/bytes: host arrays of `capacity`
 * entries; *count receives the launch count.  Synchronises the stream.  Errors: ENG_ESTATE (no decode batch), ENG_EINVAL (capacity too small).
 */
int eng_profile(eng_t* e, int32_t capacity, int32_t* kinds, float* ms, int64_t* bytes, int32_t* count);

/*
 * eng_pool_alloc / eng_pool_free -- the paged KV block pool ("One forward per
 * step": a pool of fixed-size blocks, blocks reserved when a request is
 * admitted).  The free list starts as 0..num_blocks-1; allocation takes from
 * the front, freeing appends to the back.  The scratch block (num_blocks) is
 * never handed out.  alloc: out_ids[n] host; ENG_EPOOL if fewer than n are
 * free (nothing allocated).  free: ENG_EINVAL if an id is not allocated
 * (nothing freed).
 */
int eng_pool_alloc(eng_t* e, int32_t n, int32_t* out_ids);
int eng_pool_free(eng_t* e, const int32_t* ids, int32_t n);
int32_t eng_pool_free_count(const eng_t* e);

/*
 * eng_status -- synchronise the stream and return the device status word
 * (ENG_STATUS_* bits, 0 = clean), or a negative ENG_E* code if the stream
 * holds a CUDA error.  reset != 0 clears the word afterwards.
 */
int eng_status(eng_t* e, int32_t reset);

/* eng_set_eager -- 1: never replay graphs (debugging; "(7) Graph Mode", section 6: disable graphs when debugging). */
int eng_set_eager(eng_t* e, int32_t eager);

/*
 * eng_kv_pool -- device address and size of the paged KV pool, laid out as
 * bf16 [layers][2 (K, V)][num_blocks + 1][kv_heads][16][head_dim].  Lets a
 * caller pre-fill context K/V for synthetic workloads or inspect the cache.
 */
int eng_kv_pool(eng_t* e, void** dev_ptr, int64_t* bytes);

/*
 * eng_debug_buffer -- device address and byte size of a named static buffer
 * holding the last step's intermediate values: "hidden" (float [max_tokens][hidden],
 * residual stream after the last layer), "slots" (int32 [max_tokens], KV slot
 * of each packed token, -1 for padding rows), "logits" (float [max_reqs][vocab]),
 * "ids" (int32 [max_reqs]).  Read-only for the caller.
 */
int eng_debug_buffer(eng_t* e, const char* name, void** dev_ptr, int64_t* bytes);

/* eng_stream -- the cudaStream_t the engine runs on. */
void* eng_stream(const eng_t* e);

/* eng_last_error -- message of the last failure on this engine (or of the last failed eng_create if e is NULL). */
const char* eng_last_error(const eng_t* e);

/* eng_destroy -- free every resource of the engine (synchronises its stream).  NULL is a no-op. */
void eng_destroy(eng_t* e);

/* ------------------------------------------------------------------
 * Standalone kernels, for unit tests of the device arithmetic.
 * ------------------------------------------------------------------ */

/*
 * eng_philox_uniforms -- the sampler's uniforms ("19. Fast decode", section
 * "Sampling without the CPU") for rows x vocab entries: out[r][v] =
 * (2 * (x >> 9) + 1) * 2^-24 with x word (v & 3) of Philox4x32-10 under key
 * (seed_lo, seed_hi) at counter (v >> 2, r, offset_lo, offset_hi).
 * out_dev: device float[rows][vocab].  stream: cudaStream_t or NULL (legacy default stream).
 */
int eng_philox_uniforms(uint64_t seed, uint64_t offset, int32_t rows, int32_t vocab, float* out_dev, void* stream);

/*
 * eng_gumbel -- g[i] = -ln(-ln u[i]) with the sampler's own float32 logarithm
 * (correctly rounded +, -, *, / only).  u_dev, g_dev: device float[n]; u in (0, 1).
 */
int eng_gumbel(const float* u_dev, float* g_dev, int64_t n, void* stream);

/*
 * eng_sample -- the sampler on caller logits: out_ids[r] = argmax_v of
 * logits[r][v] (temperature 0) or of logits[r][v] * (1/T_r) + g[r][v] with the
 * Gumbel noise of eng_philox_uniforms / eng_gumbel; ties go to the lowest index.
 * logits_dev: device float[rows][vocab]; temperature: host float[rows];
 * out_ids_dev: device int32[rows].
 */
int eng_sample(const float* logits_dev, int32_t rows, int32_t vocab, const float* temperature, uint64_t seed,
               uint64_t offset, int32_t* out_ids_dev, void* stream);

/*
 * eng_sample_noalloc -- eng_sample without any device allocation.  The pages have no counterpart: this
 * entry point exists for callers that may not allocate device memory during a call -- for example a
 * serving runtime that has handed all free device memory to its own pool or caching allocator, or a
 * latency-critical loop that cannot take an allocation's implicit synchronisation.
 * Arguments, results and errors are those of eng_sample, with rows <= 4096 (ENG_EINVAL beyond that,
 * with a message).  The per-call scratch (the rows' inverse temperatures and the four Philox words) lives
 * in one fixed array of 16 KiB + 16 bytes inside this library; every GPU that loads the library holds it
 * until the process exits.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and keeps it; make that first call before any stream
 * capture.  The kept address is not valid after cudaDeviceReset.  All calls on a device share the array,
 * and each call rewrites every word it reads, so nothing carries over between calls -- but calls whose
 * work overlaps on the GPU (for example on two unordered streams) race on it.  The words reach the array
 * as the launch parameters of a small staging kernel on `stream`, so the call neither synchronises nor
 * reads host memory after it returns; synchronise the stream before reading out_ids_dev.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 */
int eng_sample_noalloc(const float* logits_dev, int32_t rows, int32_t vocab, const float* temperature,
                       uint64_t seed, uint64_t offset, int32_t* out_ids_dev, void* stream);

/*
 * eng_sample_filtered -- the sampler with top-k and top-p filters ahead of the draw ("19. Fast decode",
 * section "Sampling without the CPU": filtered logits become -inf before the argmax; a fixed k and a
 * sort-and-mask top-p keep the shapes static).  Per row r, with s = logits[r][v] * (1/T_r) in float32:
 *   - rank order: larger logit first, equal logits (+0 and -0 equal) by increasing index;
 *   - top-k keeps the first top_k[r] entries of that order (top_k[r] <= 0 or >= vocab: no filter);
 *   - top-p keeps, among the top-k survivors, the shortest prefix of the order whose softmax(s) mass
 *     reaches p = top_p[r] (no filter unless 0 < p < 1).  The cut is exact integer arithmetic: weights
 *     w_v = floor(e^(s_v - s_max) * 2^32) with the library's own float32 exp (eng_exp_f32), p rounded
 *     to units of 2^-24 (at least one), and entry v survives iff the weight ahead of it, times 2^24, is
 *     below p_units * (total weight).  The top entry always survives.
 *   - out_ids[r] = argmax over the survivors of s + g, g the Gumbel noise of eng_sample (same seed, offset
 *     and row), ties to the lowest index; temperature 0 takes the plain argmax (no filter can drop it).
 * logits_dev: device float[rows][vocab], finite (a non-finite logit is skipped; it never survives);
 * z / T must stay finite.  temperature: host float[rows], finite, >= 0.  top_k: host int32[rows] or NULL
 * (no top-k).  top_p: host float[rows], finite, or NULL (no top-p).  out_ids_dev: device int32[rows].
 * out_kept_dev: device int32[rows] or NULL; receives each row's survivor count (1 at temperature 0).
 * The call allocates a small device block for the per-row parameters and synchronises `stream` before it
 * returns.  Errors: ENG_EINVAL (arguments, with a message), ENG_ENOMEM, ENG_ECUDA.
 */
int eng_sample_filtered(const float* logits_dev, int32_t rows, int32_t vocab, const float* temperature,
                        const int32_t* top_k, const float* top_p, uint64_t seed, uint64_t offset, int32_t* out_ids_dev,
                        int32_t* out_kept_dev, void* stream);

/*
 * eng_exp_f32 -- out[i] = e^d[i] for float32 d[i] <= 0, the exp of eng_sample_filtered's top-p weights:
 * n = rint(d / ln 2), r = d - n ln2_hi - n ln2_lo, e^r by its Taylor series to r^7/7! (Horner), times 2^n;
 * every step one correctly rounded float32 operation; 0 for d < -23.  d_dev, out_dev: device float[n].
 */
int eng_exp_f32(const float* d_dev, float* out_dev, int64_t n, void* stream);

/* ---------------------------------------------------------------- a mixture-of-experts layer
 * "33. Removing overhead", section "A MoE layer that never asks the host": the assignments (token, slot)
 * are grouped by expert on the device, each group padded to whole blocks, and one grouped GEMM multiplies
 * every block by its expert's weights.  These are standalone calls (no engine configuration has experts):
 * every pointer is device memory, nothing is allocated or synchronised, and every launch's shape depends only
 * on the token count N, the experts per token k, the expert count E and the block size, so the calls can be
 * captured in a CUDA graph.  Expert weights are bf16 (16-bit patterns); gate_up[e] holds the expert's gate
 * rows first, then its up rows; the activation is silu(gate) * up.
 */

/*
 * eng_moe_route -- for each token row t: logits x[t] . w_router[e] (bf16 operands, float32 accumulation),
 * softmax over the E experts, the top_k most probable experts (ties to the lower id, most probable first)
 * and their probabilities renormalised to sum to 1 (Qwen3-MoE's router; the pages call it from a chapter
 * not included).  x: bf16 [N][hidden]; w_router: bf16 [E][hidden]; weights: float [N][top_k]; expert_ids:
 * int32 [N][top_k].  hidden % 8 == 0, 1 <= top_k <= min(32, E), E <= 4096.  Errors: ENG_EINVAL, ENG_ECUDA.
 */
int eng_moe_route(const void* x, const void* w_router, int32_t num_tokens, int32_t hidden, int32_t num_experts,
                  int32_t top_k, float* weights, int32_t* expert_ids, void* stream);

/* Rows of the grouped layout: N k assignments plus block_m - 1 padding rows per expert, in whole blocks. */
int64_t eng_moe_padded_rows(int32_t num_tokens, int32_t top_k, int32_t num_experts, int32_t block_m);

/*
 * eng_moe_align -- group the flat assignments a = t * top_k + j by expert.  expert_ids: int32 [N][top_k].
 * sorted_ids: int32 [M], M = eng_moe_padded_rows(...): the assignment each row of the grouped GEMM handles,
 * expert 0's group first, ascending inside a group, N * top_k on a padding row.  block_expert: int32
 * [M / block_m]: the expert owning each block (E - 1 for blocks past the groups).  info: int32 [2]:
 * [0] the rows the groups occupy (a multiple of block_m), [1] the assignments whose expert id is outside
 * [0, E) (placed in no group).  E <= 1024.  Errors: ENG_EINVAL, ENG_ECUDA.
 */
int eng_moe_align(const int32_t* expert_ids, int32_t num_tokens, int32_t top_k, int32_t num_experts, int32_t block_m,
                  int32_t* sorted_ids, int32_t* block_expert, int32_t* info, void* stream);

/* Bytes of device workspace eng_moe_mlp needs for these sizes. */
int64_t eng_moe_workspace_bytes(int32_t num_tokens, int32_t top_k, int32_t num_experts, int32_t hidden,
                                int32_t inter);

/*
 * eng_moe_mlp -- out[t] = sum over j < top_k (in order) of weights[t][j] * down[e] (silu(gate[e] x[t]) *
 * up[e] x[t]), e = expert_ids[t][j]: eng_moe_align with blocks of 16 rows, then one grouped tensor-core GEMM
 * for gate|up with SiLU * up fused (the products in float32, kept as bf16 hi/lo pairs), one for down scaled
 * by the router weight, and the sum of each token's assignment rows.  x: bf16 [N][hidden]; gate_up: bf16
 * [E][2 inter][hidden]; down: bf16 [E][hidden][inter]; weights: float [N][top_k]; expert_ids: int32
 * [N][top_k] in [0, E) (an id outside adds nothing); out: float [N][hidden].  hidden % 64 == 0,
 * inter % 64 == 0, E <= 1024.  workspace: device memory of at least eng_moe_workspace_bytes(...) bytes,
 * owned by the caller and not shared by overlapping calls.  Errors: ENG_EINVAL, ENG_ECUDA.
 */
int eng_moe_mlp(const void* x, const void* gate_up, const void* down, const float* weights, const int32_t* expert_ids,
                int32_t num_tokens, int32_t hidden, int32_t inter, int32_t num_experts, int32_t top_k, float* out,
                void* workspace, int64_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ENG_H */
