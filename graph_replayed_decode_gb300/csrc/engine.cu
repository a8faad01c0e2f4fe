// engine.cu -- host side of libeng: the C ABI of include/eng.h.
//
// Owns the fused device weights, the paged KV pool, the static step buffers (the only memory a captured
// graph reads), the KV block pool policy and the per-step kernel sequence:
//
//   embed + RMSNorm -> per layer [ QKV GEMM (+bias) -> QK-norm + RoPE + KV write -> attention
//   (prefill rows packed, decode rows one per request) -> o_proj GEMM + residual -> RMSNorm ->
//   gate|up GEMM + SiLU*up -> down GEMM + residual -> RMSNorm (next layer) ] -> final RMSNorm at each
//   request's last token -> LM head GEMM + greedy / Gumbel-max sampling.
//
// "33. Removing overhead", section "CUDA graphs for a changing batch": decode-only steps are padded to
// the smallest captured bucket and replayed from static buffers; every host value a kernel grid depends
// on is the bucket's, never the step's.  Section "Async scheduling" of the same page and "19. Fast
// decode", section "Host synchronizations": the step never waits for the GPU -- inputs go through a
// pinned staging ring whose slots are reused only after their copy has completed.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <deque>
#include <map>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/eng.h"
#include "kernels.h"

using namespace grd;

namespace {

thread_local std::string g_create_error;

constexpr int kSlots = 4;  // pinned staging ring depth

struct Layer {
  bf16* qkv = nullptr;        // packed [(Hq + 2 Hkv) d][H]
  float* qkv_bias = nullptr;  // [(Hq + 2 Hkv) d] or null
  float* q_norm = nullptr;    // [d] or null
  float* k_norm = nullptr;
  bf16* o = nullptr;          // packed [H][Hq d]
  bf16* gu = nullptr;         // packed [2I][H], gate/up rows interleaved per 16-row tile
  bf16* down = nullptr;       // packed [H][I]
  float* in_norm = nullptr;   // [H]
  float* post_norm = nullptr; // [H]
  // tensor-core path (steps of kTcTokens tokens or more): row-major copies (gate|up rows interleaved as in
  // the packed copy) and their tensor maps; null when the projection's shape does not allow it
  bf16* qkv_rm = nullptr;
  bf16* o_rm = nullptr;
  bf16* gu_rm = nullptr;
  bf16* down_rm = nullptr;
  CUtensorMap m_qkv{}, m_o{}, m_gu{}, m_down{};
};

// Word offsets of the step inputs inside one staging slot (host) and the device input region.
struct InLayout {
  size_t ids, pos, prev, tok2req, cu, seq, last, invt, topk, punit, rng, wlog, wkey, step, items, bt, words;
};

// One projection of the step with its two launch plans: [0] for steps of at most 8 tokens, [1] for
// larger ones (the plan only depends on the weight shape and the class, so every token count of a class
// computes each output with the same summation order).
struct GemmPlan {
  int RG = 1, S = 1, ktn = 0;
};
struct GemmSite {
  int N = 0, K = 0, rg_fixed = 0;
  GemmPlan plan[2];
  bool tc = false;      // the shape allows the tensor-core path (128-row tiles)
  bool tc_mid = false;  //   and it serves steps of kTcTokens..kTcPrefillTokens-1 tokens too
  int tc_S = 1;         //   with this many K splits there (prefill-sized steps: none)
  bool use_tc(int T) const { return tc && (T >= kTcPrefillTokens || (tc_mid && T >= kTcTokens)); }
  int tc_splits(int T) const { return T >= kTcPrefillTokens ? 1 : tc_S; }
  const GemmPlan& for_tokens(int T) const { return plan[T >= kLargePlanTokens ? 1 : 0]; }
  int groups(int T) const { return use_tc(T) ? N / 128 : N / 16 / for_tokens(T).RG; }
  int max_groups() const { return std::max(N / 16 / plan[0].RG, N / 16 / plan[1].RG); }
};

}  // namespace

struct eng {
  eng_config_t c{};
  int device = 0;
  int sms = 0;  // SM count of the device (grid sizing)
  bool f16 = false;  // IEEE binary16 weights, K/V and operand planes (the grd::f16 kernels)
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  cudaStream_t cap_stream = nullptr;
  std::vector<void*> allocations;
  std::string err;

  // weights
  bf16* embed = nullptr;  // packed [V][H]
  bf16* lm = nullptr;     // packed [V][H] (== embed when tied)
  float* final_norm = nullptr;
  std::vector<Layer> layers;
  float* rope = nullptr;  // [max_pos][d/2][2]
  int max_pos = 0;

  // KV pool [L][2][NB + 1][Hkv][16][d]
  bf16* kv = nullptr;
  size_t kv_elems = 0;

  // inputs
  InLayout in{};
  int* d_in = nullptr;
  int* h_in[kSlots] = {};
  cudaEvent_t ev[kSlots] = {};
  int slot = 0;
  int max_items = 0;

  // activations and outputs
  float* h = nullptr;      // [Tm][H]
  float* sq = nullptr;     // [Tm][sq_stride] per-token partial sums of squares of the residual
  int sq_stride = 1;
  // activations: q stays fp32 (the attention splits it); every projection input is written by its
  // producer as two bf16 planes hi = bf16(x), lo = bf16(x - hi)
  float* q = nullptr;      // [Tm][Hq][d]
  bf16* xn_h = nullptr;    // [Tm][H]     h * (next norm weight): QKV, gate|up and LM-head input
  bf16* xn_l = nullptr;
  bf16* attn_h = nullptr;  // [Tm][Hq d]  attention output: o_proj input
  bf16* attn_l = nullptr;
  bf16* act_h = nullptr;   // [Tm][I]     silu(gate) * up: down-projection input
  bf16* act_l = nullptr;
  float* logits = nullptr; // [Rm][V]
  int* ids = nullptr;      // [Rm]
  int* slots = nullptr;    // [Tm]
  unsigned long long* best = nullptr;
  float* keys = nullptr;            // [Rm][V] sampling keys from the LM head (engines with sampling filters)
  unsigned int* row_ext = nullptr;  // [Rm][2] the LM head's logit extremes, reset by the filter kernel
  int* done_counter = nullptr;
  int* status = nullptr;
  GemmSite g_qkv, g_o, g_gu, g_down, g_lm;
  CUtensorMap m_xn_h{}, m_xn_l{}, m_attn_h{}, m_attn_l{}, m_act_h{}, m_act_l{};  // activation planes (TC path)
  int split_blocks = 4, max_splits = 1;
  int attn_flat = 0;           // CTAs of the flat-partition decode attention
  float* attn_ws = nullptr;    // its partials of segments split between warps
  int* attn_counters = nullptr;
  int* ring = nullptr;  // [ring_cap][bucket] ids recorded by the advance kernel
  int ring_cap = 1024;

  // persistent decode step (decode_step.cu): decode-only steps of at most ds_rows tokens
  bool ds_on = false;
  int ds_rows = 0, ds_slots = 0, ds_kx = 0;
  size_t ds_smem = 0;
  DsLayer* ds_layers = nullptr;  // device [layers]
  unsigned long long *ds_h = nullptr, *ds_qkv = nullptr, *ds_act = nullptr;
  CUtensorMap ds_kv_map{};  // the KV pool as [rows][head_dim] bf16 for the kernel's swizzled block copies
  unsigned long long *ds_ws = nullptr, *ds_out = nullptr;
  unsigned int* ds_epoch = nullptr;
  int* ds_diag = nullptr;  // [4] the first wait of the persistent kernel that gave up (site, block, thread, layer)
  std::map<int, std::pair<int*, int*>> ds_sched;  // token count -> device (ranges, items)

  // the decode batch that eng_decode continues (host mirror of its lengths)
  int dec_R = 0, dec_rows = 0, dec_bt_stride = 0;
  int prev_rows = 0;  // requests of the last step (rows an async step may gather sampled ids from)
  std::vector<int> dec_seq;

  // per-launch event timing (eng_profile)
  bool prof_on = false;
  std::vector<cudaEvent_t> prof_ev;
  std::vector<int> prof_kind;
  std::vector<int64_t> prof_bytes;

  // pool
  std::deque<int> free_list;
  std::vector<uint8_t> used;

  // graphs
  std::map<int, cudaGraphExec_t> graphs;
  std::map<int, int> graph_launches;
  // piecewise graphs of mixed steps: token bucket -> the L + 1 projection pieces (enqueue_piece)
  std::map<int, std::vector<cudaGraphExec_t>> pieces;
  std::map<int, int> piece_launches;
  bool eager_only = false;
  bool pdl = false;
  bool l2_prefetch = true;
  int launches = 0;
  eng_step_info_t last{};
};

// ------------------------------------------------------------------ error helpers

static int fail(eng_t* e, int code, const std::string& msg) {
  if (e)
    e->err = msg;
  else
    g_create_error = msg;
  return code;
}

#define CUDA_OR_FAIL(e, call)                                                                        \
  do {                                                                                               \
    cudaError_t err_ = (call);                                                                       \
    if (err_ != cudaSuccess)                                                                         \
      return fail((e), ENG_ECUDA, std::string(#call) + ": " + cudaGetErrorString(err_));             \
  } while (0)

template <typename T>
static int dev_alloc(eng_t* e, T** p, size_t count) {
  void* v = nullptr;
  const size_t bytes = std::max<size_t>(count * sizeof(T), 16);
  cudaError_t r = cudaMalloc(&v, bytes);
  if (r != cudaSuccess) return fail(e, ENG_ENOMEM, std::string("cudaMalloc failed: ") + cudaGetErrorString(r));
  r = cudaMemset(v, 0, bytes);
  if (r != cudaSuccess) return fail(e, ENG_ECUDA, std::string("cudaMemset failed: ") + cudaGetErrorString(r));
  e->allocations.push_back(v);
  *p = static_cast<T*>(v);
  return ENG_OK;
}

#define TRY(x)                   \
  do {                           \
    int rc_ = (x);               \
    if (rc_ != ENG_OK) return rc_; \
  } while (0)

// ------------------------------------------------------------------ config checks

static std::string check_config(const eng_config_t& c) {
  if (c.layers < 1 || c.hidden < 32 || c.q_heads < 1 || c.kv_heads < 1 || c.intermediate < 32 || c.vocab < 16)
    return "non-positive model dimension";
  if (c.head_dim != 64 && c.head_dim != 128) return "head_dim must be 64 or 128";
  if (c.q_heads % c.kv_heads != 0) return "q_heads must be a multiple of kv_heads";
  if (c.q_heads / c.kv_heads > 8) return "at most 8 query heads per KV head";
  if (c.hidden % 32 || c.intermediate % 32 || (c.q_heads * c.head_dim) % 32) return "reduction widths must be multiples of 32";
  if (c.vocab % 16) return "vocab must be a multiple of 16";
  if (c.dtype != ENG_DTYPE_BF16 && c.dtype != ENG_DTYPE_F16) return "dtype must be ENG_DTYPE_BF16 or ENG_DTYPE_F16";
  if (c.block_size != 16) return "block_size must be 16";
  if (c.num_blocks < 1 || c.max_reqs < 1 || c.max_tokens < c.max_reqs || c.max_blocks_per_seq < 1)
    return "bad engine capacity (num_blocks, max_reqs <= max_tokens, max_blocks_per_seq)";
  if (!(c.rms_eps > 0.f) || !(c.rope_theta > 0.0)) return "rms_eps and rope_theta must be positive";
  if (c.sampling_filters != 0 && c.sampling_filters != 1) return "sampling_filters must be 0 or 1";
  return "";
}

// ------------------------------------------------------------------ weight loading

namespace {
struct WeightMap {
  std::unordered_map<std::string, const eng_tensor_t*> m;
  const eng_tensor_t* get(const std::string& n) const {
    auto it = m.find(n);
    return it == m.end() ? nullptr : it->second;
  }
};
}  // namespace

// Copies `numel` 16-bit values (the model's element type) of tensor `t` to device memory at dst.
static int copy_bf16(eng_t* e, const eng_tensor_t* t, bf16* dst, int64_t numel, const char* name) {
  if (!t) return fail(e, ENG_EINVAL, std::string("missing weight ") + name);
  if (t->numel != numel) return fail(e, ENG_EINVAL, std::string("wrong numel for ") + name);
  if (t->dtype != e->c.dtype)
    return fail(e, ENG_EINVAL, std::string(e->c.dtype == ENG_DTYPE_F16 ? "expected fp16 for " : "expected bf16 for ") + name);
  if (!t->data) return fail(e, ENG_EINVAL, std::string("null data for ") + name);
  CUDA_OR_FAIL(e, cudaMemcpyAsync(dst, t->data, numel * 2, t->on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice,
                                  e->stream));
  return ENG_OK;
}

// Loads a 1-D weight (f32, or the model's element type) as f32 at dst; tmp is a 16-bit scratch of at least
// numel values.
static int load_f32(eng_t* e, const eng_tensor_t* t, float* dst, int64_t numel, bf16* tmp, const char* name) {
  if (!t) return fail(e, ENG_EINVAL, std::string("missing weight ") + name);
  if (t->numel != numel) return fail(e, ENG_EINVAL, std::string("wrong numel for ") + name);
  if (!t->data) return fail(e, ENG_EINVAL, std::string("null data for ") + name);
  const cudaMemcpyKind k = t->on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
  if (t->dtype == ENG_DTYPE_F32) {
    CUDA_OR_FAIL(e, cudaMemcpyAsync(dst, t->data, numel * 4, k, e->stream));
  } else if (t->dtype == e->c.dtype) {
    CUDA_OR_FAIL(e, cudaMemcpyAsync(tmp, t->data, numel * 2, k, e->stream));
    CUDA_OR_FAIL(e, e->f16 ? f16::launch_bf16_to_f32(tmp, dst, numel, e->stream)
                           : launch_bf16_to_f32(tmp, dst, numel, e->stream));
  } else {
    return fail(e, ENG_EINVAL, std::string("unsupported dtype for ") + name);
  }
  return ENG_OK;
}

// For a projection on the tensor-core path: keep a row-major copy of the fused matrix in `src` ([N][K];
// with interleave_half > 0 the rows [A; B] are reordered as A rows 8i..8i+7 then B rows 8i..8i+7 per
// 16-row group, like the packed copy) and encode its tensor map.  A map the driver refuses turns the
// tensor-core path off for that projection.
static int keep_row_major(eng_t* e, GemmSite& site, const bf16* src, bf16** dst, CUtensorMap* map, int N, int K,
                          int interleave_half) {
  if (!site.tc) return ENG_OK;
  TRY(dev_alloc(e, dst, (size_t)N * K));
  if (interleave_half > 0) {
    const size_t row = (size_t)K * 2;
    CUDA_OR_FAIL(e, cudaMemcpy2DAsync(*dst, 16 * row, src, 8 * row, 8 * row, interleave_half / 8,
                                      cudaMemcpyDeviceToDevice, e->stream));
    CUDA_OR_FAIL(e, cudaMemcpy2DAsync(*dst + (size_t)8 * K, 16 * row, src + (size_t)interleave_half * K, 8 * row,
                                      8 * row, interleave_half / 8, cudaMemcpyDeviceToDevice, e->stream));
  } else {
    CUDA_OR_FAIL(e, cudaMemcpyAsync(*dst, src, (size_t)N * K * 2, cudaMemcpyDeviceToDevice, e->stream));
  }
  if (!make_tc_map(map, *dst, N, K, 128)) site.tc = false;
  return ENG_OK;
}

static int load_weights(eng_t* e, const eng_tensor_t* w, int32_t n) {
  const eng_config_t& c = e->c;
  WeightMap wm;
  for (int i = 0; i < n; ++i) {
    if (!w[i].name) return fail(e, ENG_EINVAL, "weight with null name");
    wm.m[w[i].name] = &w[i];
  }
  const int H = c.hidden, d = c.head_dim, Hq = c.q_heads, Hkv = c.kv_heads, I = c.intermediate, V = c.vocab;
  const int QKV = (Hq + 2 * Hkv) * d;
  const size_t tmp_elems = std::max<size_t>({(size_t)V * H, (size_t)2 * I * H, (size_t)QKV * H, (size_t)H * Hq * d});
  bf16* tmp = nullptr;
  {
    void* v = nullptr;
    cudaError_t r = cudaMalloc(&v, tmp_elems * 2);
    if (r != cudaSuccess) return fail(e, ENG_ENOMEM, "cudaMalloc of the load scratch failed");
    tmp = static_cast<bf16*>(v);
  }
  auto done = [&](int rc) {
    cudaStreamSynchronize(e->stream);
    cudaFree(tmp);
    return rc;
  };
  int rc;
#define LW(x)              \
  do {                     \
    rc = (x);              \
    if (rc != ENG_OK) return done(rc); \
  } while (0)

  LW(dev_alloc(e, &e->embed, (size_t)V * H));
  LW(copy_bf16(e, wm.get("model.embed_tokens.weight"), tmp, (int64_t)V * H, "model.embed_tokens.weight"));
  if (launch_pack(tmp, e->embed, V, H, 0, e->stream) != cudaSuccess) return done(fail(e, ENG_ECUDA, "pack launch"));
  if (c.tie_embeddings) {
    e->lm = e->embed;
  } else {
    LW(dev_alloc(e, &e->lm, (size_t)V * H));
    cudaStreamSynchronize(e->stream);
    LW(copy_bf16(e, wm.get("lm_head.weight"), tmp, (int64_t)V * H, "lm_head.weight"));
    if (launch_pack(tmp, e->lm, V, H, 0, e->stream) != cudaSuccess) return done(fail(e, ENG_ECUDA, "pack launch"));
  }
  LW(dev_alloc(e, &e->final_norm, H));
  cudaStreamSynchronize(e->stream);
  LW(load_f32(e, wm.get("model.norm.weight"), e->final_norm, H, tmp, "model.norm.weight"));

  e->layers.resize(c.layers);
  for (int l = 0; l < c.layers; ++l) {
    Layer& L = e->layers[l];
    const std::string p = "model.layers." + std::to_string(l) + ".";
    auto nm = [&](const char* s) { return p + s; };
    cudaStreamSynchronize(e->stream);
    // fused QKV: rows [q | k | v] ("33. Removing overhead", section "Fewer, larger matmuls")
    LW(dev_alloc(e, &L.qkv, (size_t)QKV * H));
    LW(copy_bf16(e, wm.get(nm("self_attn.q_proj.weight")), tmp, (int64_t)Hq * d * H, nm("self_attn.q_proj.weight").c_str()));
    LW(copy_bf16(e, wm.get(nm("self_attn.k_proj.weight")), tmp + (size_t)Hq * d * H, (int64_t)Hkv * d * H,
                 nm("self_attn.k_proj.weight").c_str()));
    LW(copy_bf16(e, wm.get(nm("self_attn.v_proj.weight")), tmp + (size_t)(Hq + Hkv) * d * H, (int64_t)Hkv * d * H,
                 nm("self_attn.v_proj.weight").c_str()));
    if (launch_pack(tmp, L.qkv, QKV, H, 0, e->stream) != cudaSuccess) return done(fail(e, ENG_ECUDA, "pack launch"));
    LW(keep_row_major(e, e->g_qkv, tmp, &L.qkv_rm, &L.m_qkv, QKV, H, 0));
    if (c.qkv_bias) {
      LW(dev_alloc(e, &L.qkv_bias, QKV));
      cudaStreamSynchronize(e->stream);
      LW(load_f32(e, wm.get(nm("self_attn.q_proj.bias")), L.qkv_bias, Hq * d, tmp, nm("self_attn.q_proj.bias").c_str()));
      cudaStreamSynchronize(e->stream);
      LW(load_f32(e, wm.get(nm("self_attn.k_proj.bias")), L.qkv_bias + Hq * d, Hkv * d, tmp,
                  nm("self_attn.k_proj.bias").c_str()));
      cudaStreamSynchronize(e->stream);
      LW(load_f32(e, wm.get(nm("self_attn.v_proj.bias")), L.qkv_bias + (Hq + Hkv) * d, Hkv * d, tmp,
                  nm("self_attn.v_proj.bias").c_str()));
    }
    if (c.qk_norm) {
      LW(dev_alloc(e, &L.q_norm, d));
      LW(dev_alloc(e, &L.k_norm, d));
      cudaStreamSynchronize(e->stream);
      LW(load_f32(e, wm.get(nm("self_attn.q_norm.weight")), L.q_norm, d, tmp, nm("self_attn.q_norm.weight").c_str()));
      cudaStreamSynchronize(e->stream);
      LW(load_f32(e, wm.get(nm("self_attn.k_norm.weight")), L.k_norm, d, tmp, nm("self_attn.k_norm.weight").c_str()));
    }
    cudaStreamSynchronize(e->stream);
    LW(dev_alloc(e, &L.o, (size_t)H * Hq * d));
    LW(copy_bf16(e, wm.get(nm("self_attn.o_proj.weight")), tmp, (int64_t)H * Hq * d, nm("self_attn.o_proj.weight").c_str()));
    if (launch_pack(tmp, L.o, H, Hq * d, 0, e->stream) != cudaSuccess) return done(fail(e, ENG_ECUDA, "pack launch"));
    LW(keep_row_major(e, e->g_o, tmp, &L.o_rm, &L.m_o, H, Hq * d, 0));
    cudaStreamSynchronize(e->stream);
    // fused gate|up, interleaved per 16-row tile for the SiLU epilogue
    LW(dev_alloc(e, &L.gu, (size_t)2 * I * H));
    LW(copy_bf16(e, wm.get(nm("mlp.gate_proj.weight")), tmp, (int64_t)I * H, nm("mlp.gate_proj.weight").c_str()));
    LW(copy_bf16(e, wm.get(nm("mlp.up_proj.weight")), tmp + (size_t)I * H, (int64_t)I * H, nm("mlp.up_proj.weight").c_str()));
    if (launch_pack(tmp, L.gu, 2 * I, H, I, e->stream) != cudaSuccess) return done(fail(e, ENG_ECUDA, "pack launch"));
    LW(keep_row_major(e, e->g_gu, tmp, &L.gu_rm, &L.m_gu, 2 * I, H, I));
    cudaStreamSynchronize(e->stream);
    LW(dev_alloc(e, &L.down, (size_t)H * I));
    LW(copy_bf16(e, wm.get(nm("mlp.down_proj.weight")), tmp, (int64_t)H * I, nm("mlp.down_proj.weight").c_str()));
    if (launch_pack(tmp, L.down, H, I, 0, e->stream) != cudaSuccess) return done(fail(e, ENG_ECUDA, "pack launch"));
    LW(keep_row_major(e, e->g_down, tmp, &L.down_rm, &L.m_down, H, I, 0));
    LW(dev_alloc(e, &L.in_norm, H));
    LW(dev_alloc(e, &L.post_norm, H));
    cudaStreamSynchronize(e->stream);
    LW(load_f32(e, wm.get(nm("input_layernorm.weight")), L.in_norm, H, tmp, nm("input_layernorm.weight").c_str()));
    cudaStreamSynchronize(e->stream);
    LW(load_f32(e, wm.get(nm("post_attention_layernorm.weight")), L.post_norm, H, tmp,
                nm("post_attention_layernorm.weight").c_str()));
  }
#undef LW
  if (cudaStreamSynchronize(e->stream) != cudaSuccess) return done(fail(e, ENG_ECUDA, "weight load failed"));
  return done(ENG_OK);
}

// ------------------------------------------------------------------ buffers

static int setup_buffers(eng_t* e) {
  const eng_config_t& c = e->c;
  const int Tm = c.max_tokens, Rm = c.max_reqs, H = c.hidden, d = c.head_dim;
  const int QKV = (c.q_heads + 2 * c.kv_heads) * d;

  // RoPE table in float64, stored as float32: angle = pos * theta^(-2i/d)
  e->max_pos = c.max_blocks_per_seq * 16;
  {
    std::vector<float> tab((size_t)e->max_pos * d);
    for (int pos = 0; pos < e->max_pos; ++pos)
      for (int i = 0; i < d / 2; ++i) {
        const double inv = std::pow(c.rope_theta, -2.0 * i / d);
        const double ang = (double)pos * inv;
        tab[((size_t)pos * (d / 2) + i) * 2] = (float)std::cos(ang);
        tab[((size_t)pos * (d / 2) + i) * 2 + 1] = (float)std::sin(ang);
      }
    TRY(dev_alloc(e, &e->rope, tab.size()));
    CUDA_OR_FAIL(e, cudaMemcpy(e->rope, tab.data(), tab.size() * 4, cudaMemcpyHostToDevice));
  }

  e->kv_elems = (size_t)c.layers * 2 * (size_t)(c.num_blocks + 1) * c.kv_heads * 16 * d;
  TRY(dev_alloc(e, &e->kv, e->kv_elems));

  // input layout (int32 words); block tables last so a step copies only the rows it uses
  e->max_items = Tm / 64 + Rm + 1;
  InLayout& L = e->in;
  size_t o = 0;
  L.ids = o; o += Tm;
  L.pos = o; o += Tm;
  L.prev = o; o += Tm;
  L.tok2req = o; o += Tm;
  L.cu = o; o += Rm + 1;
  L.seq = o; o += Rm;
  L.last = o; o += Rm;
  L.invt = o; o += Rm;
  L.topk = o; o += Rm;
  L.punit = o; o += Rm;
  L.rng = o; o += 4;
  L.wlog = o; o += 1;
  L.wkey = o; o += 1;
  L.step = o; o += 2;
  o = (o + 3) & ~(size_t)3;
  L.items = o; o += (size_t)4 * e->max_items;
  L.bt = o; o += (size_t)Rm * c.max_blocks_per_seq;
  L.words = o;
  TRY(dev_alloc(e, &e->d_in, L.words));
  for (int i = 0; i < kSlots; ++i) {
    void* hp = nullptr;
    if (cudaMallocHost(&hp, L.words * 4) != cudaSuccess) return fail(e, ENG_ENOMEM, "cudaMallocHost failed");
    memset(hp, 0, L.words * 4);
    e->h_in[i] = static_cast<int*>(hp);
    CUDA_OR_FAIL(e, cudaEventCreateWithFlags(&e->ev[i], cudaEventDisableTiming));
  }

  TRY(dev_alloc(e, &e->h, (size_t)Tm * H));
  TRY(dev_alloc(e, &e->q, (size_t)Tm * c.q_heads * d));
  TRY(dev_alloc(e, &e->xn_h, (size_t)Tm * H));
  TRY(dev_alloc(e, &e->xn_l, (size_t)Tm * H));
  TRY(dev_alloc(e, &e->attn_h, (size_t)Tm * c.q_heads * d));
  TRY(dev_alloc(e, &e->attn_l, (size_t)Tm * c.q_heads * d));
  TRY(dev_alloc(e, &e->act_h, (size_t)Tm * c.intermediate));
  TRY(dev_alloc(e, &e->act_l, (size_t)Tm * c.intermediate));
  TRY(dev_alloc(e, &e->logits, (size_t)Rm * c.vocab));
  TRY(dev_alloc(e, &e->ids, Rm));
  TRY(dev_alloc(e, &e->slots, Tm));
  TRY(dev_alloc(e, &e->best, Rm));
  if (c.sampling_filters) {
    TRY(dev_alloc(e, &e->keys, (size_t)Rm * c.vocab));
    TRY(dev_alloc(e, &e->row_ext, (size_t)Rm * 2));
  }
  TRY(dev_alloc(e, &e->done_counter, 4));
  TRY(dev_alloc(e, &e->status, 4));
  TRY(dev_alloc(e, &e->ring, (size_t)e->ring_cap * Rm));

  auto site = [&](GemmSite& s, int N, int K, int rg_fixed, int /*T*/) -> int {
    s.N = N;
    s.K = K;
    s.rg_fixed = rg_fixed;
    s.tc = N % 128 == 0 && K % 64 == 0 && (rg_fixed == 0 || 128 % (16 * rg_fixed) == 0);
    if (s.tc) {  // K splits for about one CTA per SM, dividing the k-blocks of 64
      const int tiles = N / 128, nkb = K / 64;
      int sp = std::min(8, std::max(1, (e->sms + tiles / 2) / tiles));
      while (sp > 1 && (nkb % sp != 0 || sp > nkb || !tc_split_fits(sp))) --sp;
      s.tc_S = sp;
    }
    gemm_plan(N, K, rg_fixed, e->sms, &s.plan[0].RG, &s.plan[0].S, &s.plan[0].ktn);
    gemm_plan_large(N, K, rg_fixed, e->sms, &s.plan[1].RG, &s.plan[1].S, &s.plan[1].ktn);
    // mid-sized steps take the tensor cores where the warp-MMA plan's weight slice is too large to stage
    s.tc_mid = s.tc && !gemm_slice_fits(s.plan[1].RG, s.plan[1].ktn);
    return ENG_OK;
  };
  TRY(site(e->g_qkv, QKV, H, d / 16, Tm));  // a CTA owns one whole head (QK-norm and RoPE in the epilogue)
  TRY(site(e->g_o, H, c.q_heads * d, 0, Tm));
  TRY(site(e->g_gu, 2 * c.intermediate, H, 0, Tm));
  TRY(site(e->g_down, H, c.intermediate, 0, Tm));
  TRY(site(e->g_lm, c.vocab, H, 0, Rm));
  e->g_lm.tc = false;  // the LM head gathers its rows and samples: warp-MMA path only
  // tensor maps of the activation planes (64-token boxes); without them no projection takes the TC path
  const bool maps_ok = make_tc_map(&e->m_xn_h, e->xn_h, Tm, H, 64) && make_tc_map(&e->m_xn_l, e->xn_l, Tm, H, 64) &&
                       make_tc_map(&e->m_attn_h, e->attn_h, Tm, c.q_heads * d, 64) &&
                       make_tc_map(&e->m_attn_l, e->attn_l, Tm, c.q_heads * d, 64) &&
                       make_tc_map(&e->m_act_h, e->act_h, Tm, c.intermediate, 64) &&
                       make_tc_map(&e->m_act_l, e->act_l, Tm, c.intermediate, 64);
  if (!maps_ok) e->g_qkv.tc = e->g_o.tc = e->g_gu.tc = e->g_down.tc = false;
  e->sq_stride = std::max(e->g_o.max_groups(), e->g_down.max_groups());
  TRY(dev_alloc(e, &e->sq, (size_t)Tm * e->sq_stride));

  // decode attention: each row's blocks in at most 8 splits (merged on chip for a few rows, through the
  // workspace for more rows with query groups larger than two), or the flat partition over a grid of the
  // CTAs resident at once (more rows, groups of at most two).  All fixed per engine, so eager and replayed
  // steps agree bit for bit.
  e->split_blocks = (c.max_blocks_per_seq + kAttnMaxSplits - 1) / kAttnMaxSplits;
  e->max_splits = (c.max_blocks_per_seq + e->split_blocks - 1) / e->split_blocks;
  e->attn_flat = e->f16 ? f16::attn_flat_ctas(d, Rm, e->sms) : attn_flat_ctas(d, Rm, e->sms);
  if (e->attn_flat < 1) return fail(e, ENG_ECUDA, "occupancy query of the decode attention kernel failed");
  if ((int64_t)c.kv_heads * Rm * (c.max_blocks_per_seq + 8) >= (1ll << 30))
    return fail(e, ENG_EINVAL, "kv_heads * max_reqs * max_blocks_per_seq too large for decode attention");
  // partials: the flat partition's pieces, or the splits of each (row, KV head)
  const size_t ws_slots = std::max((size_t)Rm * c.kv_heads + 4 * (size_t)e->attn_flat, (size_t)Rm * c.kv_heads * e->max_splits);
  TRY(dev_alloc(e, &e->attn_ws, ws_slots * (c.q_heads / c.kv_heads) * (d + 2)));
  TRY(dev_alloc(e, &e->attn_counters, (size_t)Rm * c.kv_heads));

  e->used.assign(c.num_blocks, 0);
  e->free_list.clear();
  for (int b = 0; b < c.num_blocks; ++b) e->free_list.push_back(b);
  return ENG_OK;
}

// ------------------------------------------------------------------ persistent decode step set-up

// Decides whether decode-only steps of a few tokens run on the persistent kernel (decode_step.cu) and
// allocates its buffers.  The kernel stages its input rows in shared memory, so the token count it takes
// is the largest power of two (at most 8) whose rows of the widest projection input fit 50 KB; it needs
// one CTA per SM, all resident together (a cooperative launch).  ENG_DECODE_KERNEL=0 in the environment when
// the engine is created keeps every step on the per-layer kernels (for comparison).
static int setup_decode_step(eng_t* e) {
  const eng_config_t& c = e->c;
  const char* v = getenv("ENG_DECODE_KERNEL");
  if (v && v[0] == '0') return ENG_OK;
  if (e->f16) return ENG_OK;  // built for bfloat16 only: fp16 models run every step on the per-layer kernels
  const int d = c.head_dim, G = c.q_heads / c.kv_heads;
  if (c.layers > 50 || G > 8 || c.kv_heads > 255 || (d != 64 && d != 128)) return ENG_OK;
  const int kx = std::max({c.hidden, c.q_heads * d, c.intermediate}) + 8;
  const size_t stage_cap = 50 * 1024;
  int rows = 8;
  while (rows > 1 && ((size_t)4 * rows * kx > stage_cap || rows > c.max_reqs)) rows >>= 1;
  if ((size_t)4 * rows * kx > stage_cap) return ENG_OK;
  int slots = 5;
  size_t smem = decode_step_smem(slots, rows, kx, d, G, c.hidden, c.layers);
  while (slots > 2 && smem > 227 * 1024) smem = decode_step_smem(--slots, rows, kx, d, G, c.hidden, c.layers);
  if (smem > 227 * 1024) return ENG_OK;
  int coop = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, e->device) != cudaSuccess || !coop) return ENG_OK;
  if (decode_step_prepare(smem, &per_sm) != cudaSuccess || per_sm < 1) {
    cudaGetLastError();
    return ENG_OK;
  }
  const uint64_t kv_rows = (uint64_t)c.layers * 2 * (c.num_blocks + 1) * c.kv_heads * 16;
  if (kv_rows >= (1ull << 31) || !make_tc_map(&e->ds_kv_map, e->kv, kv_rows, d, 16)) return ENG_OK;
  e->ds_rows = rows;
  e->ds_kx = kx;
  e->ds_slots = slots;
  e->ds_smem = smem;
  const int QKV = (c.q_heads + 2 * c.kv_heads) * d;
  TRY(dev_alloc(e, &e->ds_h, (size_t)rows * c.hidden));
  TRY(dev_alloc(e, &e->ds_qkv, (size_t)rows * QKV));
  TRY(dev_alloc(e, &e->ds_act, (size_t)rows * c.intermediate));
  TRY(dev_alloc(e, &e->ds_ws, (size_t)rows * c.kv_heads * kDsMaxSplits * G * (d + 2)));
  TRY(dev_alloc(e, &e->ds_out, (size_t)rows * c.q_heads * d));
  TRY(dev_alloc(e, &e->ds_epoch, 2));
  TRY(dev_alloc(e, &e->ds_diag, 4 + 4 * (size_t)e->sms));
  const unsigned int ep[2] = {1u, 0u};  // tags start above the zero-filled buffers' tag 0
  CUDA_OR_FAIL(e, cudaMemcpy(e->ds_epoch, ep, sizeof(ep), cudaMemcpyHostToDevice));
  TRY(dev_alloc(e, &e->ds_layers, (size_t)c.layers));
  e->ds_on = true;
  return ENG_OK;
}

// The persistent kernel's table of per-layer weight pointers (after the weights are loaded).
static int fill_decode_layers(eng_t* e) {
  if (!e->ds_on) return ENG_OK;
  std::vector<DsLayer> v(e->layers.size());
  // the kernel copies norm weights to shared memory in 16-byte pieces (each tensor is its own allocation)
  auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
  for (size_t l = 0; l < v.size(); ++l) {
    const Layer& L = e->layers[l];
    v[l] = DsLayer{L.qkv, L.o, L.gu, L.down, L.qkv_bias, L.q_norm, L.k_norm, L.in_norm, L.post_norm};
    if (!a16(L.q_norm) || !a16(L.k_norm) || !a16(L.in_norm) || !a16(L.post_norm))
      return fail(e, ENG_EINVAL, "decode step: norm weights must be 16-byte aligned");
  }
  if (!a16(e->final_norm) || !a16(e->rope)) return fail(e, ENG_EINVAL, "decode step: misaligned table");
  CUDA_OR_FAIL(e, cudaMemcpy(e->ds_layers, v.data(), v.size() * sizeof(DsLayer), cudaMemcpyHostToDevice));
  return ENG_OK;
}

// ------------------------------------------------------------------ the step's kernel sequence

// Event pair around one launch when eng_profile is collecting (no-op otherwise).
static void prof_begin(eng_t* e, cudaStream_t st, int kind, int64_t bytes) {
  if (!e->prof_on) return;
  const size_t i = e->prof_kind.size();
  if (2 * i + 2 > e->prof_ev.size()) return;
  cudaEventRecord(e->prof_ev[2 * i], st);
  e->prof_kind.push_back(kind);
  e->prof_bytes.push_back(bytes);
}
static void prof_end(eng_t* e, cudaStream_t st) {
  if (!e->prof_on || e->prof_kind.empty()) return;
  cudaEventRecord(e->prof_ev[2 * (e->prof_kind.size() - 1) + 1], st);
}

static int64_t gemm_bytes(const GemmSite& s, int T, int epi, bool norm_in) {
  (void)norm_in;
  int64_t b = (int64_t)s.N * s.K * 2;                          // weights once
  b += (int64_t)T * s.K * 4;                                    // activation planes in
  if (epi == EPI_STORE_F32) b += (int64_t)T * s.N * 4;
  if (epi == EPI_RESID) b += (int64_t)T * s.N * 12;             // residual read + write, planes out
  if (epi == EPI_SILU) b += (int64_t)T * (s.N / 2) * 4;
  if (epi == EPI_LMHEAD) b += (int64_t)T * 4;
  return b;
}

// Weights of the GEMM two launches ahead, prefetched into L2 by the current kernel when they take a small
// share of L2 (large models stream their weights straight from HBM).
static void set_prefetch(eng_t* e, const void*& ptr, unsigned long long& bytes, const bf16* w, const GemmSite& s) {
  const unsigned long long b = (unsigned long long)s.N * s.K * 2;
  if (e->l2_prefetch && b <= 24ull << 20) {
    ptr = w;
    bytes = b;
  } else {
    ptr = nullptr;
    bytes = 0;
  }
}

// Parameters shared by every GEMM launch of the engine.
static GemmParams gemm_params(eng_t* e, const GemmSite& s, const bf16* W, int T) {
  GemmParams p{};
  p.W = W;
  p.ldx = s.K;
  p.T = T;
  p.N = s.N;
  p.K = s.K;
  const GemmPlan& pl = s.for_tokens(T);
  p.RG = pl.RG;
  p.S = pl.S;
  p.kt_per_split = pl.ktn;
  if (s.use_tc(T)) {  // tensor-core path: 128-row tiles
    p.RG = 8;
    p.S = s.tc_splits(T);
    p.kt_per_split = s.K / 32 / p.S;
  }
  p.ldo = s.N;
  p.eps = e->c.rms_eps;
  p.sq_stride = e->sq_stride;
  int* in = e->d_in;
  p.logits = e->logits;
  p.write_logits = in + e->in.wlog;
  p.inv_temp = reinterpret_cast<const float*>(in + e->in.invt);
  p.rng = reinterpret_cast<const uint32_t*>(in + e->in.rng);
  p.best = e->best;
  p.done_counter = e->done_counter;
  p.out_ids = e->ids;
  p.status = e->status;
  return p;
}

// w, xh, xl: the tensor maps the tensor-core path would use (ignored when the step is too small for it).
static cudaError_t gemm_launch(eng_t* e, const GemmParams& p, const GemmSite& s, int epi, bool norm_in, int kind,
                               cudaStream_t st, const CUtensorMap* w = nullptr, const CUtensorMap* xh = nullptr,
                               const CUtensorMap* xl = nullptr) {
  LaunchOpts o;
  o.pdl = e->pdl;
  e->launches++;
  prof_begin(e, st, kind, gemm_bytes(s, p.T, epi, norm_in));
  TcMaps tm;
  const bool tc = s.use_tc(p.T) && w;
  if (tc) {
    tm.w = *w;
    tm.xh = *xh;
    tm.xl = *xl;
  }
  const cudaError_t r = e->f16 ? f16::launch_gemm(p, epi, norm_in, o, st, tc ? &tm : nullptr)
                               : launch_gemm(p, epi, norm_in, o, st, tc ? &tm : nullptr);
  prof_end(e, st);
  return r;
}

static cudaError_t enqueue_tail(eng_t* e, int T, int R, int sq_parts, bool advance, cudaStream_t st);

// True when a step runs on the persistent decode kernel: decode-only (every request one token) with at
// most ds_rows tokens.  Only the token count decides, so an eager step and its padded bucket take the same
// path whenever ds_rows is a capture size.
static bool ds_applies(const eng_t* e, int T, int R, int P) { return e->ds_on && P == 0 && T == R && T <= e->ds_rows; }

// The persistent kernel's schedule for T tokens, built on first use: every CTA's items of each phase,
// handed out largest first to the CTA with the fewest bytes so far (weights of a tile, or the K/V of a
// full attention split), so that every SM streams about the same share of the layer.
// Attention splits per (row, KV head) of a T-row step: enough items for one per SM, at most kDsMaxSplits.
// A row's last split merges the others, which it waits for; a CTA running several attention items takes
// them in item order, where a row's last split comes after the row's other splits.
static int ds_splits(const eng_t* e, int T) {
  return std::max(1, std::min(kDsMaxSplits, e->sms / (T * e->c.kv_heads)));
}

static int ds_schedule(eng_t* e, int T, int** d_off, int** d_items) {
  auto it = e->ds_sched.find(T);
  if (it != e->ds_sched.end()) {
    *d_off = it->second.first;
    *d_items = it->second.second;
    return ENG_OK;
  }
  const eng_config_t& c = e->c;
  const int grid = e->sms, d = c.head_dim;
  std::vector<std::vector<int>> lists((size_t)grid * DS_PHASES);
  std::vector<int64_t> load(grid, 0);
  auto assign = [&](int phase, int count, int64_t bytes) {
    for (int i = 0; i < count; ++i) {
      int best = 0;
      for (int k = 1; k < grid; ++k)
        if (load[k] < load[best]) best = k;
      load[best] += bytes;
      lists[(size_t)best * DS_PHASES + phase].push_back(i);
    }
  };
  const int64_t kv_item = kDsSlotBytes;  // about one ring chunk of keys per attention split
  assign(DS_DOWN, c.hidden / 16, (int64_t)c.intermediate / 32 * 1024);
  assign(DS_O, c.hidden / 16, (int64_t)c.q_heads * d / 32 * 1024);
  assign(DS_GU, 2 * c.intermediate / 16, (int64_t)c.hidden / 32 * 1024);
  assign(DS_QKV, (c.q_heads + 2 * c.kv_heads) * d / 16, (int64_t)c.hidden / 32 * 1024);
  assign(DS_ATTN, T * c.kv_heads * ds_splits(e, T), kv_item);
  // attention items as (row << 16) | (KV head << 8) | split (the kernel decodes them with shifts)
  const int ns = ds_splits(e, T);
  for (int b = 0; b < grid; ++b)
    for (int& it : lists[(size_t)b * DS_PHASES + DS_ATTN]) {
      const int sp = it % ns, rg = it / ns;
      it = ((rg / c.kv_heads) << 16) | ((rg % c.kv_heads) << 8) | sp;
    }
  std::vector<int> off((size_t)grid * (DS_PHASES + 1)), items;
  for (int b = 0; b < grid; ++b) {
    const size_t first = items.size();
    for (int ph = 0; ph < DS_PHASES; ++ph) {
      off[(size_t)b * (DS_PHASES + 1) + ph] = (int)items.size();
      auto& l = lists[(size_t)b * DS_PHASES + ph];
      std::sort(l.begin(), l.end());
      items.insert(items.end(), l.begin(), l.end());
      off[(size_t)b * (DS_PHASES + 1) + ph + 1] = (int)items.size();
    }
    if (items.size() - first > (size_t)kDsMaxItems) return fail(e, ENG_EINVAL, "decode step schedule too long");
  }
  int *o = nullptr, *itm = nullptr;
  TRY(dev_alloc(e, &o, off.size()));
  TRY(dev_alloc(e, &itm, items.size()));
  CUDA_OR_FAIL(e, cudaMemcpy(o, off.data(), off.size() * 4, cudaMemcpyHostToDevice));
  CUDA_OR_FAIL(e, cudaMemcpy(itm, items.data(), items.size() * 4, cudaMemcpyHostToDevice));
  e->ds_sched[T] = {o, itm};
  *d_off = o;
  *d_items = itm;
  return ENG_OK;
}

// Enqueues one forward over T packed tokens of R requests; requests [0, P) go to the packed prefill
// kernel (n_items work items), [P, R) to the decode kernel with `splits` splits per row.  With
// `advance`, a decode-only step ends by feeding its sampled ids back as the next inputs (advance.cu).
// Piece `piece` of a step's forward over T tokens: the projections between two attention launches.
// Piece 0 is the embedding and layer 0's input norm + QKV projection (QK-norm, RoPE, paged KV write);
// piece l (1 <= l < L) is layer l - 1's output projection, gate|up and down and layer l's QKV; piece L is
// the last layer's output projection, gate|up and down.  An eager step runs the pieces with the attention
// launches between them; piecewise graphs ("(7) Graph Mode", section PIECEWISE) record the same calls.
static cudaError_t enqueue_piece(eng_t* e, int T, int piece, cudaStream_t st) {
  const eng_config_t& c = e->c;
  const int H = c.hidden, d = c.head_dim, Hq = c.q_heads, Hkv = c.kv_heads;
  int* in = e->d_in;
  const size_t plane = (size_t)(c.num_blocks + 1) * Hkv * 16 * d;
  LaunchOpts o;
  o.pdl = e->pdl;
  cudaError_t r;
  int sq_parts = 1;  // producers of the residual's partial sums: embed (1), then o_proj / down row groups
  if (piece == 0) {
    EmbedParams ep{};
    ep.embed = e->embed;
    ep.ids = in + e->in.ids;
    ep.h_out = e->h;
    ep.sq_out = e->sq;
    ep.sq_stride = e->sq_stride;
    ep.norm_w = e->layers[0].in_norm;
    ep.prev_row = in + e->in.prev;
    ep.prev_ids = e->ids;
    ep.prev_rows = c.max_reqs;
    ep.xh_out = e->xn_h;
    ep.xl_out = e->xn_l;
    ep.rows = T;
    ep.H = H;
    ep.V = c.vocab;
    ep.status = e->status;
    e->launches++;
    prof_begin(e, st, ENG_K_EMBED_NORM, (int64_t)T * H * (2 + 4 + 4));
    r = e->f16 ? f16::launch_embed(ep, o, st) : launch_embed(ep, o, st);
    prof_end(e, st);
    if (r != cudaSuccess) return r;
  } else {
    const int l = piece - 1;
    const Layer& L = e->layers[l];
    // ---- output projection + residual (+ sums of squares for the next norm)
    GemmParams po = gemm_params(e, e->g_o, L.o, T);
    po.Xh = e->attn_h;
    po.Xl = e->attn_l;
    po.resid = e->h;
    po.sq_out = e->sq;
    po.next_norm_w = L.post_norm;
    po.xh_out = e->xn_h;
    po.xl_out = e->xn_l;
    set_prefetch(e, po.pf_ptr, po.pf_bytes, L.down, e->g_down);
    if ((r = gemm_launch(e, po, e->g_o, EPI_RESID, false, ENG_K_GEMM_O, st, &L.m_o, &e->m_attn_h, &e->m_attn_l)) !=
        cudaSuccess)
      return r;

    // ---- post-attention RMSNorm + fused gate|up projection + SiLU * up
    GemmParams pg = gemm_params(e, e->g_gu, L.gu, T);
    pg.Xh = e->xn_h;
    pg.Xl = e->xn_l;
    pg.sq_in = e->sq;
    pg.sq_parts = e->g_o.groups(T);
    pg.xh_out = e->act_h;
    pg.xl_out = e->act_l;
    if (l + 1 < c.layers) set_prefetch(e, pg.pf_ptr, pg.pf_bytes, e->layers[l + 1].qkv, e->g_qkv);
    if ((r = gemm_launch(e, pg, e->g_gu, EPI_SILU, true, ENG_K_GEMM_GATE_UP, st, &L.m_gu, &e->m_xn_h, &e->m_xn_l)) !=
        cudaSuccess)
      return r;

    // ---- down projection + residual
    GemmParams pd = gemm_params(e, e->g_down, L.down, T);
    pd.Xh = e->act_h;
    pd.Xl = e->act_l;
    pd.resid = e->h;
    pd.sq_out = e->sq;
    pd.next_norm_w = l + 1 < c.layers ? e->layers[l + 1].in_norm : e->final_norm;
    pd.xh_out = e->xn_h;
    pd.xl_out = e->xn_l;
    if ((r = gemm_launch(e, pd, e->g_down, EPI_RESID, false, ENG_K_GEMM_DOWN, st, &L.m_down, &e->m_act_h,
                         &e->m_act_l)) != cudaSuccess)
      return r;
    sq_parts = e->g_down.groups(T);
  }
  if (piece == c.layers) return cudaSuccess;

  const int l = piece;
  const Layer& L = e->layers[l];
  bf16* kplane = e->kv + (size_t)l * 2 * plane;
  bf16* vplane = kplane + plane;
  // ---- input RMSNorm + fused QKV projection + QK-norm + RoPE + paged KV write
  GemmParams q = gemm_params(e, e->g_qkv, L.qkv, T);
  q.Xh = e->xn_h;
  q.Xl = e->xn_l;
  q.sq_in = e->sq;
  q.sq_parts = sq_parts;
  q.bias = L.qkv_bias;
  q.positions = in + e->in.pos;
  q.tok2req = in + e->in.tok2req;
  q.seq_lens = in + e->in.seq;
  q.bt = in + e->in.bt;
  q.mbs = c.max_blocks_per_seq;
  q.q_norm = L.q_norm;
  q.k_norm = L.k_norm;
  q.cos_sin = e->rope;
  q.max_pos = e->max_pos;
  q.q_out = e->q;
  q.k_pool = kplane;
  q.v_pool = vplane;
  q.slots = e->slots;
  q.Hq = Hq;
  q.Hkv = Hkv;
  q.d = d;
  q.NB = c.num_blocks;
  set_prefetch(e, q.pf_ptr, q.pf_bytes, L.o, e->g_o);
  return gemm_launch(e, q, e->g_qkv, EPI_QKV_ROPE, true, ENG_K_GEMM_QKV, st, &L.m_qkv, &e->m_xn_h, &e->m_xn_l);
}

// Layer l's attention over the staged step: the packed prefill kernel for the first P requests (n_items work
// items) and the split decode kernel for requests P .. R - 1.
static cudaError_t enqueue_attention(eng_t* e, int l, int R, int P, int n_items, int splits, cudaStream_t st) {
  const eng_config_t& c = e->c;
  const int d = c.head_dim, Hq = c.q_heads, Hkv = c.kv_heads;
  int* in = e->d_in;
  const size_t plane = (size_t)(c.num_blocks + 1) * Hkv * 16 * d;
  const int64_t kv_tok = (int64_t)2 * Hkv * d * 2;  // K and V bytes of one position in one layer
  int64_t kv_read = 0;                              // decode rows' K/V bytes per layer (profiling only)
  if (e->prof_on)
    for (int v : e->dec_seq) kv_read += (int64_t)v * kv_tok;
  LaunchOpts o;
  o.pdl = e->pdl;
  cudaError_t r;
  const Layer& L = e->layers[l];
  bf16* kplane = e->kv + (size_t)l * 2 * plane;
  bf16* vplane = kplane + plane;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)d);
  if (P > 0) {
    AttnPrefillParams ap{};
    ap.q = e->q;
    ap.k_pool = kplane;
    ap.v_pool = vplane;
    ap.bt = in + e->in.bt;
    ap.mbs = c.max_blocks_per_seq;
    ap.positions = in + e->in.pos;
    ap.items = reinterpret_cast<const int4*>(in + e->in.items);
    ap.n_items = n_items;
    ap.out_h = e->attn_h;
    ap.out_l = e->attn_l;
    ap.Hq = Hq;
    ap.Hkv = Hkv;
    ap.d = d;
    ap.NB = c.num_blocks;
    ap.scale_log2 = scale_log2;
    ap.status = e->status;
    e->launches++;
    prof_begin(e, st, ENG_K_ATTN_PREFILL, 0);
    r = e->f16 ? f16::launch_attn_prefill(ap, o, st) : launch_attn_prefill(ap, o, st);
    prof_end(e, st);
    if (r != cudaSuccess) return r;
  }
  if (R > P) {
    AttnDecodeParams dp{};
    dp.q = e->q;
    dp.k_pool = kplane;
    dp.v_pool = vplane;
    dp.bt = in + e->in.bt;
    dp.mbs = c.max_blocks_per_seq;
    dp.seq_lens = in + e->in.seq;
    dp.cu = in + e->in.cu;
    dp.r0 = P;
    dp.rows = R - P;
    dp.out_h = e->attn_h;
    dp.out_l = e->attn_l;
    dp.Hq = Hq;
    dp.Hkv = Hkv;
    dp.d = d;
    dp.NB = c.num_blocks;
    dp.split_blocks = e->split_blocks;
    dp.max_splits = splits;
    dp.ws = e->attn_ws;
    dp.counters = e->attn_counters;
    dp.flat_ctas = e->attn_flat;
    dp.scale_log2 = scale_log2;
    dp.status = e->status;
    set_prefetch(e, dp.pf_ptr, dp.pf_bytes, L.gu, e->g_gu);
    e->launches++;
    prof_begin(e, st, ENG_K_ATTN_DECODE, kv_read + (int64_t)(R - P) * Hq * d * 8);
    r = e->f16 ? f16::launch_attn_decode(dp, o, st) : launch_attn_decode(dp, o, st);
    prof_end(e, st);
    if (r != cudaSuccess) return r;
  }
  return cudaSuccess;
}

static cudaError_t enqueue_forward(eng_t* e, int T, int R, int P, int n_items, int splits, bool advance,
                                   cudaStream_t st) {
  const eng_config_t& c = e->c;
  const int H = c.hidden, d = c.head_dim, Hq = c.q_heads, Hkv = c.kv_heads;
  int* in = e->d_in;
  const size_t plane = (size_t)(c.num_blocks + 1) * Hkv * 16 * d;
  const int64_t kv_tok = (int64_t)2 * Hkv * d * 2;  // K and V bytes of one position in one layer
  int64_t kv_read = 0;                              // decode rows' K/V bytes per layer (profiling only)
  if (e->prof_on)
    for (int v : e->dec_seq) kv_read += (int64_t)v * kv_tok;
  LaunchOpts o;
  o.pdl = e->pdl;
  cudaError_t r;

  if (ds_applies(e, T, R, P)) {
    int* d_off = nullptr;
    int* d_items = nullptr;
    if (ds_schedule(e, T, &d_off, &d_items) != ENG_OK) return cudaErrorInvalidValue;
    DecodeStepParams dp{};
    dp.kv_map = e->ds_kv_map;
    dp.L = c.layers;
    dp.H = H;
    dp.Hq = Hq;
    dp.Hkv = Hkv;
    dp.d = d;
    dp.I = c.intermediate;
    dp.V = c.vocab;
    dp.NB = c.num_blocks;
    dp.mbs = c.max_blocks_per_seq;
    dp.max_pos = e->max_pos;
    dp.eps = c.rms_eps;
    dp.scale_log2 = 1.4426950408889634f / sqrtf((float)d);
    dp.layers = e->ds_layers;
    dp.embed = e->embed;
    dp.final_norm = e->final_norm;
    dp.rope = e->rope;
    dp.kv = e->kv;
    dp.T = T;
    dp.ids = in + e->in.ids;
    dp.prev_row = in + e->in.prev;
    dp.prev_ids = e->ids;
    dp.prev_rows = c.max_reqs;
    dp.pos = in + e->in.pos;
    dp.seq = in + e->in.seq;
    dp.bt = in + e->in.bt;
    dp.sched_off = d_off;
    dp.sched_items = d_items;
    dp.asplits = ds_splits(e, T);
    dp.trows = e->ds_rows;
    dp.kx = e->ds_kx;
    dp.slots_n = e->ds_slots;
    dp.h_ll = e->ds_h;
    dp.qkv_ll = e->ds_qkv;
    dp.act_ll = e->ds_act;
    dp.attn_ws = e->ds_ws;
    dp.attn_out = e->ds_out;
    dp.epoch = e->ds_epoch;
    dp.xn_h = e->xn_h;
    dp.xn_l = e->xn_l;
    dp.sq = e->sq;
    dp.sq_stride = e->sq_stride;
    dp.h_out = e->h;
    dp.slots = e->slots;
    dp.status = e->status;
    dp.diag = e->ds_diag;
    dp.pf_ptr = e->lm;
    dp.pf_bytes = std::min<unsigned long long>((unsigned long long)c.vocab * H * 2, 80ull << 20);
    int64_t wbytes = 0;
    for (const GemmSite* g : {&e->g_qkv, &e->g_o, &e->g_gu, &e->g_down}) wbytes += (int64_t)g->N * g->K * 2;
    e->launches++;
    prof_begin(e, st, ENG_K_DECODE_LAYERS, wbytes * c.layers + kv_read * c.layers + (int64_t)T * kv_tok * c.layers);
    r = launch_decode_step(dp, e->sms, e->ds_smem, st);
    prof_end(e, st);
    if (r != cudaSuccess) return r;
    return enqueue_tail(e, T, R, 1, advance, st);
  }

  for (int l = 0; l <= c.layers; ++l) {
    if ((r = enqueue_piece(e, T, l, st)) != cudaSuccess) return r;
    if (l < c.layers && (r = enqueue_attention(e, l, R, P, n_items, splits, st)) != cudaSuccess) return r;
  }
  return enqueue_tail(e, T, R, e->g_down.groups(T), advance, st);
}

// The end of a step: final RMSNorm at each request's last token, LM head and sampling, the optional
// top-k / top-p redraw, and for a device-resident decode loop the in-place advance of the inputs.
static cudaError_t enqueue_tail(eng_t* e, int T, int R, int sq_parts, bool advance, cudaStream_t st) {
  (void)T;
  const eng_config_t& c = e->c;
  int* in = e->d_in;
  LaunchOpts o;
  o.pdl = e->pdl;
  cudaError_t r;
  // ---- final RMSNorm at each request's last token + LM head + sampling
  GemmParams pl = gemm_params(e, e->g_lm, e->lm, R);
  pl.Xh = e->xn_h;
  pl.Xl = e->xn_l;
  pl.sq_in = e->sq;
  pl.sq_parts = sq_parts;
  pl.x_rows = in + e->in.last;
  pl.keys_out = e->keys;  // (null unless the engine has sampling filters)
  pl.write_keys = in + e->in.wkey;
  pl.row_ext = e->row_ext;
  if ((r = gemm_launch(e, pl, e->g_lm, EPI_LMHEAD, true, ENG_K_LM_HEAD, st)) != cudaSuccess) return r;

  // ---- top-k / top-p: rows with a filter redraw from the logits the LM head wrote (the others keep the
  // fused draw); a plain launch, so it starts after the LM head has finished
  if (c.sampling_filters) {
    FilterParams fp{};
    fp.logits = e->logits;
    fp.vocab = c.vocab;
    fp.inv_temp = reinterpret_cast<const float*>(in + e->in.invt);
    fp.top_k = in + e->in.topk;
    fp.p_units = in + e->in.punit;
    fp.rng = reinterpret_cast<const uint32_t*>(in + e->in.rng);
    fp.out_ids = e->ids;
    fp.out_kept = nullptr;
    fp.status = e->status;
    fp.only_filtered = 1;
    fp.keys = e->keys;
    fp.keys_valid = in + e->in.wkey;
    fp.row_ext = e->row_ext;
    e->launches++;
    prof_begin(e, st, ENG_K_SAMPLE_FILTER, (int64_t)R * c.vocab * 4);
    r = launch_sample_filtered(fp, R, st);
    prof_end(e, st);
    if (r != cudaSuccess) return r;
  }

  if (advance) {
    AdvanceParams ad{};
    ad.sampled = e->ids;
    ad.ids = in + e->in.ids;
    ad.prev_row = in + e->in.prev;
    ad.pos = in + e->in.pos;
    ad.seq = in + e->in.seq;
    ad.rng = reinterpret_cast<uint32_t*>(in + e->in.rng);
    ad.step = in + e->in.step;
    ad.ring = e->ring;
    ad.ring_cap = e->ring_cap;
    ad.rows = R;
    ad.vocab = c.vocab;
    ad.max_pos = e->max_pos;
    ad.status = e->status;
    e->launches++;
    prof_begin(e, st, ENG_K_ADVANCE, (int64_t)R * 16);
    r = launch_advance(ad, o, st);
    prof_end(e, st);
    if (r != cudaSuccess) return r;
  }
  return cudaSuccess;
}

// ------------------------------------------------------------------ staging

static float inv_temperature(float T) { return T == 0.f ? 0.f : 1.0f / T; }

// top-p in units of 2^-24: 0 (off) unless 0 < p < 1; at least 1 unit; 2^24 units (p rounds to 1) is off.
static int top_p_units(float p) {
  if (!(p > 0.f && p < 1.f)) return 0;
  const float units = std::rint(p * 16777216.0f);  // exact scaling; rint rounds half to even
  if (units >= 16777216.0f) return 0;
  return units < 1.0f ? 1 : (int)units;
}

// Waits (rarely) for the copy that last used this staging slot, then returns it cleared.
static int* take_slot(eng_t* e, int* slot_index) {
  const int k = e->slot;
  e->slot = (e->slot + 1) % kSlots;
  cudaEventSynchronize(e->ev[k]);
  *slot_index = k;
  return e->h_in[k];
}

static int push_slot(eng_t* e, int k, size_t words) {
  CUDA_OR_FAIL(e, cudaMemcpyAsync(e->d_in, e->h_in[k], words * 4, cudaMemcpyHostToDevice, e->stream));
  CUDA_OR_FAIL(e, cudaEventRecord(e->ev[k], e->stream));
  return ENG_OK;
}

// Fills a staging slot with a decode-only batch of `size` padding rows (capture and warm-up).
static void stage_padding(eng_t* e, int* h, int size) {
  const InLayout& L = e->in;
  for (int i = 0; i < size; ++i) {
    h[L.ids + i] = 0;
    h[L.pos + i] = 0;
    h[L.prev + i] = -1;
    h[L.tok2req + i] = i;
    h[L.seq + i] = 0;
    h[L.last + i] = i;
    reinterpret_cast<float*>(h)[L.invt + i] = 0.f;
    h[L.topk + i] = 0;
    h[L.punit + i] = 0;
  }
  for (int i = 0; i <= size; ++i) h[L.cu + i] = i;
  h[L.rng + 0] = h[L.rng + 1] = h[L.rng + 2] = h[L.rng + 3] = 0;
  h[L.wlog] = 0;
  h[L.wkey] = 0;
}

// ------------------------------------------------------------------ C ABI

extern "C" {

int eng_create(const eng_config_t* cfg, const eng_tensor_t* weights, int32_t n_weights, void* cuda_stream, eng_t** out) {
  if (!out) return fail(nullptr, ENG_EINVAL, "out is NULL");
  *out = nullptr;
  if (!cfg || (!weights && n_weights > 0) || n_weights < 0) return fail(nullptr, ENG_EINVAL, "null config or weights");
  const std::string why = check_config(*cfg);
  if (!why.empty()) return fail(nullptr, ENG_EINVAL, why);
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0)
    return fail(nullptr, ENG_ECUDA, "no CUDA device: the engine has no CPU path");
  eng_t* e = new eng_t();
  e->c = *cfg;
  e->f16 = cfg->dtype == ENG_DTYPE_F16;
  {
    // programmatic dependent launch between the step's kernels (ENG_PDL=0 turns it off for comparison)
    const char* v = getenv("ENG_PDL");
    e->pdl = !(v && v[0] == '0');
    // L2 prefetch of the next GEMM's weights (ENG_L2_PREFETCH=0 turns it off for comparison)
    const char* w = getenv("ENG_L2_PREFETCH");
    e->l2_prefetch = !(w && w[0] == '0');
  }
  cudaGetDevice(&e->device);
  e->sms = device_sm_count();
  int rc = ENG_OK;
  if (e->sms < 1) rc = fail(e, ENG_ECUDA, "cannot read the device's SM count");
  if (cuda_stream) {
    e->stream = static_cast<cudaStream_t>(cuda_stream);
  } else {
    if (cudaStreamCreateWithFlags(&e->stream, cudaStreamNonBlocking) != cudaSuccess) rc = ENG_ECUDA;
    e->own_stream = true;
  }
  if (rc == ENG_OK && cudaStreamCreateWithFlags(&e->cap_stream, cudaStreamNonBlocking) != cudaSuccess) rc = ENG_ECUDA;
  if (rc == ENG_OK) rc = setup_buffers(e);
  if (rc == ENG_OK) rc = setup_decode_step(e);
  if (rc == ENG_OK) rc = load_weights(e, weights, n_weights);
  if (rc == ENG_OK) rc = fill_decode_layers(e);
  if (rc == ENG_OK && cudaDeviceSynchronize() != cudaSuccess) rc = fail(e, ENG_ECUDA, "device error after load");
  if (rc != ENG_OK) {
    g_create_error = e->err.empty() ? g_create_error : e->err;
    eng_destroy(e);
    return rc;
  }
  *out = e;
  return ENG_OK;
}

void eng_destroy(eng_t* e) {
  if (!e) return;
  if (e->stream) cudaStreamSynchronize(e->stream);
  for (auto& kv : e->graphs) cudaGraphExecDestroy(kv.second);
  for (auto& kv : e->pieces)
    for (cudaGraphExec_t g : kv.second) cudaGraphExecDestroy(g);
  for (cudaEvent_t ev : e->prof_ev) cudaEventDestroy(ev);
  for (int i = 0; i < kSlots; ++i) {
    if (e->ev[i]) cudaEventDestroy(e->ev[i]);
    if (e->h_in[i]) cudaFreeHost(e->h_in[i]);
  }
  for (void* p : e->allocations) cudaFree(p);
  if (e->cap_stream) cudaStreamDestroy(e->cap_stream);
  if (e->own_stream && e->stream) cudaStreamDestroy(e->stream);
  delete e;
}

const char* eng_last_error(const eng_t* e) { return e ? e->err.c_str() : g_create_error.c_str(); }

void* eng_stream(const eng_t* e) { return e ? static_cast<void*>(e->stream) : nullptr; }

int eng_set_eager(eng_t* e, int32_t eager) {
  if (!e) return ENG_EINVAL;
  e->eager_only = eager != 0;
  return ENG_OK;
}

int eng_kv_pool(eng_t* e, void** dev_ptr, int64_t* bytes) {
  if (!e || !dev_ptr || !bytes) return ENG_EINVAL;
  *dev_ptr = e->kv;
  *bytes = (int64_t)e->kv_elems * 2;
  return ENG_OK;
}

int eng_debug_buffer(eng_t* e, const char* name, void** dev_ptr, int64_t* bytes) {
  if (!e || !name || !dev_ptr || !bytes) return ENG_EINVAL;
  const eng_config_t& c = e->c;
  const std::string n(name);
  if (n == "hidden") {
    *dev_ptr = e->h;
    *bytes = (int64_t)c.max_tokens * c.hidden * 4;
  } else if (n == "slots") {
    *dev_ptr = e->slots;
    *bytes = (int64_t)c.max_tokens * 4;
  } else if (n == "logits") {
    *dev_ptr = e->logits;
    *bytes = (int64_t)c.max_reqs * c.vocab * 4;
  } else if (n == "decode_diag") {
    if (!e->ds_diag) return fail(e, ENG_EINVAL, "the engine has no persistent decode kernel");
    *dev_ptr = e->ds_diag;
    *bytes = 16 + 16 * (int64_t)e->sms;
  } else if (n == "ids") {
    *dev_ptr = e->ids;
    *bytes = (int64_t)c.max_reqs * 4;
  } else {
    return fail(e, ENG_EINVAL, "unknown debug buffer " + n);
  }
  return ENG_OK;
}

int eng_status(eng_t* e, int32_t reset) {
  if (!e) return ENG_EINVAL;
  CUDA_OR_FAIL(e, cudaStreamSynchronize(e->stream));
  int st = 0;
  CUDA_OR_FAIL(e, cudaMemcpy(&st, e->status, 4, cudaMemcpyDeviceToHost));
  if (reset) CUDA_OR_FAIL(e, cudaMemset(e->status, 0, 4));
  return st;
}

int eng_pool_alloc(eng_t* e, int32_t n, int32_t* out_ids) {
  if (!e || n < 0 || (n > 0 && !out_ids)) return e ? fail(e, ENG_EINVAL, "bad pool_alloc arguments") : ENG_EINVAL;
  if ((size_t)n > e->free_list.size())
    return fail(e, ENG_EPOOL, "KV pool exhausted: " + std::to_string(n) + " blocks requested, " +
                                  std::to_string(e->free_list.size()) + " free");
  for (int i = 0; i < n; ++i) {
    const int b = e->free_list.front();
    e->free_list.pop_front();
    e->used[b] = 1;
    out_ids[i] = b;
  }
  return ENG_OK;
}

int eng_pool_free(eng_t* e, const int32_t* ids, int32_t n) {
  if (!e || n < 0 || (n > 0 && !ids)) return e ? fail(e, ENG_EINVAL, "bad pool_free arguments") : ENG_EINVAL;
  std::vector<uint8_t> seen(e->c.num_blocks, 0);
  for (int i = 0; i < n; ++i) {
    const int b = ids[i];
    if (b < 0 || b >= e->c.num_blocks || !e->used[b] || seen[b])
      return fail(e, ENG_EINVAL, "block " + std::to_string(b) + " is not allocated");
    seen[b] = 1;
  }
  for (int i = 0; i < n; ++i) {
    e->used[ids[i]] = 0;
    e->free_list.push_back(ids[i]);
  }
  return ENG_OK;
}

int32_t eng_pool_free_count(const eng_t* e) { return e ? (int32_t)e->free_list.size() : 0; }

int eng_last_step_info(const eng_t* e, eng_step_info_t* info) {
  if (!e || !info) return ENG_EINVAL;
  *info = e->last;
  return ENG_OK;
}

int eng_capture(eng_t* e, const int32_t* sizes, int32_t n) {
  if (!e || !sizes || n < 1) return e ? fail(e, ENG_EINVAL, "bad capture sizes") : ENG_EINVAL;
  std::vector<int> v(sizes, sizes + n);
  std::sort(v.begin(), v.end());
  for (size_t i = 0; i < v.size(); ++i) {
    if (v[i] < 1 || v[i] > e->c.max_reqs) return fail(e, ENG_EINVAL, "capture size outside [1, max_reqs]");
    if (i && v[i] == v[i - 1]) return fail(e, ENG_EINVAL, "duplicate capture size");
  }
  CUDA_OR_FAIL(e, cudaStreamSynchronize(e->stream));
  e->prev_rows = 0;  // the warm-ups below overwrite the sampled ids: nothing to gather from afterwards
  for (auto it = v.rbegin(); it != v.rend(); ++it) {  // largest first
    const int size = *it;
    if (e->graphs.count(size)) {
      cudaGraphExecDestroy(e->graphs[size]);
      e->graphs.erase(size);
    }
    int k;
    int* h = take_slot(e, &k);
    stage_padding(e, h, size);
    TRY(push_slot(e, k, e->in.words));
    // warm up on the engine stream (lazy attribute setup, first-touch), then record on a side stream
    for (int w = 0; w < 2; ++w) {
      e->launches = 0;
      CUDA_OR_FAIL(e, enqueue_forward(e, size, size, 0, 0, e->max_splits, true, e->stream));
    }
    CUDA_OR_FAIL(e, cudaStreamSynchronize(e->stream));
    cudaGraph_t graph = nullptr;
    CUDA_OR_FAIL(e, cudaStreamBeginCapture(e->cap_stream, cudaStreamCaptureModeThreadLocal));
    e->launches = 0;
    const cudaError_t le = enqueue_forward(e, size, size, 0, 0, e->max_splits, true, e->cap_stream);
    const cudaError_t ce = cudaStreamEndCapture(e->cap_stream, &graph);
    if (le != cudaSuccess || ce != cudaSuccess) {
      if (graph) cudaGraphDestroy(graph);
      return fail(e, ENG_ECUDA, std::string("graph capture failed: ") + cudaGetErrorString(le != cudaSuccess ? le : ce));
    }
    cudaGraphExec_t exec = nullptr;
    const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ie != cudaSuccess) return fail(e, ENG_ECUDA, std::string("graph instantiate failed: ") + cudaGetErrorString(ie));
    e->graphs[size] = exec;
    e->graph_launches[size] = e->launches;
  }
  CUDA_OR_FAIL(e, cudaStreamSynchronize(e->stream));
  return ENG_OK;
}

int eng_capture_mixed(eng_t* e, const int32_t* token_buckets, int32_t n) {
  if (!e || !token_buckets || n < 1) return e ? fail(e, ENG_EINVAL, "bad mixed capture sizes") : ENG_EINVAL;
  std::vector<int> v(token_buckets, token_buckets + n);
  std::sort(v.begin(), v.end());
  for (size_t i = 0; i < v.size(); ++i) {
    if (v[i] < kTcPrefillTokens || v[i] > e->c.max_tokens)
      return fail(e, ENG_EINVAL, "mixed capture size outside [" + std::to_string(kTcPrefillTokens) + ", max_tokens]");
    if (i && v[i] == v[i - 1]) return fail(e, ENG_EINVAL, "duplicate mixed capture size");
  }
  CUDA_OR_FAIL(e, cudaStreamSynchronize(e->stream));
  const int L = e->c.layers;
  for (int size : v) {
    auto old = e->pieces.find(size);
    if (old != e->pieces.end()) {
      for (cudaGraphExec_t g : old->second) cudaGraphExecDestroy(g);
      e->pieces.erase(old);
    }
    // every token a padding token of request 0 (length 0: its K/V go to the scratch block)
    int k;
    int* h = take_slot(e, &k);
    stage_padding(e, h, 1);
    for (int t = 0; t < size; ++t) {
      h[e->in.ids + t] = 0;
      h[e->in.pos + t] = 0;
      h[e->in.prev + t] = -1;
      h[e->in.tok2req + t] = 0;
    }
    TRY(push_slot(e, k, e->in.words));
    for (int w = 0; w < 2; ++w)  // warm-up (lazy attribute setup, first touch)
      for (int p = 0; p <= L; ++p) CUDA_OR_FAIL(e, enqueue_piece(e, size, p, e->stream));
    CUDA_OR_FAIL(e, cudaStreamSynchronize(e->stream));
    std::vector<cudaGraphExec_t> execs;
    int launches = 0;
    for (int p = 0; p <= L; ++p) {
      cudaGraph_t graph = nullptr;
      CUDA_OR_FAIL(e, cudaStreamBeginCapture(e->cap_stream, cudaStreamCaptureModeThreadLocal));
      e->launches = 0;
      const cudaError_t le = enqueue_piece(e, size, p, e->cap_stream);
      const cudaError_t ce = cudaStreamEndCapture(e->cap_stream, &graph);
      cudaGraphExec_t exec = nullptr;
      const cudaError_t ie = le == cudaSuccess && ce == cudaSuccess ? cudaGraphInstantiate(&exec, graph, 0) : le;
      if (graph) cudaGraphDestroy(graph);
      if (le != cudaSuccess || ce != cudaSuccess || ie != cudaSuccess) {
        for (cudaGraphExec_t g : execs) cudaGraphExecDestroy(g);
        return fail(e, ENG_ECUDA, std::string("piecewise capture failed: ") +
                                      cudaGetErrorString(le != cudaSuccess ? le : ce != cudaSuccess ? ce : ie));
      }
      execs.push_back(exec);
      launches += e->launches;
    }
    e->pieces[size] = execs;
    e->piece_launches[size] = launches;
  }
  CUDA_OR_FAIL(e, cudaStreamSynchronize(e->stream));
  return ENG_OK;
}

static int step_impl(eng_t* e, const eng_step_t* s, const int32_t* prev_row, int32_t* out_ids_dev,
                     float* out_logits_dev) {
  if (!e) return ENG_EINVAL;
  if (!s || !out_ids_dev) return fail(e, ENG_EINVAL, "null step or out_ids");
  const eng_config_t& c = e->c;
  const int T = s->num_tokens, R = s->num_reqs, bs = s->bt_stride;
  if (R < 1 || R > c.max_reqs) return fail(e, ENG_EINVAL, "num_reqs outside [1, max_reqs]");
  if (T < R || T > c.max_tokens) return fail(e, ENG_EINVAL, "num_tokens outside [num_reqs, max_tokens]");
  if (bs < 1 || bs > c.max_blocks_per_seq) return fail(e, ENG_EINVAL, "bt_stride outside [1, max_blocks_per_seq]");
  if (!s->token_ids || !s->positions || !s->cu_seqlens || !s->block_tables || !s->seq_lens || !s->temperature)
    return fail(e, ENG_EINVAL, "null step array");
  const int32_t* cu = s->cu_seqlens;
  if (cu[0] != 0 || cu[R] != T) return fail(e, ENG_EINVAL, "cu_seqlens must start at 0 and end at num_tokens");
  int P = 0;
  bool seen_decode = false, any_filter = false, need_keys = false;
  for (int r = 0; r < R; ++r) {
    const int ql = cu[r + 1] - cu[r];
    if (ql < 1) return fail(e, ENG_EINVAL, "every request needs at least one token");
    if (ql > 1) {
      if (seen_decode) return fail(e, ENG_EINVAL, "multi-token (prefill) requests must precede single-token ones");
      P = r + 1;
    } else {
      seen_decode = true;
    }
    const int sl = s->seq_lens[r];
    if (sl < ql) return fail(e, ENG_EINVAL, "seq_len smaller than the request's token count");
    if (sl > c.max_blocks_per_seq * 16)
      return fail(e, ENG_ECAPACITY, "sequence of " + std::to_string(sl) + " positions exceeds the engine capacity of " +
                                        std::to_string(c.max_blocks_per_seq * 16));
    if ((sl + 15) / 16 > bs) return fail(e, ENG_EINVAL, "block table row shorter than the sequence");
    for (int i = 0; i < ql; ++i) {
      if (s->positions[cu[r] + i] != sl - ql + i)
        return fail(e, ENG_EINVAL, "positions of a request must be consecutive and end at seq_len - 1");
      const int src = prev_row ? prev_row[cu[r] + i] : -1;
      if (src < -1 || src >= e->prev_rows)
        return fail(e, ENG_EINVAL, "prev_row entry outside [-1, num_reqs of the previous step)");
      const int id = s->token_ids[cu[r] + i];
      if (src < 0 && (id < 0 || id >= c.vocab)) return fail(e, ENG_EINVAL, "token id outside [0, vocab)");
    }
    for (int b = 0; b < (sl + 15) / 16; ++b) {
      const int blk = s->block_tables[(size_t)r * bs + b];
      if (blk < 0 || blk >= c.num_blocks) return fail(e, ENG_EINVAL, "block id outside [0, num_blocks)");
    }
    const float tp = s->temperature[r];
    if (!(tp >= 0.f) || !std::isfinite(tp)) return fail(e, ENG_EINVAL, "temperature must be finite and >= 0");
    if (s->top_p && !std::isfinite(s->top_p[r])) return fail(e, ENG_EINVAL, "top_p must be finite");
    const bool filtered = (s->top_k && s->top_k[r] > 0 && s->top_k[r] < c.vocab) ||
                          (s->top_p && top_p_units(s->top_p[r]) > 0);
    if (filtered && !c.sampling_filters)
      return fail(e, ENG_EINVAL, "top_k / top_p need an engine created with sampling_filters = 1");
    any_filter = any_filter || filtered;
    // rows whose draw may run over the whole row: the LM head then stores every key for the filter kernel
    const int tk = s->top_k ? s->top_k[r] : 0;
    if (s->top_p && top_p_units(s->top_p[r]) > 0 && (tk <= 0 || tk > kFilterGatherCap)) need_keys = true;
  }

  const bool decode_only = (T == R);
  int bucket = 0;
  if (decode_only && !e->eager_only) {
    for (auto& kv : e->graphs)
      if (kv.first >= R) {
        bucket = kv.first;
        break;
      }
  }
  const bool replay = bucket > 0;
  const int rows = replay ? bucket : R;  // rows staged (padding included)
  // a mixed (or prefill) step of at least kTcPrefillTokens tokens replays the projection pieces of the smallest
  // captured token bucket that holds it (same token class, so the same kernels and summation orders as the
  // eager step); its padding tokens belong to request R, of length 0, so a free request row is needed
  int tbucket = 0;
  if (!decode_only && !e->eager_only && T >= kTcPrefillTokens && R < c.max_reqs) {
    for (auto& kv : e->pieces)
      if (kv.first >= T) {
        tbucket = kv.first;
        break;
      }
  }

  int k;
  int* h = take_slot(e, &k);
  const InLayout& L = e->in;
  float* hf = reinterpret_cast<float*>(h);
  for (int t = 0; t < T; ++t) {
    const int src = prev_row ? prev_row[t] : -1;
    h[L.ids + t] = src < 0 ? s->token_ids[t] : 0;
    h[L.pos + t] = s->positions[t];
    h[L.prev + t] = src;
  }
  for (int r = 0; r < R; ++r) {
    for (int t = cu[r]; t < cu[r + 1]; ++t) h[L.tok2req + t] = r;
    h[L.cu + r] = cu[r];
    h[L.seq + r] = s->seq_lens[r];
    h[L.last + r] = cu[r + 1] - 1;
    hf[L.invt + r] = inv_temperature(s->temperature[r]);
    h[L.topk + r] = s->top_k ? s->top_k[r] : 0;
    h[L.punit + r] = s->top_p ? top_p_units(s->top_p[r]) : 0;
    int* row = h + L.bt + (size_t)r * c.max_blocks_per_seq;
    memcpy(row, s->block_tables + (size_t)r * bs, (size_t)bs * 4);
    if (bs < c.max_blocks_per_seq) memset(row + bs, 0, (size_t)(c.max_blocks_per_seq - bs) * 4);
  }
  h[L.cu + R] = T;
  if (tbucket) {  // token-bucket padding: token 0 at position 0 of request R, of length 0
    for (int t = T; t < tbucket; ++t) {
      h[L.ids + t] = 0;
      h[L.pos + t] = 0;
      h[L.prev + t] = -1;
      h[L.tok2req + t] = R;
    }
    h[L.seq + R] = 0;
  }
  for (int r = R; r < rows; ++r) {  // bucket padding: token 0, position 0, length 0
    h[L.ids + r] = 0;
    h[L.pos + r] = 0;
    h[L.prev + r] = -1;
    h[L.tok2req + r] = r;
    h[L.cu + r + 1] = r + 1;
    h[L.seq + r] = 0;
    h[L.last + r] = r;
    hf[L.invt + r] = 0.f;
    h[L.topk + r] = 0;
    h[L.punit + r] = 0;
  }
  h[L.rng + 0] = (int)(uint32_t)s->seed;
  h[L.rng + 1] = (int)(uint32_t)(s->seed >> 32);
  h[L.rng + 2] = (int)(uint32_t)s->offset;
  h[L.rng + 3] = (int)(uint32_t)(s->offset >> 32);
  h[L.wlog] = (out_logits_dev || any_filter) ? 1 : 0;  // the filter kernel reads the logits
  h[L.wkey] = need_keys ? 1 : 0;

  // prefill work items: (request, first token, count <= 64)
  int n_items = 0;
  for (int r = 0; r < P; ++r)
    for (int t0 = cu[r]; t0 < cu[r + 1]; t0 += 64) {
      int* it = h + L.items + 4 * n_items;
      it[0] = r;
      it[1] = t0;
      it[2] = std::min(64, cu[r + 1] - t0);
      it[3] = 0;
      ++n_items;
    }
  if (n_items > e->max_items) return fail(e, ENG_EINVAL, "too many prefill work items");

  const size_t words = L.bt + (size_t)R * c.max_blocks_per_seq;
  TRY(push_slot(e, k, words));

  e->launches = 0;
  if (replay) {
    CUDA_OR_FAIL(e, cudaGraphLaunch(e->graphs[bucket], e->stream));
    e->launches = e->graph_launches[bucket];
  } else if (tbucket) {
    int max_blocks = 1;
    for (int r = P; r < R; ++r) max_blocks = std::max(max_blocks, (s->seq_lens[r] + 15) / 16);
    const int splits = (max_blocks + e->split_blocks - 1) / e->split_blocks;
    const std::vector<cudaGraphExec_t>& pc = e->pieces[tbucket];
    for (int l = 0; l <= c.layers; ++l) {
      CUDA_OR_FAIL(e, cudaGraphLaunch(pc[l], e->stream));
      if (l < c.layers) CUDA_OR_FAIL(e, enqueue_attention(e, l, R, P, n_items, splits, e->stream));
    }
    CUDA_OR_FAIL(e, enqueue_tail(e, tbucket, R, e->g_down.groups(tbucket), false, e->stream));
    e->launches += e->piece_launches[tbucket];
  } else {
    int max_blocks = 1;
    for (int r = P; r < R; ++r) max_blocks = std::max(max_blocks, (s->seq_lens[r] + 15) / 16);
    const int splits = (max_blocks + e->split_blocks - 1) / e->split_blocks;
    CUDA_OR_FAIL(e, enqueue_forward(e, T, R, P, n_items, splits, decode_only, e->stream));
  }
  CUDA_OR_FAIL(e, cudaMemcpyAsync(out_ids_dev, e->ids, (size_t)R * 4, cudaMemcpyDeviceToDevice, e->stream));
  if (out_logits_dev)
    CUDA_OR_FAIL(e, cudaMemcpyAsync(out_logits_dev, e->logits, (size_t)R * c.vocab * 4, cudaMemcpyDeviceToDevice,
                                    e->stream));
  e->last.replayed = replay ? 1 : tbucket ? 2 : 0;
  e->last.bucket = tbucket ? tbucket : rows;
  e->last.launches = e->launches;
  e->last.num_prefill = P;
  e->last.h2d_bytes = (int64_t)words * 4;
  // the device inputs now hold the next decode step of this batch (advanced in place)
  if (decode_only) {
    e->dec_R = R;
    e->dec_rows = rows;
    e->dec_bt_stride = bs;
    e->dec_seq.assign(s->seq_lens, s->seq_lens + R);
    for (int& v : e->dec_seq) v += 1;
  } else {
    e->dec_R = 0;
  }
  e->prev_rows = R;
  return ENG_OK;
}

int eng_step(eng_t* e, const eng_step_t* s, int32_t* out_ids_dev, float* out_logits_dev) {
  return step_impl(e, s, nullptr, out_ids_dev, out_logits_dev);
}

int eng_step_async(eng_t* e, const eng_step_t* s, const int32_t* prev_row, int32_t* out_ids_dev,
                   float* out_logits_dev) {
  if (e && !prev_row) return fail(e, ENG_EINVAL, "null prev_row");
  return step_impl(e, s, prev_row, out_ids_dev, out_logits_dev);
}

static int decode_capacity_check(eng_t* e, int n) {
  if (e->dec_R == 0) return fail(e, ENG_ESTATE, "no decode batch to continue: the last eng_step was not decode-only");
  int mx = 0;
  for (int v : e->dec_seq) mx = std::max(mx, v);
  const int limit = std::min(e->dec_bt_stride, e->c.max_blocks_per_seq) * 16;
  if (mx + n - 1 > limit)
    return fail(e, ENG_ECAPACITY, "decoding " + std::to_string(n) + " more steps needs " + std::to_string(mx + n - 1) +
                                      " positions; the block tables hold " + std::to_string(limit));
  return ENG_OK;
}

int eng_decode(eng_t* e, int32_t n_steps, int32_t* out_ids_dev) {
  if (!e) return ENG_EINVAL;
  if (n_steps < 0 || (n_steps > 0 && !out_ids_dev)) return fail(e, ENG_EINVAL, "bad eng_decode arguments");
  if (n_steps == 0) return ENG_OK;
  TRY(decode_capacity_check(e, n_steps));
  const int R = e->dec_R, rows = e->dec_rows;
  auto it = e->graphs.find(rows);
  const bool replay = !e->eager_only && it != e->graphs.end();
  int* step_word = e->d_in + e->in.step;
  int done = 0;
  while (done < n_steps) {
    const int chunk = std::min(n_steps - done, e->ring_cap);
    CUDA_OR_FAIL(e, cudaMemsetAsync(step_word, 0, 4, e->stream));
    for (int i = 0; i < chunk; ++i) {
      if (replay) {
        CUDA_OR_FAIL(e, cudaGraphLaunch(it->second, e->stream));
      } else {
        e->launches = 0;
        CUDA_OR_FAIL(e, enqueue_forward(e, rows, rows, 0, 0, e->max_splits, true, e->stream));
      }
    }
    CUDA_OR_FAIL(e, cudaMemcpy2DAsync(out_ids_dev + (size_t)done * R, (size_t)R * 4, e->ring, (size_t)rows * 4,
                                      (size_t)R * 4, chunk, cudaMemcpyDeviceToDevice, e->stream));
    done += chunk;
  }
  for (int& v : e->dec_seq) v += n_steps;
  e->last.replayed = replay ? 1 : 0;
  e->last.bucket = rows;
  e->last.launches = replay ? e->graph_launches[rows] : e->launches;
  e->last.num_prefill = 0;
  e->last.h2d_bytes = 0;
  return ENG_OK;
}

int eng_generate(eng_t* e, int32_t max_steps, int32_t check_every, const int32_t* stop_ids, int32_t n_stop,
                 int32_t* out_tokens, int32_t* out_lengths) {
  if (!e) return ENG_EINVAL;
  if (max_steps < 0 || check_every < 1 || n_stop < 0 || (n_stop > 0 && !stop_ids) ||
      (max_steps > 0 && (!out_tokens || !out_lengths)))
    return fail(e, ENG_EINVAL, "bad eng_generate arguments");
  if (e->dec_R <= 0) return fail(e, ENG_ESTATE, "no decode batch to continue (the last eng_step was not decode-only)");
  const int R = e->dec_R;
  if (max_steps == 0) return 0;
  TRY(decode_capacity_check(e, max_steps));
  std::vector<int32_t> stops(stop_ids, stop_ids + n_stop);
  std::sort(stops.begin(), stops.end());
  const int group = std::min(check_every, max_steps);
  int32_t* d_buf = nullptr;
  int32_t* h_buf = nullptr;
  if (cudaMallocAsync(reinterpret_cast<void**>(&d_buf), (size_t)group * R * 4, e->stream) != cudaSuccess)
    return fail(e, ENG_ENOMEM, "eng_generate: device buffer");
  if (cudaMallocHost(reinterpret_cast<void**>(&h_buf), (size_t)group * R * 4) != cudaSuccess) {
    cudaFreeAsync(d_buf, e->stream);
    return fail(e, ENG_ENOMEM, "eng_generate: pinned host buffer");
  }
  std::vector<int32_t> len(R, -1);  // tokens up to and including the first stop id; -1: none met yet
  int produced = 0, rc = ENG_OK;
  while (produced < max_steps) {
    const int steps = std::min(group, max_steps - produced);
    if ((rc = eng_decode(e, steps, d_buf)) != ENG_OK) break;
    // the one synchronisation of the group
    if (cudaMemcpyAsync(h_buf, d_buf, (size_t)steps * R * 4, cudaMemcpyDeviceToHost, e->stream) != cudaSuccess ||
        cudaStreamSynchronize(e->stream) != cudaSuccess) {
      rc = fail(e, ENG_ECUDA, "eng_generate: reading a group's ids");
      break;
    }
    int alive = 0;
    for (int r = 0; r < R; ++r) {
      for (int k = 0; k < steps; ++k) {
        const int32_t tok = h_buf[(size_t)k * R + r];
        out_tokens[(size_t)r * max_steps + produced + k] = tok;
        if (len[r] < 0 && std::binary_search(stops.begin(), stops.end(), tok)) len[r] = produced + k + 1;
      }
      alive += len[r] < 0;
    }
    produced += steps;
    if (alive == 0) break;
  }
  cudaFreeAsync(d_buf, e->stream);
  cudaStreamSynchronize(e->stream);  // h_buf is freed below
  cudaFreeHost(h_buf);
  if (rc != ENG_OK) return rc;
  for (int r = 0; r < R; ++r) {  // trim what follows a stop (and the steps never run)
    const int n = len[r] < 0 ? produced : len[r];
    out_lengths[r] = n;
    for (int k = n; k < max_steps; ++k) out_tokens[(size_t)r * max_steps + k] = -1;
  }
  return produced;
}

int eng_profile(eng_t* e, int32_t capacity, int32_t* kinds, float* ms, int64_t* bytes, int32_t* count) {
  if (!e) return ENG_EINVAL;
  if (capacity < 1 || !kinds || !ms || !bytes || !count) return fail(e, ENG_EINVAL, "bad eng_profile arguments");
  TRY(decode_capacity_check(e, 1));
  const int rows = e->dec_rows;
  while ((int)e->prof_ev.size() < 2 * capacity) {
    cudaEvent_t ev;
    CUDA_OR_FAIL(e, cudaEventCreate(&ev));
    e->prof_ev.push_back(ev);
  }
  e->prof_kind.clear();
  e->prof_bytes.clear();
  e->prof_on = true;
  e->launches = 0;
  // hold the stream while the host enqueues the step, so each event pair times device work only
  CUDA_OR_FAIL(e, launch_hold(20ull * 1000 * 1000, e->stream));
  const cudaError_t r = enqueue_forward(e, rows, rows, 0, 0, e->max_splits, true, e->stream);
  e->prof_on = false;
  CUDA_OR_FAIL(e, r);
  CUDA_OR_FAIL(e, cudaStreamSynchronize(e->stream));
  const int n = (int)e->prof_kind.size();
  if (n > capacity) return fail(e, ENG_EINVAL, "eng_profile capacity too small");
  for (int i = 0; i < n; ++i) {
    float t = 0.f;
    CUDA_OR_FAIL(e, cudaEventElapsedTime(&t, e->prof_ev[2 * i], e->prof_ev[2 * i + 1]));
    kinds[i] = e->prof_kind[i];
    ms[i] = t;
    bytes[i] = e->prof_bytes[i];
  }
  *count = n;
  for (int& v : e->dec_seq) v += 1;
  return ENG_OK;
}

// ------------------------------------------------------------------ standalone kernels

int eng_philox_uniforms(uint64_t seed, uint64_t offset, int32_t rows, int32_t vocab, float* out_dev, void* stream) {
  if (rows < 0 || vocab < 0 || (!out_dev && rows * (int64_t)vocab > 0)) return ENG_EINVAL;
  return launch_philox_uniforms(seed, offset, rows, vocab, out_dev, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? ENG_OK
             : ENG_ECUDA;
}

int eng_gumbel(const float* u_dev, float* g_dev, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!u_dev || !g_dev))) return ENG_EINVAL;
  return launch_gumbel(u_dev, g_dev, n, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ENG_OK : ENG_ECUDA;
}

int eng_sample(const float* logits_dev, int32_t rows, int32_t vocab, const float* temperature, uint64_t seed,
               uint64_t offset, int32_t* out_ids_dev, void* stream) {
  if (rows < 0 || vocab < 1 || (rows > 0 && (!logits_dev || !temperature || !out_ids_dev))) return ENG_EINVAL;
  if (rows == 0) return ENG_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // small per-call device block: [inv_temp rows][rng 4]
  std::vector<uint32_t> hbuf((size_t)rows + 4);
  for (int r = 0; r < rows; ++r) {
    if (!(temperature[r] >= 0.f) || !std::isfinite(temperature[r])) return ENG_EINVAL;
    const float it = inv_temperature(temperature[r]);
    memcpy(&hbuf[r], &it, 4);
  }
  hbuf[rows + 0] = (uint32_t)seed;
  hbuf[rows + 1] = (uint32_t)(seed >> 32);
  hbuf[rows + 2] = (uint32_t)offset;
  hbuf[rows + 3] = (uint32_t)(offset >> 32);
  void* d = nullptr;
  if (cudaMallocAsync(&d, hbuf.size() * 4, st) != cudaSuccess) return ENG_ENOMEM;
  int rc = ENG_OK;
  if (cudaMemcpyAsync(d, hbuf.data(), hbuf.size() * 4, cudaMemcpyHostToDevice, st) != cudaSuccess) rc = ENG_ECUDA;
  const float* it = static_cast<const float*>(d);
  const uint32_t* rng = static_cast<const uint32_t*>(d) + rows;
  if (rc == ENG_OK && launch_sample(logits_dev, rows, vocab, it, rng, nullptr, out_ids_dev, nullptr, st) != cudaSuccess)
    rc = ENG_ECUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) rc = ENG_ECUDA;  // hbuf is pageable host memory
  cudaFreeAsync(d, st);
  return rc;
}

int eng_moe_route(const void* x, const void* w_router, int32_t num_tokens, int32_t hidden, int32_t num_experts,
                  int32_t top_k, float* weights, int32_t* expert_ids, void* stream) {
  if (num_tokens < 0 || hidden < 8 || hidden % 8 || num_experts < 1 || num_experts > 4096 || top_k < 1 || top_k > 32 ||
      top_k > num_experts || (num_tokens > 0 && (!x || !w_router || !weights || !expert_ids)))
    return fail(nullptr, ENG_EINVAL, "bad eng_moe_route arguments");
  const cudaError_t r = launch_moe_route(static_cast<const bf16*>(x), static_cast<const bf16*>(w_router), num_tokens,
                                         hidden, num_experts, top_k, weights, expert_ids, static_cast<cudaStream_t>(stream));
  return r == cudaSuccess ? ENG_OK : fail(nullptr, ENG_ECUDA, std::string("eng_moe_route: ") + cudaGetErrorString(r));
}

int64_t eng_moe_padded_rows(int32_t num_tokens, int32_t top_k, int32_t num_experts, int32_t block_m) {
  if (num_tokens < 0 || top_k < 1 || num_experts < 1 || block_m < 1) return -1;
  return moe_padded_rows(num_tokens * top_k, num_experts, block_m);
}

int eng_moe_align(const int32_t* expert_ids, int32_t num_tokens, int32_t top_k, int32_t num_experts, int32_t block_m,
                  int32_t* sorted_ids, int32_t* block_expert, int32_t* info, void* stream) {
  if (num_tokens < 0 || top_k < 1 || num_experts < 1 || num_experts > 1024 || block_m < 1 || !sorted_ids ||
      !block_expert || !info || (num_tokens > 0 && !expert_ids))
    return fail(nullptr, ENG_EINVAL, "bad eng_moe_align arguments");
  const cudaError_t r = launch_moe_align(expert_ids, num_tokens * top_k, num_experts, block_m, sorted_ids, block_expert,
                                         info, static_cast<cudaStream_t>(stream));
  return r == cudaSuccess ? ENG_OK : fail(nullptr, ENG_ECUDA, std::string("eng_moe_align: ") + cudaGetErrorString(r));
}

int64_t eng_moe_workspace_bytes(int32_t num_tokens, int32_t top_k, int32_t num_experts, int32_t hidden,
                                int32_t inter) {
  if (num_tokens < 0 || top_k < 1 || num_experts < 1 || hidden < 1 || inter < 1) return -1;
  return (int64_t)moe_workspace_bytes(num_tokens, top_k, num_experts, hidden, inter);
}

int eng_moe_mlp(const void* x, const void* gate_up, const void* down, const float* weights, const int32_t* expert_ids,
                int32_t num_tokens, int32_t hidden, int32_t inter, int32_t num_experts, int32_t top_k, float* out,
                void* workspace, int64_t workspace_bytes, void* stream) {
  if (num_tokens < 0 || hidden < 64 || hidden % 64 || inter < 64 || inter % 64 || num_experts < 1 ||
      num_experts > 1024 || top_k < 1 ||
      (num_tokens > 0 && (!x || !gate_up || !down || !weights || !expert_ids || !out || !workspace)))
    return fail(nullptr, ENG_EINVAL, "bad eng_moe_mlp arguments");
  if (num_tokens > 0 && workspace_bytes < (int64_t)moe_workspace_bytes(num_tokens, top_k, num_experts, hidden, inter))
    return fail(nullptr, ENG_EINVAL, "eng_moe_mlp: workspace too small");
  const cudaError_t r = launch_moe_mlp(static_cast<const bf16*>(x), static_cast<const bf16*>(gate_up),
                                       static_cast<const bf16*>(down), weights, expert_ids, num_tokens, hidden, inter,
                                       num_experts, top_k, out, workspace, (size_t)workspace_bytes,
                                       static_cast<cudaStream_t>(stream));
  return r == cudaSuccess ? ENG_OK : fail(nullptr, ENG_ECUDA, std::string("eng_moe_mlp: ") + cudaGetErrorString(r));
}

int eng_sample_noalloc(const float* logits_dev, int32_t rows, int32_t vocab, const float* temperature,
                       uint64_t seed, uint64_t offset, int32_t* out_ids_dev, void* stream) {
  if (rows < 0 || vocab < 1 || (rows > 0 && (!logits_dev || !temperature || !out_ids_dev)))
    return fail(nullptr, ENG_EINVAL, "bad eng_sample_noalloc arguments");
  if (rows > kNoAllocMaxRows)
    return fail(nullptr, ENG_EINVAL, "eng_sample_noalloc takes at most " + std::to_string(kNoAllocMaxRows) +
                                         " rows per call (got " + std::to_string(rows) + ")");
  if (rows == 0) return ENG_OK;
  uint32_t* scratch = nullptr;
  const cudaError_t se = noalloc_scratch(&scratch);
  if (se != cudaSuccess)
    return fail(nullptr, ENG_ECUDA, std::string("cudaGetSymbolAddress of the sampler scratch failed: ") +
                                        cudaGetErrorString(se));
  std::vector<float> inv_temp((size_t)rows);  // host memory only: the staging kernel's parameters carry it
  for (int r = 0; r < rows; ++r) {
    if (!(temperature[r] >= 0.f) || !std::isfinite(temperature[r]))
      return fail(nullptr, ENG_EINVAL, "temperature must be finite and >= 0");
    inv_temp[r] = inv_temperature(temperature[r]);
  }
  const uint32_t rng[4] = {(uint32_t)seed, (uint32_t)(seed >> 32), (uint32_t)offset, (uint32_t)(offset >> 32)};
  const cudaError_t r = launch_sample_noalloc(logits_dev, rows, vocab, inv_temp.data(), rng, scratch, out_ids_dev,
                                              static_cast<cudaStream_t>(stream));
  if (r != cudaSuccess) return fail(nullptr, ENG_ECUDA, std::string("eng_sample_noalloc: ") + cudaGetErrorString(r));
  return ENG_OK;
}

int eng_sample_filtered(const float* logits_dev, int32_t rows, int32_t vocab, const float* temperature,
                        const int32_t* top_k, const float* top_p, uint64_t seed, uint64_t offset, int32_t* out_ids_dev,
                        int32_t* out_kept_dev, void* stream) {
  if (rows < 0 || vocab < 1 || (rows > 0 && (!logits_dev || !temperature || !out_ids_dev)))
    return fail(nullptr, ENG_EINVAL, "bad eng_sample_filtered arguments");
  if (rows == 0) return ENG_OK;
  // per-call device block: [inv_temp rows][top_k rows][top-p units rows][seed_lo, seed_hi, offset_lo, offset_hi]
  std::vector<uint32_t> hbuf((size_t)rows * 3 + 4);
  for (int r = 0; r < rows; ++r) {
    if (!(temperature[r] >= 0.f) || !std::isfinite(temperature[r]))
      return fail(nullptr, ENG_EINVAL, "temperature must be finite and >= 0");
    if (top_p && !std::isfinite(top_p[r])) return fail(nullptr, ENG_EINVAL, "top_p must be finite");
    const float it = inv_temperature(temperature[r]);
    memcpy(&hbuf[r], &it, 4);
    hbuf[(size_t)rows + r] = top_k ? (uint32_t)top_k[r] : 0u;
    hbuf[(size_t)rows * 2 + r] = top_p ? (uint32_t)top_p_units(top_p[r]) : 0u;
  }
  const size_t rb = (size_t)rows * 3;
  hbuf[rb + 0] = (uint32_t)seed;
  hbuf[rb + 1] = (uint32_t)(seed >> 32);
  hbuf[rb + 2] = (uint32_t)offset;
  hbuf[rb + 3] = (uint32_t)(offset >> 32);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* d = nullptr;
  if (cudaMallocAsync(&d, hbuf.size() * 4, st) != cudaSuccess) return fail(nullptr, ENG_ENOMEM, "cudaMallocAsync");
  int rc = ENG_OK;
  cudaError_t ce = cudaMemcpyAsync(d, hbuf.data(), hbuf.size() * 4, cudaMemcpyHostToDevice, st);
  if (ce == cudaSuccess) {
    const uint32_t* w = static_cast<const uint32_t*>(d);
    FilterParams fp{};
    fp.logits = logits_dev;
    fp.vocab = vocab;
    fp.inv_temp = reinterpret_cast<const float*>(w);
    fp.top_k = reinterpret_cast<const int*>(w + rows);
    fp.p_units = reinterpret_cast<const int*>(w + (size_t)rows * 2);
    fp.rng = w + rb;
    fp.out_ids = out_ids_dev;
    fp.out_kept = out_kept_dev;
    fp.status = nullptr;
    fp.only_filtered = 0;
    ce = launch_sample_filtered(fp, rows, st);
  }
  if (ce != cudaSuccess) rc = fail(nullptr, ENG_ECUDA, std::string("eng_sample_filtered: ") + cudaGetErrorString(ce));
  if (cudaStreamSynchronize(st) != cudaSuccess && rc == ENG_OK) rc = ENG_ECUDA;  // hbuf is pageable host memory
  cudaFreeAsync(d, st);
  return rc;
}

int eng_exp_f32(const float* d_dev, float* out_dev, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!d_dev || !out_dev))) return ENG_EINVAL;
  return launch_exp_rn(d_dev, out_dev, n, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ENG_OK : ENG_ECUDA;
}

}  // extern "C"
