// predictor.cu -- the masked-latent predictor of V-JEPA 2 behind the jepa_pred_* entry points of
// include/jepa.h ("GGUF schema (v1)", Predictor; the SkyVision V-JEPA 2 notes, masked-latent
// predictor). Launch sequence of one jepa_predict:
//
//   ids (checked)  ->  gather the context rows of the encoder output (bf16)
//   -> pred.embed GEMM (+bias) into rows [0, n_ctx) of each item  ->  mask token into the target rows
//   per layer: LN1 -> QKV GEMM (+bias, 3-D RoPE at the ids' positions) -> attention (head_dim
//              32 in 64-byte-swizzled tiles)
//              -> out GEMM (+bias, +=X) -> LN2 -> up GEMM (+bias, GELU) -> down GEMM (+bias, +=X)
//   pred.norm LN -> gather the target rows -> pred.proj GEMM (+bias) -> [B, n_tgt, out_dim] fp32
//
// The pages order the tokens by position id before the blocks and restore the order after the
// norm. Every step is per token except attention, which is full and takes each token's position
// from its own id, so the order changes no result: the sequence stays [context ; targets].
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "internal.h"
#include "jepa.h"
#include "jepa_synth.h"
#include "kernels.h"
#include "ptx.cuh"
#include "seq.h"

using namespace jepa;

// ------------------------------------------------------------------ kernels
namespace {

// Per row r of item b: the token's position id (context ids first, then the targets). A context
// id must index the encoder rows and every id the position grid; an id outside is replaced by 0
// and flagged (kErrBadIds), so no later kernel reads out of bounds.
__global__ void pred_ids_kernel(const int* __restrict__ ctx, int n_ctx, const int* __restrict__ tgt, int n_tgt, int B,
                                int n_enc, int n_pos, int* __restrict__ ids, int* err) {
  pdl_trigger();
  pdl_wait();
  const int n_total = n_ctx + n_tgt;
  const long long total = (long long)B * n_total;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int b = (int)(i / n_total), r = (int)(i % n_total);
    const bool is_ctx = r < n_ctx;
    const int id = is_ctx ? ctx[(size_t)b * n_ctx + r] : tgt[(size_t)b * n_tgt + (r - n_ctx)];
    const bool ok = id >= 0 && id < n_pos && (!is_ctx || id < n_enc);
    if (!ok) atomicOr(err, kErrBadIds);
    ids[i] = ok ? id : 0;
  }
}

// A[b*n_ctx + s, :] = bf16(enc[b, ids[b*n_total + s], :]), 8 columns per thread (E % 8 == 0).
__global__ void pred_gather_ctx_kernel(const float* __restrict__ enc, int n_enc, int E, const int* __restrict__ ids,
                                       int n_total, int n_ctx, int B, __nv_bfloat16* __restrict__ A) {
  pdl_trigger();
  pdl_wait();
  const int E8 = E / 8;
  const long long total = (long long)B * n_ctx * E8;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int c8 = (int)(i % E8);
    const long long row = i / E8;
    const int b = (int)(row / n_ctx), s = (int)(row % n_ctx);
    const int id = __ldg(ids + (size_t)b * n_total + s);
    const float4* src = reinterpret_cast<const float4*>(enc + ((size_t)b * n_enc + id) * E) + 2 * c8;
    const float4 x0 = __ldg(src), x1 = __ldg(src + 1);
    uint4 w;
    w.x = pack_bf16x2(x0.x, x0.y);
    w.y = pack_bf16x2(x0.z, x0.w);
    w.z = pack_bf16x2(x1.x, x1.y);
    w.w = pack_bf16x2(x1.z, x1.w);
    reinterpret_cast<uint4*>(A + (size_t)row * E)[c8] = w;
  }
}

// X[b*n_total + n_ctx + j, :] = token (fp32, P % 4 == 0).
__global__ void pred_fill_targets_kernel(float* __restrict__ X, int B, int n_total, int n_ctx, int P,
                                         const float* __restrict__ token) {
  pdl_trigger();
  pdl_wait();
  const int P4 = P / 4, n_tgt = n_total - n_ctx;
  const long long total = (long long)B * n_tgt * P4;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int c4 = (int)(i % P4);
    const long long row = i / P4;
    const int b = (int)(row / n_tgt), j = (int)(row % n_tgt);
    reinterpret_cast<float4*>(X + ((size_t)b * n_total + n_ctx + j) * P)[c4] =
        __ldg(reinterpret_cast<const float4*>(token) + c4);
  }
}

// Y[b*n_tgt + j, :] = Xn[b*n_total + n_ctx + j, :] (bf16 rows, P % 8 == 0).
__global__ void pred_gather_tgt_kernel(const __nv_bfloat16* __restrict__ Xn, int B, int n_total, int n_ctx, int P,
                                       __nv_bfloat16* __restrict__ Y) {
  pdl_trigger();
  pdl_wait();
  const int P8 = P / 8, n_tgt = n_total - n_ctx;
  const long long total = (long long)B * n_tgt * P8;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int c8 = (int)(i % P8);
    const long long row = i / P8;
    const int b = (int)(row / n_tgt), j = (int)(row % n_tgt);
    reinterpret_cast<uint4*>(Y + (size_t)row * P)[c8] =
        reinterpret_cast<const uint4*>(Xn + ((size_t)b * n_total + n_ctx + j) * P)[c8];
  }
}

int blocks_for(long long work, int threads) {
  long long b = (work + threads - 1) / threads;
  const long long cap = (long long)num_sms() * 16;
  if (b > cap) b = cap;
  return (int)(b < 1 ? 1 : b);
}

struct Rec {
  std::string name;
  size_t offset, n;
  bool bf16;
};
struct PredLayer {
  const float *ln1_w, *ln1_b, *b_qkv, *b_out, *ln2_w, *ln2_b, *b_up, *b_down;
  const void *w_qkv, *w_out, *w_up, *w_down;
  CUtensorMap tm_qkv[3], tm_out[3], tm_up[3], tm_down[3];  // B boxes of 64 / 128 / 256 rows
};
int slot(int bn) { return bn == 64 ? 0 : ((bn == 128 || bn == kPairTile) ? 1 : 2); }
}  // namespace

struct jepa_predictor {
  jepa_pred_hparams hp;
  int dtype = 0, device = 0;
  uint8_t* arena = nullptr;
  std::vector<Rec> tensors;
  const void *w_embed = nullptr, *w_proj = nullptr;
  const float *b_embed = nullptr, *mask_tokens = nullptr, *norm_w = nullptr, *norm_b = nullptr, *b_proj = nullptr;
  std::vector<PredLayer> layers;
  CUtensorMap tm_embed[3], tm_proj[3];
  const Rec* find(const char* name) const {
    for (const auto& t : tensors)
      if (t.name == name) return &t;
    return nullptr;
  }
};

// Kernel classes of the profiling hook.
namespace {
enum PredClass { kQIds, kQGather, kQEmbed, kQFill, kQLn, kQQkv, kQAttn, kQOut, kQUp, kQDown, kQLnFinal, kQGatherTgt,
                 kQProj, kQClasses };
const char* kQNames[kQClasses] = {"pred_ids", "pred_gather_ctx", "gemm_embed", "pred_fill_targets", "layernorm",
                                  "gemm_qkv", "attention", "gemm_out", "gemm_up", "gemm_down", "layernorm_final",
                                  "pred_gather_tgt", "gemm_proj"};
}  // namespace

struct jepa_pred_context {
  const jepa_predictor* p = nullptr;
  SeqRunner run;
  int max_B = 0, max_ctx = 0, max_tgt = 0;
  uint8_t* ws = nullptr;
  size_t ws_bytes = 0;
  float* X = nullptr;
  void *Xn = nullptr, *qkv = nullptr, *ao = nullptr, *Hh = nullptr, *A = nullptr, *Y = nullptr;
  int* ids = nullptr;
  float2* rope = nullptr;
  int* err = nullptr;
  // per-shape state
  int kB = -1, kC = -1, kT = -1, kgt = -1, kgh = -1, kgw = -1;
  float* kout = nullptr;
  CUtensorMap tm_A, tm_Xn, tm_ao, tm_Hh, tm_Y, tm_qkv3, tm_o_qkv, tm_o_hh, tm_o_x, tm_o_out;
  int bn_embed = 0, bn_qkv = 0, bn_out = 0, bn_up = 0, bn_down = 0, bn_proj = 0;
};

// ------------------------------------------------------------------ hyper-parameters
extern "C" jepa_status jepa_pred_preset(const char* name, jepa_pred_hparams* out) {
  if (!name || !out) return fail(JEPA_E_INVALID_ARG, "jepa_pred_preset: null argument");
  jepa_pred_hparams h;
  memset(&h, 0, sizeof h);
  if (std::string(name) == "vjepa2_vitl16") {
    h.embed_dim = 384; h.n_layer = 12; h.n_head = 12; h.ffn_dim = 1536;
    h.enc_dim = 1024; h.out_dim = 1024; h.n_mask_tokens = 10; h.mask_index = 1;
    h.ln_eps = 1e-6f; h.rope_theta = 10000.0f; h.rope_layout = JEPA_ROPE_TILED;
  } else {
    return fail(JEPA_E_INVALID_ARG, "jepa_pred_preset: unknown preset '%s'", name);
  }
  *out = h;
  return JEPA_OK;
}

extern "C" jepa_status jepa_pred_hparams_validate(const jepa_pred_hparams* hp) {
  if (!hp) return fail(JEPA_E_INVALID_ARG, "pred hparams: null");
  auto in = [](int v, int lo, int hi) { return v >= lo && v <= hi; };
  if (!in(hp->embed_dim, 1, 65536)) return fail(JEPA_E_INVALID_ARG, "pred embed_dim %d outside [1, 65536]", hp->embed_dim);
  if (!in(hp->n_layer, 1, 1024)) return fail(JEPA_E_INVALID_ARG, "pred n_layer %d outside [1, 1024]", hp->n_layer);
  if (!in(hp->n_head, 1, 1024)) return fail(JEPA_E_INVALID_ARG, "pred n_head %d outside [1, 1024]", hp->n_head);
  if (!in(hp->ffn_dim, 1, 1 << 20)) return fail(JEPA_E_INVALID_ARG, "pred ffn_dim %d outside [1, 2^20]", hp->ffn_dim);
  if (!in(hp->enc_dim, 1, 65536) || !in(hp->out_dim, 1, 65536))
    return fail(JEPA_E_INVALID_ARG, "pred enc_dim %d / out_dim %d outside [1, 65536]", hp->enc_dim, hp->out_dim);
  if (!in(hp->n_mask_tokens, 1, 1 << 16) || hp->mask_index < 0)
    return fail(JEPA_E_INVALID_ARG, "pred n_mask_tokens %d / mask_index %d", hp->n_mask_tokens, hp->mask_index);
  if (!std::isfinite(hp->ln_eps) || hp->ln_eps < 0.0f || hp->ln_eps > 1.0f)
    return fail(JEPA_E_INVALID_ARG, "pred ln_eps %g not finite in [0, 1]", (double)hp->ln_eps);
  if (!std::isfinite(hp->rope_theta) || hp->rope_theta <= 0.0f)
    return fail(JEPA_E_INVALID_ARG, "pred rope_theta %g must be finite and > 0", (double)hp->rope_theta);
  if (!in(hp->rope_layout, 0, 1)) return fail(JEPA_E_INVALID_ARG, "pred rope_layout %d unknown", hp->rope_layout);
  if (hp->embed_dim % hp->n_head)
    return fail(JEPA_E_INVALID_ARG, "pred embed_dim %d not divisible by n_head %d", hp->embed_dim, hp->n_head);
  if ((hp->embed_dim / hp->n_head) % 2)
    return fail(JEPA_E_INVALID_ARG, "pred head width %d is odd (3-D RoPE rotates pairs)", hp->embed_dim / hp->n_head);
  return JEPA_OK;
}

// ------------------------------------------------------------------ weights
extern "C" void jepa_pred_free(jepa_predictor* p) {
  if (!p) return;
  if (p->arena) {
    cudaSetDevice(p->device);
    cudaFree(p->arena);
  }
  delete p;
}

extern "C" jepa_status jepa_pred_load(const jepa_pred_hparams* hp, uint64_t seed, int32_t dtype, int32_t device,
                                      jepa_predictor** out) {
  if (!hp || !out) return fail(JEPA_E_INVALID_ARG, "jepa_pred_load: null argument");
  *out = nullptr;
  jepa_status st = jepa_pred_hparams_validate(hp);
  if (st != JEPA_OK) return st;
  if (dtype != JEPA_BF16) return fail(JEPA_E_UNSUPPORTED, "the predictor runs in bf16 only (dtype %d)", dtype);
  const int P = hp->embed_dim, F = hp->ffn_dim, E = hp->enc_dim, O = hp->out_dim, L = hp->n_layer;
  const int hd = P / hp->n_head;
  if (hd != 32 && hd != 64) return fail(JEPA_E_UNSUPPORTED, "predictor head_dim %d: 32 or 64 only", hd);
  if (P % 64 || F % 64 || E % 64 || O % 64 || P > 2048)
    return fail(JEPA_E_UNSUPPORTED, "predictor widths (embed %d, ffn %d, enc %d, out %d) must be multiples of 64, "
                "embed at most 2048", P, F, E, O);
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
    return fail(JEPA_E_CUDA, "CUDA device %d not available (%d devices)", device, ndev);
  CUDA_TRY(cudaSetDevice(device));
  jepa_predictor* p = new jepa_predictor();
  p->hp = *hp;
  p->dtype = dtype;
  p->device = device;
  auto add = [&](const std::string& name, size_t n, bool matrix) { p->tensors.push_back({name, 0, n, matrix}); };
  add("pred.embed.weight", (size_t)P * E, true);
  add("pred.embed.bias", P, false);
  add("pred.mask_tokens", (size_t)hp->n_mask_tokens * P, false);
  for (int l = 0; l < L; ++l) {
    const std::string s = "pred.blk." + std::to_string(l) + ".";
    add(s + "ln1.weight", P, false);
    add(s + "ln1.bias", P, false);
    add(s + "attn_qkv.weight", (size_t)3 * P * P, true);
    add(s + "attn_qkv.bias", (size_t)3 * P, false);
    add(s + "attn_out.weight", (size_t)P * P, true);
    add(s + "attn_out.bias", P, false);
    add(s + "ln2.weight", P, false);
    add(s + "ln2.bias", P, false);
    add(s + "ffn_up.weight", (size_t)F * P, true);
    add(s + "ffn_up.bias", F, false);
    add(s + "ffn_down.weight", (size_t)P * F, true);
    add(s + "ffn_down.bias", P, false);
  }
  add("pred.norm.weight", P, false);
  add("pred.norm.bias", P, false);
  add("pred.proj.weight", (size_t)O * P, true);
  add("pred.proj.bias", O, false);
  size_t off = 0, largest = 0;
  for (auto& t : p->tensors) {
    t.offset = off;
    off = align256(off + t.n * (t.bf16 ? 2 : 4));
    largest = std::max(largest, t.n);
  }
  cudaError_t e = cudaMalloc(&p->arena, off);
  if (e != cudaSuccess) {
    delete p;
    return fail(JEPA_E_OOM, "predictor weights: cudaMalloc(%zu bytes) failed: %s", off, cudaGetErrorString(e));
  }
  std::vector<float> host(largest);
  std::vector<uint16_t> bits;
  for (const auto& t : p->tensors) {
    synth_parallel(seed, t.name, 1, t.n, host.data());
    if (t.bf16) {
      bits.resize(t.n);
      for (size_t i = 0; i < t.n; ++i) bits[i] = jsynth_f32_to_bf16_bits(host[i]);
      e = cudaMemcpy(p->arena + t.offset, bits.data(), t.n * 2, cudaMemcpyHostToDevice);
    } else {
      e = cudaMemcpy(p->arena + t.offset, host.data(), t.n * 4, cudaMemcpyHostToDevice);
    }
    if (e != cudaSuccess) {
      jepa_pred_free(p);
      return fail(JEPA_E_CUDA, "predictor weights upload: %s", cudaGetErrorString(e));
    }
  }
  auto ptr = [&](const std::string& n) -> void* { return p->arena + p->find(n.c_str())->offset; };
  auto fptr = [&](const std::string& n) -> const float* { return reinterpret_cast<const float*>(ptr(n)); };
  p->w_embed = ptr("pred.embed.weight");
  p->b_embed = fptr("pred.embed.bias");
  p->mask_tokens = fptr("pred.mask_tokens");
  p->norm_w = fptr("pred.norm.weight");
  p->norm_b = fptr("pred.norm.bias");
  p->w_proj = ptr("pred.proj.weight");
  p->b_proj = fptr("pred.proj.bias");
  const uint32_t boxes[3] = {64, 128, 256};
  bool ok = true;
  for (int s = 0; s < 3; ++s) {
    ok &= make_tmap_2d_bf16(&p->tm_embed[s], p->w_embed, P, E, boxes[s]);
    ok &= make_tmap_2d_bf16(&p->tm_proj[s], p->w_proj, O, P, boxes[s]);
  }
  p->layers.resize(L);
  for (int l = 0; l < L; ++l) {
    const std::string s = "pred.blk." + std::to_string(l) + ".";
    PredLayer& w = p->layers[l];
    w.ln1_w = fptr(s + "ln1.weight");
    w.ln1_b = fptr(s + "ln1.bias");
    w.w_qkv = ptr(s + "attn_qkv.weight");
    w.b_qkv = fptr(s + "attn_qkv.bias");
    w.w_out = ptr(s + "attn_out.weight");
    w.b_out = fptr(s + "attn_out.bias");
    w.ln2_w = fptr(s + "ln2.weight");
    w.ln2_b = fptr(s + "ln2.bias");
    w.w_up = ptr(s + "ffn_up.weight");
    w.b_up = fptr(s + "ffn_up.bias");
    w.w_down = ptr(s + "ffn_down.weight");
    w.b_down = fptr(s + "ffn_down.bias");
    for (int b = 0; b < 3; ++b) {
      ok &= make_tmap_2d_bf16(&w.tm_qkv[b], w.w_qkv, 3 * P, P, boxes[b]);
      ok &= make_tmap_2d_bf16(&w.tm_out[b], w.w_out, P, P, boxes[b]);
      ok &= make_tmap_2d_bf16(&w.tm_up[b], w.w_up, F, P, boxes[b]);
      ok &= make_tmap_2d_bf16(&w.tm_down[b], w.w_down, P, F, boxes[b]);
    }
  }
  if (!ok) {
    jepa_pred_free(p);
    return fail(JEPA_E_CUDA, "cuTensorMapEncodeTiled refused a predictor weight map");
  }
  *out = p;
  return JEPA_OK;
}

extern "C" jepa_status jepa_pred_tensor(const jepa_predictor* p, const char* name, float* h_dst, size_t n_elems) {
  if (!p || !name || !h_dst) return fail(JEPA_E_INVALID_ARG, "jepa_pred_tensor: null argument");
  const Rec* t = p->find(name);
  if (!t) return fail(JEPA_E_INVALID_ARG, "jepa_pred_tensor: no tensor named '%s'", name);
  if (t->n != n_elems) return fail(JEPA_E_INVALID_ARG, "tensor '%s' has %zu elements, not %zu", name, t->n, n_elems);
  CUDA_TRY(cudaSetDevice(p->device));
  if (t->bf16) {
    std::vector<uint16_t> bits(t->n);
    CUDA_TRY(cudaMemcpy(bits.data(), p->arena + t->offset, t->n * 2, cudaMemcpyDeviceToHost));
    for (size_t i = 0; i < t->n; ++i) h_dst[i] = jsynth_bf16_bits_to_f32(bits[i]);
  } else {
    CUDA_TRY(cudaMemcpy(h_dst, p->arena + t->offset, t->n * 4, cudaMemcpyDeviceToHost));
  }
  return JEPA_OK;
}

// ------------------------------------------------------------------ context
namespace {
// qkv columns of the workspace: [q | k | v], n_head heads of head_dim each.
int qkv_cols(const jepa_pred_hparams& hp) { return 3 * hp.embed_dim; }

size_t pred_ws_layout(const jepa_predictor* p, long long B, long long n_ctx, long long n_tgt, int rope_rows,
                      jepa_pred_context* c) {
  const jepa_pred_hparams& hp = p->hp;
  const size_t P = hp.embed_dim, F = hp.ffn_dim, E = hp.enc_dim;
  const size_t rows = (size_t)(B * (n_ctx + n_tgt));
  const int dh = rope_d(hp.embed_dim / hp.n_head) / 2;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const size_t oX = take(rows * P * 4), oXn = take(rows * P * 2), oQ = take(rows * qkv_cols(hp) * 2),
               oA = take(rows * P * 2), oH = take(rows * F * 2), oC = take((size_t)(B * n_ctx) * E * 2),
               oY = take((size_t)(B * n_tgt) * P * 2), oI = take(rows * 4),
               oR = take((size_t)rope_rows * std::max(dh, 1) * sizeof(float2)), oE = take(sizeof(int));
  if (c) {
    c->X = reinterpret_cast<float*>(c->ws + oX);
    c->Xn = c->ws + oXn;
    c->qkv = c->ws + oQ;
    c->ao = c->ws + oA;
    c->Hh = c->ws + oH;
    c->A = c->ws + oC;
    c->Y = c->ws + oY;
    c->ids = reinterpret_cast<int*>(c->ws + oI);
    c->rope = reinterpret_cast<float2*>(c->ws + oR);
    c->err = reinterpret_cast<int*>(c->ws + oE);
  }
  return off;
}
constexpr int kMaxRopeRows = 1 << 16;  // gt + gh + gw of the position grid
}  // namespace

extern "C" jepa_status jepa_pred_context_new(const jepa_predictor* p, int32_t max_batch, int32_t max_ctx,
                                             int32_t max_tgt, size_t max_workspace_bytes, jepa_pred_context** out) {
  if (!p || !out) return fail(JEPA_E_INVALID_ARG, "jepa_pred_context_new: null argument");
  *out = nullptr;
  if (max_batch <= 0 || max_ctx < 0 || max_tgt <= 0 || (long long)max_ctx + max_tgt > (1 << 22))
    return fail(JEPA_E_INVALID_ARG, "predictor context %d x (%d + %d) tokens out of range", max_batch, max_ctx, max_tgt);
  const size_t need = pred_ws_layout(p, max_batch, max_ctx, max_tgt, kMaxRopeRows, nullptr);
  const size_t budget = max_workspace_bytes ? max_workspace_bytes : kDefaultBudget;
  if (need > budget)
    return fail(JEPA_E_BUDGET, "predictor workspace of %zu bytes for %d x (%d + %d) tokens exceeds the budget of %zu bytes",
                need, max_batch, max_ctx, max_tgt, budget);
  CUDA_TRY(cudaSetDevice(p->device));
  CUDA_TRY(tc_kernels_init());
  jepa_pred_context* c = new jepa_pred_context();
  c->p = p;
  c->max_B = max_batch;
  c->max_ctx = max_ctx;
  c->max_tgt = max_tgt;
  cudaError_t e = cudaMalloc(&c->ws, need);
  if (e != cudaSuccess) {
    delete c;
    return fail(JEPA_E_OOM, "predictor workspace: cudaMalloc(%zu bytes) failed: %s", need, cudaGetErrorString(e));
  }
  c->ws_bytes = need;
  pred_ws_layout(p, max_batch, max_ctx, max_tgt, kMaxRopeRows, c);
  e = cudaMemset(c->ws, 0, need);
  if (e != cudaSuccess) {
    cudaFree(c->ws);
    delete c;
    return fail(JEPA_E_CUDA, "predictor context: %s", cudaGetErrorString(e));
  }
  const jepa_status st = c->run.init(kQClasses);
  if (st != JEPA_OK) {
    cudaFree(c->ws);
    delete c;
    return st;
  }
  *out = c;
  return JEPA_OK;
}

extern "C" void jepa_pred_context_free(jepa_pred_context* c) {
  if (!c) return;
  cudaSetDevice(c->p->device);
  c->run.destroy();
  if (c->ws) cudaFree(c->ws);
  delete c;
}

extern "C" jepa_status jepa_pred_context_set_stream(jepa_pred_context* c, void* stream) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_pred_context_set_stream: null context");
  CUDA_TRY(cudaSetDevice(c->p->device));
  return c->run.set_stream(stream);
}

extern "C" jepa_status jepa_pred_context_set_graph(jepa_pred_context* c, int32_t enable) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_pred_context_set_graph: null context");
  c->run.use_graph = enable != 0;
  return JEPA_OK;
}

extern "C" jepa_status jepa_pred_context_set_profiling(jepa_pred_context* c, int32_t enable) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_pred_context_set_profiling: null context");
  c->run.profiling = enable != 0;
  return JEPA_OK;
}

namespace {
int pred_launches(const jepa_pred_hparams& hp, int n_ctx) {
  return 1 + (n_ctx > 0 ? 2 : 0) + 1 + 7 * hp.n_layer + 3;
}

// Per-shape set-up: tensor maps over the workspace and the output, GEMM tile widths, RoPE axes.
jepa_status pred_prepare(jepa_pred_context* c, int B, int n_ctx, int n_tgt, int gt, int gh, int gw, float* out) {
  if (c->kB == B && c->kC == n_ctx && c->kT == n_tgt && c->kgt == gt && c->kgh == gh && c->kgw == gw && c->kout == out)
    return JEPA_OK;
  const jepa_pred_hparams& hp = c->p->hp;
  const int P = hp.embed_dim, F = hp.ffn_dim, E = hp.enc_dim, O = hp.out_dim;
  const long long M = (long long)B * (n_ctx + n_tgt), Mc = (long long)B * n_ctx, Mt = (long long)B * n_tgt;
  bool ok = true;
  if (Mc > 0) ok &= make_tmap_2d_bf16(&c->tm_A, c->A, Mc, E, 128);
  ok &= make_tmap_2d_bf16(&c->tm_Xn, c->Xn, M, P, 128);
  ok &= make_tmap_2d_bf16(&c->tm_ao, c->ao, M, P, 128);
  ok &= make_tmap_2d_bf16(&c->tm_Hh, c->Hh, M, F, 128);
  ok &= make_tmap_2d_bf16(&c->tm_Y, c->Y, Mt, P, 128);
  ok &= make_tmap_3d_bf16(&c->tm_qkv3, c->qkv, B, n_ctx + n_tgt, qkv_cols(hp), 128, hp.embed_dim / hp.n_head);
  ok &= make_tmap_2d_out(&c->tm_o_qkv, c->qkv, M, qkv_cols(hp), 2);
  ok &= make_tmap_2d_out(&c->tm_o_hh, c->Hh, M, F, 2);
  ok &= make_tmap_2d_out(&c->tm_o_x, c->X, M, P, 4);
  ok &= make_tmap_2d_out(&c->tm_o_out, out, Mt, O, 4);
  if (!ok) return fail(JEPA_E_CUDA, "cuTensorMapEncodeTiled refused a predictor workspace map");
  c->bn_embed = Mc > 0 ? gemm_tc_pick_bn((int)Mc, P) : 64;
  c->bn_qkv = gemm_tc_pick_bn((int)M, 3 * P);
  c->bn_out = gemm_tc_pick_bn((int)M, P);
  c->bn_up = gemm_tc_pick_bn((int)M, F);
  c->bn_down = gemm_tc_pick_bn((int)M, P);
  c->bn_proj = gemm_tc_pick_bn((int)Mt, O);
  CUDA_TRY(rope_axes_launch(gt, gh, gw, P / hp.n_head, hp.rope_theta, 0, 0, c->rope, c->run.stream));
  c->kB = B;
  c->kC = n_ctx;
  c->kT = n_tgt;
  c->kgt = gt;
  c->kgh = gh;
  c->kgw = gw;
  c->kout = out;
  return JEPA_OK;
}

EpiArgs epi_of(int kind, int M, int N, const float* bias, void* out) {
  EpiArgs e;
  memset(&e, 0, sizeof e);
  e.kind = kind;
  e.M = M;
  e.N = N;
  e.bias = bias;
  e.out = out;
  e.rows_per_item = 1;
  e.patches_per_item = 1;
  return e;
}

jepa_status pred_launch(jepa_pred_context* c, const float* enc, int B, int n_enc, const int* ctx, int n_ctx,
                        const int* tgt, int n_tgt, int gt, int gh, int gw, float* out) {
  const jepa_predictor* p = c->p;
  const jepa_pred_hparams& hp = p->hp;
  const int P = hp.embed_dim, F = hp.ffn_dim, E = hp.enc_dim, O = hp.out_dim, NH = hp.n_head, hd = P / NH;
  const int n_total = n_ctx + n_tgt, M = B * n_total, Mc = B * n_ctx, Mt = B * n_tgt;
  cudaStream_t s = c->run.stream;
  const uint64_t lim = default_wait_limit_ns();
  PdlScope pdl_scope(!c->run.profiling);
  auto timed = [c](int cls, double fl, double by, auto&& launch) { return c->run.timed(cls, fl, by, launch); };
  const double dM = M, dP = P, dF = F;
  const double ln_bytes = dM * dP * 6.0;

  CUDA_TRY(timed(kQIds, 0.0, (double)M * 8.0, [&] {
    return launch_kernel(pred_ids_kernel, dim3(blocks_for(M, 256)), dim3(256), 0, s, ctx, n_ctx, tgt, n_tgt, B, n_enc,
                         gt * gh * gw, c->ids, c->err);
  }));
  if (n_ctx > 0) {
    CUDA_TRY(timed(kQGather, 0.0, (double)Mc * E * 6.0, [&] {
      return launch_kernel(pred_gather_ctx_kernel, dim3(blocks_for((long long)Mc * (E / 8), 256)), dim3(256), 0, s,
                           enc, n_enc, E, (const int*)c->ids, n_total, n_ctx, B, reinterpret_cast<__nv_bfloat16*>(c->A));
    }));
    EpiArgs ee = epi_of(kEpiPatch, Mc, P, p->b_embed, c->X);  // row s of item b -> X row b*n_total + s
    ee.patches_per_item = n_ctx;
    ee.rows_per_item = n_total;
    CUDA_TRY(timed(kQEmbed, 2.0 * Mc * dP * E, 0.0, [&] {
      return gemm_tc_launch(c->tm_A, p->tm_embed[slot(c->bn_embed)], c->tm_o_x, c->bn_embed, ee, Mc, P, E, c->err,
                            lim, s);
    }));
  }
  const float* token = p->mask_tokens + (size_t)(hp.mask_index % hp.n_mask_tokens) * P;
  CUDA_TRY(timed(kQFill, 0.0, (double)Mt * P * 4.0, [&] {
    return launch_kernel(pred_fill_targets_kernel, dim3(blocks_for((long long)Mt * (P / 4), 256)), dim3(256), 0, s,
                         c->X, B, n_total, n_ctx, P, token);
  }));

  AttnParams ap;
  ap.B = B;
  ap.N = n_total;
  ap.H = NH;
  ap.head_dim = hd;  // width-32 heads in their own 64-byte tiles
  ap.attn_mode = 0;
  ap.prefix = 0;
  ap.frame_tokens = 1;
  ap.out = c->ao;
  const double attn_flops = 4.0 * hd * NH * B * (double)n_total * n_total;
  for (int l = 0; l < hp.n_layer; ++l) {
    const PredLayer& w = p->layers[l];
    EpiArgs qe = epi_of(kEpiQkvRope, M, 3 * P, w.b_qkv, c->qkv);
    qe.rows_per_item = n_total;
    qe.n_head = NH;
    qe.head_dim = hd;
    qe.rope_layout = hp.rope_layout;
    qe.rope_d = rope_d(hd);
    qe.rope_axes = c->rope;
    qe.rope_gt = gt;
    qe.rope_gh = gh;
    qe.rope_gw = gw;
    qe.rope_ids = c->ids;
    EpiArgs oe = epi_of(kEpiResidual, M, P, w.b_out, c->X);
    EpiArgs ue = epi_of(kEpiGelu, M, F, w.b_up, c->Hh);
    EpiArgs de = epi_of(kEpiResidual, M, P, w.b_down, c->X);
    CUDA_TRY(timed(kQLn, 0.0, ln_bytes,
                   [&] { return layernorm_launch(c->X, M, P, w.ln1_w, w.ln1_b, hp.ln_eps, true, c->Xn, s); }));
    CUDA_TRY(timed(kQQkv, 2.0 * dM * 3.0 * dP * dP, 0.0, [&] {
      return gemm_tc_launch(c->tm_Xn, w.tm_qkv[slot(c->bn_qkv)], c->tm_o_qkv, c->bn_qkv, qe, M, 3 * P, P, c->err, lim, s);
    }));
    CUDA_TRY(timed(kQAttn, attn_flops, 0.0, [&] { return attention_tc_launch(c->tm_qkv3, ap, c->err, lim, s); }));
    CUDA_TRY(timed(kQOut, 2.0 * dM * dP * dP, 0.0, [&] {
      return gemm_tc_launch(c->tm_ao, w.tm_out[slot(c->bn_out)], c->tm_o_x, c->bn_out, oe, M, P, P, c->err, lim, s);
    }));
    CUDA_TRY(timed(kQLn, 0.0, ln_bytes,
                   [&] { return layernorm_launch(c->X, M, P, w.ln2_w, w.ln2_b, hp.ln_eps, true, c->Xn, s); }));
    CUDA_TRY(timed(kQUp, 2.0 * dM * dF * dP, 0.0, [&] {
      return gemm_tc_launch(c->tm_Xn, w.tm_up[slot(c->bn_up)], c->tm_o_hh, c->bn_up, ue, M, F, P, c->err, lim, s);
    }));
    CUDA_TRY(timed(kQDown, 2.0 * dM * dP * dF, 0.0, [&] {
      return gemm_tc_launch(c->tm_Hh, w.tm_down[slot(c->bn_down)], c->tm_o_x, c->bn_down, de, M, P, F, c->err, lim, s);
    }));
  }
  CUDA_TRY(timed(kQLnFinal, 0.0, ln_bytes,
                 [&] { return layernorm_launch(c->X, M, P, p->norm_w, p->norm_b, hp.ln_eps, true, c->Xn, s); }));
  CUDA_TRY(timed(kQGatherTgt, 0.0, (double)Mt * P * 4.0, [&] {
    return launch_kernel(pred_gather_tgt_kernel, dim3(blocks_for((long long)Mt * (P / 8), 256)), dim3(256), 0, s,
                         reinterpret_cast<const __nv_bfloat16*>(c->Xn), B, n_total, n_ctx, P,
                         reinterpret_cast<__nv_bfloat16*>(c->Y));
  }));
  EpiArgs pe = epi_of(kEpiPatch, Mt, O, p->b_proj, out);  // rows are the output rows: fp32 TMA store
  pe.patches_per_item = n_tgt;
  pe.rows_per_item = n_tgt;
  CUDA_TRY(timed(kQProj, 2.0 * Mt * (double)O * P, 0.0, [&] {
    return gemm_tc_launch(c->tm_Y, p->tm_proj[slot(c->bn_proj)], c->tm_o_out, c->bn_proj, pe, Mt, O, P, c->err, lim, s);
  }));
  return JEPA_OK;
}
}  // namespace

extern "C" jepa_status jepa_pred_context_launches(const jepa_pred_context* c, int32_t n_ctx, int32_t* n_out) {
  if (!c || !n_out) return fail(JEPA_E_INVALID_ARG, "jepa_pred_context_launches: null argument");
  *n_out = pred_launches(c->p->hp, n_ctx);
  return JEPA_OK;
}

extern "C" jepa_status jepa_predict(jepa_pred_context* c, const float* d_enc, int32_t B, int32_t n_enc,
                                    const int32_t* d_ctx_ids, int32_t n_ctx, const int32_t* d_tgt_ids, int32_t n_tgt,
                                    int32_t gt, int32_t gh, int32_t gw, float* d_out) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_predict: null context");
  if (!d_enc || !d_tgt_ids || !d_out || (n_ctx > 0 && !d_ctx_ids))
    return fail(JEPA_E_INVALID_ARG, "jepa_predict: null pointer");
  if (B <= 0 || n_enc <= 0 || n_ctx < 0 || n_tgt <= 0 || gt <= 0 || gh <= 0 || gw <= 0)
    return fail(JEPA_E_INVALID_ARG, "jepa_predict: sizes B %d, n_enc %d, n_ctx %d, n_tgt %d, grid %dx%dx%d", B, n_enc,
                n_ctx, n_tgt, gt, gh, gw);
  if ((long long)gt * gh * gw > (1ll << 22) || gt + gh + gw > kMaxRopeRows)
    return fail(JEPA_E_INVALID_ARG, "jepa_predict: position grid %dx%dx%d too large", gt, gh, gw);
  if (B > c->max_B || n_ctx > c->max_ctx || n_tgt > c->max_tgt)
    return fail(JEPA_E_BUDGET, "jepa_predict: %d x (%d + %d) tokens exceed the context's %d x (%d + %d)", B, n_ctx,
                n_tgt, c->max_B, c->max_ctx, c->max_tgt);
  if (c->p->hp.enc_dim % 8) return fail(JEPA_E_UNSUPPORTED, "jepa_predict: enc_dim %d not a multiple of 8", c->p->hp.enc_dim);
  if ((reinterpret_cast<uintptr_t>(d_enc) | reinterpret_cast<uintptr_t>(d_out)) & 15)
    return fail(JEPA_E_INVALID_ARG, "jepa_predict: encoder tokens and output must be 16-byte aligned");
  CUDA_TRY(cudaSetDevice(c->p->device));
  jepa_status st = pred_prepare(c, B, n_ctx, n_tgt, gt, gh, gw, d_out);
  if (st != JEPA_OK) return st;
  const std::vector<uintptr_t> key = {(uintptr_t)B, (uintptr_t)n_enc, (uintptr_t)n_ctx, (uintptr_t)n_tgt,
                                     (uintptr_t)gt, (uintptr_t)gh, (uintptr_t)gw, (uintptr_t)d_enc,
                                     (uintptr_t)d_ctx_ids, (uintptr_t)d_tgt_ids, (uintptr_t)d_out};
  return c->run.run(key, [&] { return pred_launch(c, d_enc, B, n_enc, d_ctx_ids, n_ctx, d_tgt_ids, n_tgt, gt, gh, gw,
                                                  d_out); }, "jepa_predict");
}

extern "C" jepa_status jepa_pred_context_sync(jepa_pred_context* c) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_pred_context_sync: null context");
  CUDA_TRY(cudaSetDevice(c->p->device));
  return c->run.sync(c->err, "jepa_predict");
}

extern "C" jepa_status jepa_pred_context_profile(jepa_pred_context* c, jepa_kernel_stat* out, int32_t max,
                                                 int32_t* n_out, int32_t reset) {
  if (!c || !n_out || (max > 0 && !out)) return fail(JEPA_E_INVALID_ARG, "jepa_pred_context_profile: null argument");
  CUDA_TRY(cudaSetDevice(c->p->device));
  return c->run.profile(kQNames, out, max, n_out, reset);
}
