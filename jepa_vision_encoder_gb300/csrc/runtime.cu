// runtime.cu -- the C ABI of include/jepa.h: hyper-parameter validation, synthetic model
// load (enc.* tensors of the GGUF schema, uploaded once), the context workspace, and the
// launch sequence of one encode ("Architecture", The shared ViT graph):
//
//   patchify -> patch GEMM (+bias, +pos / modality, CLS row offset) [-> CLS prefix rows]
//   per layer: LN1 -> QKV GEMM (+bias, 3-D RoPE on q/k) -> attention -> out GEMM (+bias, +=X)
//              LN2 -> FFN-up GEMM (+bias, GELU) -> FFN-down GEMM (+bias, +=X)
//   final LN -> tokens (fp32)
//
// bf16 models run the tcgen05 GEMM and flash-attention kernels; fp32 models the SIMT ones.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "jepa.h"
#include "jepa_synth.h"
#include "internal.h"
#include "kernels.h"

using namespace jepa;

// ------------------------------------------------------------------ errors
namespace {
thread_local std::string t_err;
}  // namespace

jepa_status jepa::fail(jepa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_err = buf;
  return s;
}

extern "C" const char* jepa_error_text(void) { return t_err.c_str(); }
extern "C" void jepa_error_reset(void) { t_err.clear(); }

// ------------------------------------------------------------------ hyper-parameters
extern "C" jepa_status jepa_preset(const char* name, jepa_hparams* out) {
  if (!name || !out) return fail(JEPA_E_INVALID_ARG, "jepa_preset: null argument");
  jepa_hparams h;
  memset(&h, 0, sizeof h);
  h.in_chans = 3;
  h.ln_eps = 1e-6f;
  h.rope_theta = 10000.0f;
  const std::string n(name);
  if (n == "hfvit_ti14") {
    h.embed_dim = 192; h.n_layer = 12; h.n_head = 3; h.ffn_dim = 768;
    h.patch_size = 14; h.tubelet_size = 1; h.img_size = 224; h.n_frames = 1;
    h.pos_type = JEPA_POS_LEARNED; h.cls_token = 1; h.n_pos_rows = 257;
  } else if (n == "vjepa2_vitl16") {
    h.embed_dim = 1024; h.n_layer = 24; h.n_head = 16; h.ffn_dim = 4096;
    h.patch_size = 16; h.tubelet_size = 2; h.img_size = 256; h.n_frames = 16;
    h.pos_type = JEPA_POS_ROPE3D; h.rope_layout = JEPA_ROPE_TILED;
  } else if (n == "vjepa2_1_vitl16") {
    h.embed_dim = 1024; h.n_layer = 24; h.n_head = 16; h.ffn_dim = 4096;
    h.patch_size = 16; h.tubelet_size = 2; h.img_size = 384; h.n_frames = 16;
    h.pos_type = JEPA_POS_ROPE3D; h.rope_layout = JEPA_ROPE_INTERLEAVED;
    h.rope_interpolate = 1; h.rope_ref_grid = 256 / 16; h.modality_embed = 1;
  } else if (n == "levjepa_vitl16") {
    h.embed_dim = 1024; h.n_layer = 24; h.n_head = 16; h.ffn_dim = 4096;
    h.patch_size = 16; h.tubelet_size = 1; h.img_size = 256; h.n_frames = 16;
    h.pos_type = JEPA_POS_ROPE3D; h.rope_layout = JEPA_ROPE_TILED; h.cls_token = 1;
    h.attn_mode = JEPA_ATTN_BLOCK_CAUSAL;
  } else if (n == "vjepa2_vitg16") {
    h.embed_dim = 1408; h.n_layer = 40; h.n_head = 22; h.ffn_dim = 6144;
    h.patch_size = 16; h.tubelet_size = 2; h.img_size = 256; h.n_frames = 64;
    h.pos_type = JEPA_POS_ROPE3D; h.rope_layout = JEPA_ROPE_TILED;
  } else if (n == "vjepa_vitl16") {
    h.embed_dim = 1024; h.n_layer = 24; h.n_head = 16; h.ffn_dim = 4096;
    h.patch_size = 16; h.tubelet_size = 2; h.img_size = 224; h.n_frames = 16;
    h.pos_type = JEPA_POS_SINCOS3D; h.sincos_uniform_power = 1;
  } else if (n == "ijepa_vitl16") {
    h.embed_dim = 1024; h.n_layer = 24; h.n_head = 16; h.ffn_dim = 4096;
    h.patch_size = 16; h.tubelet_size = 1; h.img_size = 224; h.n_frames = 1;
    h.pos_type = JEPA_POS_SINCOS2D; h.sincos_w_first = 1;
  } else {
    return fail(JEPA_E_INVALID_ARG, "jepa_preset: unknown preset '%s'", name);
  }
  *out = h;
  return JEPA_OK;
}

extern "C" jepa_status jepa_hparams_validate(const jepa_hparams* hp) {
  if (!hp) return fail(JEPA_E_INVALID_ARG, "hparams: null");
  auto in = [](int v, int lo, int hi) { return v >= lo && v <= hi; };
  if (!in(hp->embed_dim, 1, 65536)) return fail(JEPA_E_INVALID_ARG, "embed_dim %d outside [1, 65536]", hp->embed_dim);
  if (!in(hp->n_layer, 1, 1024)) return fail(JEPA_E_INVALID_ARG, "n_layer %d outside [1, 1024]", hp->n_layer);
  if (!in(hp->n_head, 1, 1024)) return fail(JEPA_E_INVALID_ARG, "n_head %d outside [1, 1024]", hp->n_head);
  if (!in(hp->ffn_dim, 1, 1 << 20)) return fail(JEPA_E_INVALID_ARG, "ffn_dim %d outside [1, 2^20]", hp->ffn_dim);
  if (!in(hp->patch_size, 1, 1024)) return fail(JEPA_E_INVALID_ARG, "patch_size %d outside [1, 1024]", hp->patch_size);
  if (!in(hp->tubelet_size, 1, 1024)) return fail(JEPA_E_INVALID_ARG, "tubelet_size %d outside [1, 1024]", hp->tubelet_size);
  if (!in(hp->in_chans, 1, 1024)) return fail(JEPA_E_INVALID_ARG, "in_chans %d outside [1, 1024]", hp->in_chans);
  if (hp->img_size != 0 && !in(hp->img_size, 1, 65536)) return fail(JEPA_E_INVALID_ARG, "img_size %d outside [1, 65536]", hp->img_size);
  if (hp->n_frames != 0 && !in(hp->n_frames, 1, 65536)) return fail(JEPA_E_INVALID_ARG, "n_frames %d outside [1, 65536]", hp->n_frames);
  if (!std::isfinite(hp->ln_eps) || hp->ln_eps < 0.0f || hp->ln_eps > 1.0f)
    return fail(JEPA_E_INVALID_ARG, "ln_eps %g not finite in [0, 1]", (double)hp->ln_eps);
  if (!in(hp->pos_type, 0, 4)) return fail(JEPA_E_INVALID_ARG, "pos_type %d unknown", hp->pos_type);
  if (!in(hp->rope_layout, 0, 1)) return fail(JEPA_E_INVALID_ARG, "rope_layout %d unknown", hp->rope_layout);
  if (!in(hp->attn_mode, 0, 1)) return fail(JEPA_E_INVALID_ARG, "attn_mode %d unknown", hp->attn_mode);
  if (hp->embed_dim % hp->n_head) return fail(JEPA_E_INVALID_ARG, "embed_dim %d not divisible by n_head %d", hp->embed_dim, hp->n_head);
  const int hd = hp->embed_dim / hp->n_head;
  if (hp->pos_type == JEPA_POS_ROPE3D) {
    if (!std::isfinite(hp->rope_theta) || hp->rope_theta <= 0.0f)
      return fail(JEPA_E_INVALID_ARG, "rope_theta %g must be finite and > 0", (double)hp->rope_theta);
    if (hd % 2) return fail(JEPA_E_INVALID_ARG, "odd head width %d on a 3-D RoPE model (it rotates pairs)", hd);
    if (hp->rope_interpolate && hp->rope_ref_grid < 1)
      return fail(JEPA_E_INVALID_ARG, "rope_interpolate without a rope_ref_grid to rescale from");
  }
  if (hp->pos_type == JEPA_POS_LEARNED && !in(hp->n_pos_rows, 1, 1 << 22))
    return fail(JEPA_E_INVALID_ARG, "learned position table needs n_pos_rows in [1, 2^22] (got %d)", hp->n_pos_rows);
  if (hp->pos_type == JEPA_POS_SINCOS2D || hp->pos_type == JEPA_POS_SINCOS3D) {
    const bool three = hp->pos_type == JEPA_POS_SINCOS3D;
    if (hp->img_size < hp->patch_size || hp->img_size % hp->patch_size)
      return fail(JEPA_E_INVALID_ARG, "a sin-cos table needs img_size %d to be a multiple of patch %d", hp->img_size,
                  hp->patch_size);
    if (three && (hp->n_frames < hp->tubelet_size || hp->n_frames % hp->tubelet_size))
      return fail(JEPA_E_INVALID_ARG, "a 3-D sin-cos table needs n_frames %d to be a multiple of tubelet %d",
                  hp->n_frames, hp->tubelet_size);
    int d0, d1, d2;
    if (!sincos_widths(three ? 1 : 0, hp->embed_dim, hp->sincos_uniform_power, &d0, &d1, &d2))
      return fail(JEPA_E_INVALID_ARG, "embed_dim %d cannot be split into the %s sin-cos axes", hp->embed_dim,
                  three ? "3-D" : "2-D");
    const long long rows = (long long)(three ? hp->n_frames / hp->tubelet_size : 1) *
                           (hp->img_size / hp->patch_size) * (hp->img_size / hp->patch_size);
    if (rows > (1ll << 22)) return fail(JEPA_E_INVALID_ARG, "sin-cos training grid of %lld rows above 2^22", rows);
  }
  return JEPA_OK;
}

namespace {
struct Geo {
  int gt, gh, gw, Np, prefix, N, K;
};
jepa_status geometry(const jepa_hparams* hp, int T, int H, int W, Geo* g) {
  if (T <= 0 || H <= 0 || W <= 0) return fail(JEPA_E_INVALID_ARG, "clip size %dx%dx%d must be positive", T, H, W);
  if (T % hp->tubelet_size || H % hp->patch_size || W % hp->patch_size)
    return fail(JEPA_E_INVALID_ARG, "clip %dx%dx%d not divisible by tubelet %d / patch %d", T, H, W,
                hp->tubelet_size, hp->patch_size);
  g->gt = T / hp->tubelet_size;
  g->gh = H / hp->patch_size;
  g->gw = W / hp->patch_size;
  const long long np = (long long)g->gt * g->gh * g->gw;
  if (np + 1 > (1ll << 22)) return fail(JEPA_E_INVALID_ARG, "token count %lld above 2^22", np);
  g->Np = (int)np;
  g->prefix = hp->cls_token ? 1 : 0;
  g->N = g->Np + g->prefix;
  g->K = hp->in_chans * hp->tubelet_size * hp->patch_size * hp->patch_size;
  return JEPA_OK;
}

bool is_sincos(const jepa_hparams& hp) { return hp.pos_type == JEPA_POS_SINCOS2D || hp.pos_type == JEPA_POS_SINCOS3D; }

// The grid a sin-cos table is baked for: (n_frames/t) x (img/P) x (img/P), one frame for 2-D.
void sincos_train_grid(const jepa_hparams& hp, int* gt, int* gh, int* gw) {
  *gt = hp.pos_type == JEPA_POS_SINCOS3D ? hp.n_frames / hp.tubelet_size : 1;
  *gh = *gw = hp.img_size / hp.patch_size;
}
}  // namespace

extern "C" jepa_status jepa_n_tokens(const jepa_hparams* hp, int32_t T, int32_t H, int32_t W, int32_t* n_out) {
  if (!hp || !n_out) return fail(JEPA_E_INVALID_ARG, "jepa_n_tokens: null argument");
  jepa_status s = jepa_hparams_validate(hp);
  if (s != JEPA_OK) return s;
  Geo g;
  s = geometry(hp, T, H, W, &g);
  if (s != JEPA_OK) return s;
  *n_out = g.N;
  return JEPA_OK;
}

// ------------------------------------------------------------------ model
namespace {
struct TensorRec {
  std::string name;
  size_t offset;  // in the arena
  size_t n;
  bool bf16;
  bool fixed;     // computed by a kernel (sin-cos table), not drawn from the generator
  bool matrix;    // a weight matrix; every other tensor is an fp32 operand (norm, bias, token, table)
  std::vector<uint64_t> shape;  // PyTorch order
};

// The enc.* tensors of an encoder, in GGUF names and PyTorch row-major shapes ("GGUF schema (v1)",
// Encoder tensors). bake_sincos marks a sin-cos table as computed on the device.
std::vector<TensorRec> encoder_tensors(const jepa_hparams& hp, bool bf, bool bake_sincos) {
  const uint64_t D = hp.embed_dim, F = hp.ffn_dim;
  const uint64_t K = (uint64_t)hp.in_chans * hp.tubelet_size * hp.patch_size * hp.patch_size;
  std::vector<TensorRec> ts;
  auto add = [&](const std::string& name, std::vector<uint64_t> shape, bool matrix, bool fixed = false) {
    TensorRec r;
    r.name = name;
    r.n = 1;
    for (uint64_t d : shape) r.n *= d;
    r.bf16 = bf && matrix;
    r.fixed = fixed;
    r.matrix = matrix;
    r.shape = std::move(shape);
    r.offset = 0;
    ts.push_back(std::move(r));
  };
  add("enc.patch_embed.weight", {D, K}, true);
  add("enc.patch_embed.bias", {D}, false);
  if (hp.pos_type == JEPA_POS_LEARNED) add("enc.pos_embed", {(uint64_t)hp.n_pos_rows, D}, false);
  if (hp.pos_type == JEPA_POS_SINCOS2D || hp.pos_type == JEPA_POS_SINCOS3D) {
    const uint64_t gt = hp.pos_type == JEPA_POS_SINCOS3D ? hp.n_frames / hp.tubelet_size : 1;
    const uint64_t g = hp.img_size / hp.patch_size;
    add("enc.pos_embed", {gt * g * g, D}, false, bake_sincos);
  }
  if (hp.cls_token) add("enc.cls_token", {D}, false);
  if (hp.modality_embed) add("enc.mod_embed_video", {D}, false);
  for (int l = 0; l < hp.n_layer; ++l) {
    const std::string p = "enc.blk." + std::to_string(l) + ".";
    add(p + "ln1.weight", {D}, false);
    add(p + "ln1.bias", {D}, false);
    add(p + "attn_qkv.weight", {3 * D, D}, true);
    add(p + "attn_qkv.bias", {3 * D}, false);
    add(p + "attn_out.weight", {D, D}, true);
    add(p + "attn_out.bias", {D}, false);
    add(p + "ln2.weight", {D}, false);
    add(p + "ln2.bias", {D}, false);
    add(p + "ffn_up.weight", {F, D}, true);
    add(p + "ffn_up.bias", {F}, false);
    add(p + "ffn_down.weight", {D, F}, true);
    add(p + "ffn_down.bias", {D}, false);
  }
  add("enc.norm.weight", {D}, false);
  add("enc.norm.bias", {D}, false);
  return ts;
}

// Fills n floats of tensor `name`; the model's synthetic weights or a file's.
using TensorFill = std::function<jepa_status(const TensorRec& t, float* dst)>;
struct LayerW {
  const float *ln1_w, *ln1_b, *b_qkv, *b_out, *ln2_w, *ln2_b, *b_up, *b_down;
  const void *w_qkv, *w_out, *w_up, *w_down;
  CUtensorMap tm_qkv[3], tm_out[3], tm_up[3], tm_down[3];  // box rows 64 / 128 / 256
};
int bn_slot(int bn) { return bn == 64 ? 0 : ((bn == 128 || bn == kPairTile) ? 1 : 2); }
}  // namespace

struct jepa_model {
  jepa_hparams hp;
  int dtype = 0, device = 0;
  uint64_t seed = 0;
  uint8_t* arena = nullptr;
  size_t arena_bytes = 0;
  std::vector<TensorRec> tensors;
  const void* w_patch = nullptr;
  const float *b_patch = nullptr, *pos = nullptr, *cls = nullptr, *mod = nullptr, *norm_w = nullptr, *norm_b = nullptr;
  std::vector<LayerW> layers;
  CUtensorMap tm_patch[3];
  int K = 0;
  const TensorRec* find(const char* name) const {
    for (const auto& t : tensors)
      if (t.name == name) return &t;
    return nullptr;
  }
};

// Fill `n` values of tensor `name` (the synth recipe) using all host cores.
void jepa::synth_parallel(uint64_t seed, const std::string& name, int bf16_matrices, size_t n, float* dst) {
  int kind, is_matrix;
  double a, b;
  jsynth_param_init(name.c_str(), &kind, &a, &b, &is_matrix);
  const int round = (bf16_matrices && is_matrix) ? 1 : 0;
  unsigned nt = std::max(1u, std::thread::hardware_concurrency());
  if (n < 65536) nt = 1;
  std::vector<std::thread> th;
  const size_t per = (n + nt - 1) / nt;
  for (unsigned t = 0; t < nt; ++t) {
    const size_t first = (size_t)t * per;
    if (first >= n) break;
    const size_t len = std::min(per, n - first);
    th.emplace_back([=] { jsynth_fill(seed, name.c_str(), kind, a, b, round, first, len, dst + first); });
  }
  for (auto& x : th) x.join();
}

namespace {
// Builds a model: the tensor table, one arena, every tensor filled (fill == nullptr: the synthetic
// recipe of `seed`, sin-cos tables baked on the device; otherwise `fill`, tables included) and
// uploaded (bf16 matrices rounded to nearest even), then the weight tensor maps.
jepa_status model_create(const jepa_hparams* hp, uint64_t seed, int32_t dtype, int32_t device, const TensorFill* fill,
                         jepa_model** out) {
  if (!hp || !out) return fail(JEPA_E_INVALID_ARG, "jepa_model_load: null argument");
  *out = nullptr;
  jepa_status st = jepa_hparams_validate(hp);
  if (st != JEPA_OK) return st;
  if (dtype != JEPA_FP32 && dtype != JEPA_BF16) return fail(JEPA_E_INVALID_ARG, "dtype %d unknown", dtype);
  const int D = hp->embed_dim, F = hp->ffn_dim, L = hp->n_layer;
  const int hd = D / hp->n_head;
  const int K = hp->in_chans * hp->tubelet_size * hp->patch_size * hp->patch_size;
  if (hd != 64) return fail(JEPA_E_UNSUPPORTED, "head_dim %d: the attention kernels are built for 64", hd);
  if (D % 4 || D > 2048) return fail(JEPA_E_UNSUPPORTED, "embed_dim %d: LayerNorm needs a multiple of 4 up to 2048", D);
  if (F % 4) return fail(JEPA_E_UNSUPPORTED, "ffn_dim %d must be a multiple of 4", F);
  if (dtype == JEPA_BF16 && (D % 64 || F % 64 || K % 64))
    return fail(JEPA_E_UNSUPPORTED, "bf16 GEMMs need embed %d, ffn %d and patch K %d to be multiples of 64", D, F, K);
  if (is_sincos(*hp) && hp->cls_token)
    return fail(JEPA_E_UNSUPPORTED, "a sin-cos table with a CLS token (the tables cover patch rows only)");
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
    return fail(JEPA_E_CUDA, "CUDA device %d not available (%d devices)", device, ndev);
  CUDA_TRY(cudaSetDevice(device));

  jepa_model* m = new jepa_model();
  m->hp = *hp;
  m->dtype = dtype;
  m->device = device;
  m->seed = seed;
  m->K = K;
  const bool bf = dtype == JEPA_BF16;
  m->tensors = encoder_tensors(*hp, bf, fill == nullptr);
  int pgt = 0, pgh = 0, pgw = 0;  // training grid of a sin-cos table
  if (is_sincos(*hp)) sincos_train_grid(*hp, &pgt, &pgh, &pgw);
  size_t off = 0, largest = 0;
  for (auto& t : m->tensors) {
    t.offset = off;
    off = align256(off + t.n * (t.bf16 ? 2 : 4));
    largest = std::max(largest, t.n);
  }
  m->arena_bytes = off;
  cudaError_t e = cudaMalloc(&m->arena, off);
  if (e != cudaSuccess) {
    delete m;
    return fail(JEPA_E_OOM, "weights: cudaMalloc(%zu bytes) failed: %s", off, cudaGetErrorString(e));
  }
  std::vector<float> host(largest);
  std::vector<uint16_t> hbits;
  for (const auto& t : m->tensors) {
    if (t.fixed) continue;
    if (fill) {
      const jepa_status fs = (*fill)(t, host.data());
      if (fs != JEPA_OK) {
        jepa_model_free(m);
        return fs;
      }
    } else {
      synth_parallel(seed, t.name, bf ? 1 : 0, t.n, host.data());
    }
    if (t.bf16) {
      hbits.resize(t.n);
      for (size_t i = 0; i < t.n; ++i) hbits[i] = jsynth_f32_to_bf16_bits(host[i]);
      e = cudaMemcpy(m->arena + t.offset, hbits.data(), t.n * 2, cudaMemcpyHostToDevice);
    } else {
      e = cudaMemcpy(m->arena + t.offset, host.data(), t.n * 4, cudaMemcpyHostToDevice);
    }
    if (e != cudaSuccess) {
      jepa_model_free(m);
      return fail(JEPA_E_CUDA, "weights upload: %s", cudaGetErrorString(e));
    }
  }
  auto ptr = [&](const std::string& name) -> void* { return m->arena + m->find(name.c_str())->offset; };
  auto fptr = [&](const std::string& name) -> const float* { return reinterpret_cast<const float*>(ptr(name)); };
  m->w_patch = ptr("enc.patch_embed.weight");
  m->b_patch = fptr("enc.patch_embed.bias");
  if (hp->pos_type == JEPA_POS_LEARNED) m->pos = fptr("enc.pos_embed");
  if (is_sincos(*hp) && !fill) {  // the converter's table of the training grid, baked here on the device
    float* tab = reinterpret_cast<float*>(ptr("enc.pos_embed"));
    e = sincos_table_launch(hp->pos_type == JEPA_POS_SINCOS3D ? 1 : 0, pgt, pgh, pgw, D, hp->sincos_w_first,
                            hp->sincos_uniform_power, tab, nullptr);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      jepa_model_free(m);
      return fail(JEPA_E_CUDA, "sin-cos table: %s", cudaGetErrorString(e));
    }
    m->pos = tab;
  }
  if (is_sincos(*hp) && fill) m->pos = fptr("enc.pos_embed");  // the file's table
  if (hp->cls_token) m->cls = fptr("enc.cls_token");
  if (hp->modality_embed) m->mod = fptr("enc.mod_embed_video");
  m->norm_w = fptr("enc.norm.weight");
  m->norm_b = fptr("enc.norm.bias");
  m->layers.resize(L);
  bool maps_ok = true;
  const uint32_t boxes[3] = {64, 128, 256};
  for (int s = 0; s < 3 && bf; ++s) maps_ok &= make_tmap_2d_bf16(&m->tm_patch[s], m->w_patch, D, K, boxes[s]);
  for (int l = 0; l < L; ++l) {
    const std::string p = "enc.blk." + std::to_string(l) + ".";
    LayerW& w = m->layers[l];
    w.ln1_w = fptr(p + "ln1.weight");
    w.ln1_b = fptr(p + "ln1.bias");
    w.w_qkv = ptr(p + "attn_qkv.weight");
    w.b_qkv = fptr(p + "attn_qkv.bias");
    w.w_out = ptr(p + "attn_out.weight");
    w.b_out = fptr(p + "attn_out.bias");
    w.ln2_w = fptr(p + "ln2.weight");
    w.ln2_b = fptr(p + "ln2.bias");
    w.w_up = ptr(p + "ffn_up.weight");
    w.b_up = fptr(p + "ffn_up.bias");
    w.w_down = ptr(p + "ffn_down.weight");
    w.b_down = fptr(p + "ffn_down.bias");
    for (int s = 0; s < 3 && bf; ++s) {
      maps_ok &= make_tmap_2d_bf16(&w.tm_qkv[s], w.w_qkv, 3 * D, D, boxes[s]);
      maps_ok &= make_tmap_2d_bf16(&w.tm_out[s], w.w_out, D, D, boxes[s]);
      maps_ok &= make_tmap_2d_bf16(&w.tm_up[s], w.w_up, F, D, boxes[s]);
      maps_ok &= make_tmap_2d_bf16(&w.tm_down[s], w.w_down, D, F, boxes[s]);
    }
  }
  if (!maps_ok) {
    jepa_model_free(m);
    return fail(JEPA_E_CUDA, "cuTensorMapEncodeTiled refused a weight tensor map");
  }
  *out = m;
  return JEPA_OK;
}

// ---- GGUF encoder files ("Architecture", Robustness: what the loader validates)
bool gguf_is_int(const GgufValue& v) { return v.type <= 5 || v.type == 10 || v.type == 11; }  // u8..i32, u64, i64

jepa_status gguf_int(const GgufFile& g, const char* key, bool required, int64_t lo, int64_t hi, int32_t dflt,
                     int32_t* out) {
  const GgufValue* v = g.get(key);
  if (!v) {
    if (required) return fail(JEPA_E_INVALID_ARG, "gguf: required key %s is missing", key);
    *out = dflt;
    return JEPA_OK;
  }
  if (!gguf_is_int(*v)) return fail(JEPA_E_INVALID_ARG, "gguf: %s is not an integer (type %u)", key, v->type);
  const bool neg = (v->type == 1 || v->type == 3 || v->type == 5 || v->type == 11) && v->i < 0;
  if (neg || (!neg && v->u > (uint64_t)hi) || v->i < lo)
    return fail(JEPA_E_INVALID_ARG, "gguf: %s = %lld outside [%lld, %lld]", key, (long long)v->i, (long long)lo,
                (long long)hi);
  *out = (int32_t)v->i;
  return JEPA_OK;
}

jepa_status gguf_float(const GgufFile& g, const char* key, bool required, float dflt, float* out) {
  const GgufValue* v = g.get(key);
  if (!v) {
    if (required) return fail(JEPA_E_INVALID_ARG, "gguf: required key %s is missing", key);
    *out = dflt;
    return JEPA_OK;
  }
  if (v->type != 6 && v->type != 12) return fail(JEPA_E_INVALID_ARG, "gguf: %s is not a float (type %u)", key, v->type);
  if (!std::isfinite(v->f)) return fail(JEPA_E_INVALID_ARG, "gguf: %s is not finite", key);
  *out = (float)v->f;
  return JEPA_OK;
}

jepa_status gguf_bool(const GgufFile& g, const char* key, bool* out) {
  const GgufValue* v = g.get(key);
  *out = false;  // a flag the file does not set is off
  if (!v) return JEPA_OK;
  if (v->type != 7) return fail(JEPA_E_INVALID_ARG, "gguf: %s is not a bool (type %u)", key, v->type);
  *out = v->u != 0;
  return JEPA_OK;
}

jepa_status gguf_str(const GgufFile& g, const char* key, bool required, const char* dflt, std::string* out) {
  const GgufValue* v = g.get(key);
  if (!v) {
    if (required) return fail(JEPA_E_INVALID_ARG, "gguf: required key %s is missing", key);
    *out = dflt;
    return JEPA_OK;
  }
  if (v->type != 8) return fail(JEPA_E_INVALID_ARG, "gguf: %s is not a string (type %u)", key, v->type);
  *out = v->s;
  return JEPA_OK;
}

// Dims of a GGUF tensor in PyTorch order, without ggml's trailing unit dimensions.
std::vector<uint64_t> torch_shape(const GgufTensor& t) {
  std::vector<uint64_t> d(t.dims.rbegin(), t.dims.rend());
  while (d.size() > 1 && d.front() == 1) d.erase(d.begin());
  return d;
}

std::string shape_str(const std::vector<uint64_t>& d) {
  std::string s = "[";
  for (size_t i = 0; i < d.size(); ++i) s += (i ? ", " : "") + std::to_string(d[i]);
  return s + "]";
}

// The encoder of a GGUF file: its jepa.* keys as hyper-parameters, checked as the pages' loader
// checks them, and its tensors against those hyper-parameters (presence, dtype, shape).
jepa_status gguf_encoder(const GgufFile& g, jepa_hparams* hp, bool* qkv_fused) {
  std::string s;
  jepa_status st = gguf_str(g, "general.architecture", true, "", &s);
  if (st != JEPA_OK) return st;
  if (s != "jepa") return fail(JEPA_E_INVALID_ARG, "gguf: general.architecture is '%s', not jepa", s.c_str());
  std::string family;
  if ((st = gguf_str(g, "jepa.family", true, "", &family)) != JEPA_OK) return st;
  const char* families[] = {"ijepa", "vjepa", "vjepa2", "vjepa2_1", "levjepa", "hfvit", "lewm"};
  bool known = false;
  for (const char* f : families) known |= family == f;
  if (!known) return fail(JEPA_E_INVALID_ARG, "gguf: jepa.family '%s' is not one of the seven families", family.c_str());
  if (family == "lewm") return fail(JEPA_E_UNSUPPORTED, "gguf: family lewm (its projector is not built here)");
  jepa_hparams h;
  memset(&h, 0, sizeof h);
  struct IntKey { const char* key; int64_t lo, hi; int32_t* dst; };
  const IntKey ints[] = {
      {"jepa.enc.embed_dim", 1, 65536, &h.embed_dim},   {"jepa.enc.n_layer", 1, 1024, &h.n_layer},
      {"jepa.enc.n_head", 1, 1024, &h.n_head},          {"jepa.enc.ffn_dim", 1, 1 << 20, &h.ffn_dim},
      {"jepa.enc.patch_size", 1, 1024, &h.patch_size},  {"jepa.enc.tubelet_size", 1, 1024, &h.tubelet_size},
      {"jepa.enc.img_size", 1, 65536, &h.img_size},     {"jepa.enc.n_frames", 1, 65536, &h.n_frames},
      {"jepa.enc.in_chans", 1, 1024, &h.in_chans}};
  for (const auto& k : ints)
    if ((st = gguf_int(g, k.key, true, k.lo, k.hi, 0, k.dst)) != JEPA_OK) return st;
  if ((st = gguf_float(g, "jepa.enc.ln_eps", true, 0.0f, &h.ln_eps)) != JEPA_OK) return st;
  std::string act, pos, layout, mode;
  if ((st = gguf_str(g, "jepa.enc.act", true, "", &act)) != JEPA_OK) return st;
  if (act == "gelu_tanh" || act == "silu")
    return fail(JEPA_E_UNSUPPORTED, "gguf: jepa.enc.act %s (this build runs gelu_erf)", act.c_str());
  if (act != "gelu_erf") return fail(JEPA_E_INVALID_ARG, "gguf: jepa.enc.act '%s' unknown", act.c_str());
  if ((st = gguf_str(g, "jepa.enc.pos_type", true, "", &pos)) != JEPA_OK) return st;
  if (pos == "sincos2d") h.pos_type = JEPA_POS_SINCOS2D;
  else if (pos == "sincos3d") h.pos_type = JEPA_POS_SINCOS3D;
  else if (pos == "learned") h.pos_type = JEPA_POS_LEARNED;
  else if (pos == "rope3d") h.pos_type = JEPA_POS_ROPE3D;
  else return fail(JEPA_E_INVALID_ARG, "gguf: jepa.enc.pos_type '%s' unknown", pos.c_str());
  // the pages: attn_mode is absent from every existing file and the loader defaults it to full
  if ((st = gguf_str(g, "jepa.enc.attn_mode", false, "full", &mode)) != JEPA_OK) return st;
  if (mode == "block_causal") {
    if (family != "levjepa")
      return fail(JEPA_E_INVALID_ARG, "gguf: attn_mode block_causal on family %s, whose graph has no mask", family.c_str());
    h.attn_mode = JEPA_ATTN_BLOCK_CAUSAL;
  } else if (mode != "full") {
    return fail(JEPA_E_INVALID_ARG, "gguf: jepa.enc.attn_mode '%s' unknown", mode.c_str());
  }
  bool interp = false, cls = false, fused = false, mod = false, ls = false;
  if ((st = gguf_bool(g, "jepa.enc.cls_token", &cls)) != JEPA_OK) return st;
  if ((st = gguf_bool(g, "jepa.enc.modality_embed", &mod)) != JEPA_OK) return st;
  if ((st = gguf_bool(g, "jepa.enc.layer_scale", &ls)) != JEPA_OK) return st;
  if (ls) return fail(JEPA_E_UNSUPPORTED, "gguf: layer scale (ls1 / ls2) is not built here");
  fused = true;
  if (g.get("jepa.enc.qkv_fused") && (st = gguf_bool(g, "jepa.enc.qkv_fused", &fused)) != JEPA_OK) return st;
  int32_t n_reg = 0;
  if ((st = gguf_int(g, "jepa.enc.n_registers", false, 0, 1 << 16, 0, &n_reg)) != JEPA_OK) return st;
  if (n_reg) return fail(JEPA_E_UNSUPPORTED, "gguf: %d register tokens (not built here)", n_reg);
  h.cls_token = cls;
  h.modality_embed = mod;
  if (h.pos_type == JEPA_POS_ROPE3D) {
    if ((st = gguf_float(g, "jepa.enc.rope_theta", true, 0.0f, &h.rope_theta)) != JEPA_OK) return st;
    if ((st = gguf_str(g, "jepa.enc.rope_freq_layout", true, "", &layout)) != JEPA_OK) return st;
    if (layout == "tiled") h.rope_layout = JEPA_ROPE_TILED;
    else if (layout == "interleaved") h.rope_layout = JEPA_ROPE_INTERLEAVED;
    else return fail(JEPA_E_INVALID_ARG, "gguf: jepa.enc.rope_freq_layout '%s' unknown", layout.c_str());
    if ((st = gguf_bool(g, "jepa.enc.rope_interpolate", &interp)) != JEPA_OK) return st;
    h.rope_interpolate = interp;
    if ((st = gguf_int(g, "jepa.enc.rope_ref_grid", false, 0, 65536, 0, &h.rope_ref_grid)) != JEPA_OK) return st;
  } else {
    h.rope_theta = 10000.0f;  // unused without RoPE
  }
  if (h.pos_type == JEPA_POS_LEARNED) {  // the table's rows come from the tensor itself
    const GgufTensor* t = g.find("enc.pos_embed");
    if (!t) return fail(JEPA_E_INVALID_ARG, "gguf: required tensor enc.pos_embed is missing");
    const std::vector<uint64_t> d = torch_shape(*t);
    if (d.size() != 2 || d[0] > (1u << 22))
      return fail(JEPA_E_INVALID_ARG, "gguf: enc.pos_embed has shape %s", shape_str(d).c_str());
    h.n_pos_rows = (int32_t)d[0];
  }
  if ((st = jepa_hparams_validate(&h)) != JEPA_OK) return st;
  // tensors: present, f32 for every operand the graph adds, a float type for the matrices, shapes
  std::vector<TensorRec> want = encoder_tensors(h, false, false);
  if (!fused) {  // separate q / k / v projections, fused at load
    std::vector<TensorRec> w2;
    for (const auto& t : want) {
      const size_t at = t.name.find("attn_qkv.");
      if (at == std::string::npos) {
        w2.push_back(t);
        continue;
      }
      const bool weight = t.name.compare(at + 9, std::string::npos, "weight") == 0;
      for (const char* part : {"attn_q.", "attn_k.", "attn_v."}) {
        TensorRec r = t;
        r.name = t.name.substr(0, at) + part + (weight ? "weight" : "bias");
        r.shape = weight ? std::vector<uint64_t>{(uint64_t)h.embed_dim, (uint64_t)h.embed_dim}
                         : std::vector<uint64_t>{(uint64_t)h.embed_dim};
        r.n = t.n / 3;
        w2.push_back(r);
      }
    }
    want.swap(w2);
  }
  for (const auto& t : want) {
    const GgufTensor* gt = g.find(t.name);
    if (!gt) return fail(JEPA_E_INVALID_ARG, "gguf: required tensor %s is missing", t.name.c_str());
    if (!t.matrix && gt->type != 0)
      return fail(JEPA_E_INVALID_ARG, "gguf: %s is %s; norms, biases, tokens and tables must be f32", t.name.c_str(),
                  gguf_type_name(gt->type));
    if (torch_shape(*gt) != t.shape)
      return fail(JEPA_E_INVALID_ARG, "gguf: %s has shape %s, the hyper-parameters give %s", t.name.c_str(),
                  shape_str(torch_shape(*gt)).c_str(), shape_str(t.shape).c_str());
    if (t.matrix && gt->type != 0 && gt->type != 1 && gt->type != 30)
      return fail(JEPA_E_UNSUPPORTED, "gguf: %s is %s; this build reads f32, f16 and bf16 weights", t.name.c_str(),
                  gguf_type_name(gt->type));
  }
  *hp = h;
  *qkv_fused = fused;
  return JEPA_OK;
}
}  // namespace

extern "C" jepa_status jepa_model_load(const jepa_hparams* hp, uint64_t seed, int32_t dtype, int32_t device,
                                       jepa_model** out) {
  return model_create(hp, seed, dtype, device, nullptr, out);
}

extern "C" jepa_status jepa_gguf_hparams(const char* path, jepa_hparams* out) {
  if (!path || !out) return fail(JEPA_E_INVALID_ARG, "jepa_gguf_hparams: null argument");
  GgufFile g;
  jepa_status st = gguf_open(path, &g);
  if (st != JEPA_OK) return st;
  bool fused = true;
  return gguf_encoder(g, out, &fused);
}

extern "C" jepa_status jepa_model_load_gguf(const char* path, int32_t dtype, int32_t device, jepa_model** out) {
  if (!path || !out) return fail(JEPA_E_INVALID_ARG, "jepa_model_load_gguf: null argument");
  *out = nullptr;
  GgufFile g;
  jepa_status st = gguf_open(path, &g);
  if (st != JEPA_OK) return st;
  jepa_hparams hp;
  bool fused = true;
  if ((st = gguf_encoder(g, &hp, &fused)) != JEPA_OK) return st;
  const TensorFill fill = [&](const TensorRec& t, float* dst) -> jepa_status {
    const size_t at = t.name.find("attn_qkv.");
    if (fused || at == std::string::npos) return gguf_read_f32(g, *g.find(t.name), dst);
    const bool weight = t.name.compare(at + 9, std::string::npos, "weight") == 0;
    const size_t part = t.n / 3;  // rows [q; k; v]
    const char* names[3] = {"attn_q.", "attn_k.", "attn_v."};
    for (int i = 0; i < 3; ++i) {
      const std::string n = t.name.substr(0, at) + names[i] + (weight ? "weight" : "bias");
      const jepa_status s2 = gguf_read_f32(g, *g.find(n), dst + i * part);
      if (s2 != JEPA_OK) return s2;
    }
    return JEPA_OK;
  };
  return model_create(&hp, 0, dtype, device, &fill, out);
}

extern "C" void jepa_model_free(jepa_model* m) {
  if (!m) return;
  if (m->arena) {
    cudaSetDevice(m->device);
    cudaFree(m->arena);
  }
  delete m;
}

extern "C" jepa_status jepa_model_hparams(const jepa_model* m, jepa_hparams* out) {
  if (!m || !out) return fail(JEPA_E_INVALID_ARG, "jepa_model_hparams: null argument");
  *out = m->hp;
  return JEPA_OK;
}

extern "C" jepa_status jepa_model_tensor(const jepa_model* m, const char* name, float* h_dst, size_t n_elems) {
  if (!m || !name || !h_dst) return fail(JEPA_E_INVALID_ARG, "jepa_model_tensor: null argument");
  const TensorRec* t = m->find(name);
  if (!t) return fail(JEPA_E_INVALID_ARG, "jepa_model_tensor: no tensor named '%s'", name);
  if (t->n != n_elems) return fail(JEPA_E_INVALID_ARG, "tensor '%s' has %zu elements, not %zu", name, t->n, n_elems);
  CUDA_TRY(cudaSetDevice(m->device));
  if (t->bf16) {
    std::vector<uint16_t> bits(t->n);
    CUDA_TRY(cudaMemcpy(bits.data(), m->arena + t->offset, t->n * 2, cudaMemcpyDeviceToHost));
    for (size_t i = 0; i < t->n; ++i) h_dst[i] = jsynth_bf16_bits_to_f32(bits[i]);
  } else {
    CUDA_TRY(cudaMemcpy(h_dst, m->arena + t->offset, t->n * 4, cudaMemcpyDeviceToHost));
  }
  return JEPA_OK;
}

// ------------------------------------------------------------------ context
// Batches of this many items or more (bf16) encode as two halves on two streams.
static constexpr int kSplitMin = 4;

struct jepa_context {
  const jepa_model* m = nullptr;
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  int max_B = 0, max_T = 0, max_H = 0, max_W = 0;
  long long max_rows = 0, max_prows = 0, max_np = 0, max_pix = 0;
  uint8_t* ws = nullptr;
  size_t ws_bytes = 0;
  float* X = nullptr;
  void *Xn = nullptr, *qkv = nullptr, *ao = nullptr, *Hh = nullptr, *Pm = nullptr;
  float2* rope = nullptr;
  float* pos_buf = nullptr;         // a sin-cos table resized to the current clip grid
  const float* pos_clip = nullptr;  // the table the patch rows add: the model's, or pos_buf
  float *pix_stage = nullptr, *tok_stage = nullptr;
  int* err = nullptr;
  // per-shape state
  int kB = -1, kT = -1, kH = -1, kW = -1;
  // A lane: the items [item0, item0 + B) of the batch, their rows of every workspace buffer, the
  // tensor maps over those rows and the GEMM tile widths for their row count. lanes[0] is the
  // whole batch; a batch of kSplitMin or more items (bf16, no per-kernel profiling) runs as
  // lanes[1] and lanes[2], its two halves, on the context stream and a side stream (fork and join
  // through events): the kernels of one half fill the SMs that the other half's persistent grids
  // leave idle in their last rounds (8 clips: 11.0 -> 10.8 ms). Each row's arithmetic is the same
  // either way.
  struct Lane {
    int item0 = 0, B = 0;
    float* X = nullptr;
    void *Xn = nullptr, *qkv = nullptr, *ao = nullptr, *Hh = nullptr, *Pm = nullptr;
    CUtensorMap tm_Pm, tm_Xn, tm_ao, tm_Hh, tm_qkv3;
    CUtensorMap tm_o_qkv, tm_o_hh, tm_o_x;  // GEMM outputs: qkv and Hh (bf16), X (fp32 residual adds)
    int bn_patch = 0, bn_qkv = 0, bn_out = 0, bn_up = 0, bn_down = 0;
  };
  Lane lanes[3];
  bool halves = false;  // lanes[1] and lanes[2] are set up for the current shape
  cudaStream_t side = nullptr;  // the second half's stream (owned)
  cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
  // graph replay
  bool use_graph = false;
  bool use_pdl = true;  // programmatic dependent launches in the encode sequence
  cudaGraphExec_t gexec = nullptr;
  int gB = -1, gT = -1, gH = -1, gW = -1, glayout = -1;
  const float* gpix = nullptr;
  float* gtok = nullptr;
  // per-kernel profiling (events on the context stream)
  bool profiling = false;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_used = 0;
  struct Rec { int cls; size_t e0, e1; double flops, bytes; };
  std::vector<Rec> recs;
  // events recorded inside a captured graph (re-recorded by every replay, folded after each)
  bool capturing = false, gprof = false, gpending = false, gpdl = false;
  std::vector<cudaEvent_t> gev;
  size_t gev_used = 0;
  std::vector<Rec> grecs;
  int prof_launches[16] = {};
  double prof_ms[16] = {}, prof_flops[16] = {}, prof_bytes[16] = {};
  // pipelined host encodes: two device slots each for the pixels coming in and the tokens going
  // out, uploads and downloads on their own streams, so a step's copies overlap other steps'
  // encodes (allocated by the first jepa_encode_host_async)
  bool hp_ready = false;
  float* hp_pix[2] = {nullptr, nullptr};
  float* hp_tok[2] = {nullptr, nullptr};
  cudaStream_t hp_up = nullptr, hp_down = nullptr;
  cudaEvent_t hp_uploaded[2] = {}, hp_pix_free[2] = {}, hp_tok_ready[2] = {}, hp_downloaded[2] = {};
  long long hp_step = 0;
};

namespace {
size_t ws_layout(const jepa_model* m, long long rows, long long prows, long long np, long long pix, jepa_context* c) {
  const jepa_hparams& hp = m->hp;
  const size_t D = hp.embed_dim, F = hp.ffn_dim, K = m->K;
  const size_t es = m->dtype == JEPA_BF16 ? 2 : 4;
  const int dh = rope_d(D / hp.n_head) / 2;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const size_t oX = take(rows * D * 4), oXn = take(rows * D * es), oQ = take(rows * 3 * D * es),
               oA = take(rows * D * es), oH = take(rows * F * es), oP = take(prows * K * es),
               oR = take((size_t)np * 3 * std::max(dh, 1) * sizeof(float2)),
               oPos = take(is_sincos(hp) ? (size_t)np * D * 4 : 0), oPix = take(pix * 4),
               oTok = take(pix > 0 ? rows * D * 4 : 0),  // host staging only where pixels are staged too
               oErr = take(sizeof(int));
  if (c) {
    c->X = reinterpret_cast<float*>(c->ws + oX);
    c->Xn = c->ws + oXn;
    c->qkv = c->ws + oQ;
    c->ao = c->ws + oA;
    c->Hh = c->ws + oH;
    c->Pm = c->ws + oP;
    c->rope = reinterpret_cast<float2*>(c->ws + oR);
    c->pos_buf = is_sincos(hp) ? reinterpret_cast<float*>(c->ws + oPos) : nullptr;
    c->pix_stage = pix > 0 ? reinterpret_cast<float*>(c->ws + oPix) : nullptr;
    c->tok_stage = pix > 0 ? reinterpret_cast<float*>(c->ws + oTok) : nullptr;
    c->err = reinterpret_cast<int*>(c->ws + oErr);
  }
  return off;
}
}  // namespace

extern "C" jepa_status jepa_context_new(const jepa_model* m, int32_t max_batch, int32_t max_frames,
                                        int32_t max_height, int32_t max_width, size_t max_workspace_bytes,
                                        jepa_context** out) {
  if (!m || !out) return fail(JEPA_E_INVALID_ARG, "jepa_context_new: null argument");
  *out = nullptr;
  if (max_batch <= 0) return fail(JEPA_E_INVALID_ARG, "max_batch %d must be positive", max_batch);
  Geo g;
  jepa_status st = geometry(&m->hp, max_frames, max_height, max_width, &g);
  if (st != JEPA_OK) return st;
  const long long rows = (long long)max_batch * g.N, prows = (long long)max_batch * g.Np;
  const long long pix = (long long)max_batch * max_frames * m->hp.in_chans * max_height * max_width;
  const size_t need = ws_layout(m, rows, prows, g.Np, pix, nullptr);
  const size_t budget = max_workspace_bytes ? max_workspace_bytes : kDefaultBudget;
  if (need > budget)
    return fail(JEPA_E_BUDGET, "workspace of %zu bytes for %d x (%dx%dx%d) exceeds the budget of %zu bytes", need,
                max_batch, max_frames, max_height, max_width, budget);
  CUDA_TRY(cudaSetDevice(m->device));
  if (m->dtype == JEPA_BF16) CUDA_TRY(tc_kernels_init());
  jepa_context* c = new jepa_context();
  c->m = m;
  c->max_B = max_batch;
  c->max_T = max_frames;
  c->max_H = max_height;
  c->max_W = max_width;
  c->max_rows = rows;
  c->max_prows = prows;
  c->max_np = g.Np;
  c->max_pix = pix;
  cudaError_t e = cudaMalloc(&c->ws, need);
  if (e != cudaSuccess) {
    delete c;
    return fail(JEPA_E_OOM, "workspace: cudaMalloc(%zu bytes) failed: %s", need, cudaGetErrorString(e));
  }
  c->ws_bytes = need;
  ws_layout(m, rows, prows, g.Np, pix, c);
  e = cudaStreamCreateWithFlags(&c->stream, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    cudaFree(c->ws);
    delete c;
    return fail(JEPA_E_CUDA, "cudaStreamCreate: %s", cudaGetErrorString(e));
  }
  c->own_stream = true;
  // the side stream of the two-half encode; without it every batch runs as one lane
  if (m->dtype == JEPA_BF16 && max_batch >= kSplitMin) {
    if (cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&c->fork_ev, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c->join_ev, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      if (c->side) cudaStreamDestroy(c->side);
      if (c->fork_ev) cudaEventDestroy(c->fork_ev);
      c->side = nullptr;
      c->fork_ev = c->join_ev = nullptr;
    }
  }
  cudaMemset(c->err, 0, sizeof(int));
  *out = c;
  return JEPA_OK;
}

extern "C" void jepa_context_free(jepa_context* c) {
  if (!c) return;
  cudaSetDevice(c->m->device);
  if (c->stream) cudaStreamSynchronize(c->stream);
  if (c->hp_ready) {
    cudaStreamSynchronize(c->hp_up);
    cudaStreamSynchronize(c->hp_down);
    for (int s = 0; s < 2; ++s) {
      cudaFree(c->hp_pix[s]);
      cudaFree(c->hp_tok[s]);
      cudaEventDestroy(c->hp_uploaded[s]);
      cudaEventDestroy(c->hp_pix_free[s]);
      cudaEventDestroy(c->hp_tok_ready[s]);
      cudaEventDestroy(c->hp_downloaded[s]);
    }
    cudaStreamDestroy(c->hp_up);
    cudaStreamDestroy(c->hp_down);
  }
  if (c->gexec) cudaGraphExecDestroy(c->gexec);
  for (cudaEvent_t e : c->ev_pool) cudaEventDestroy(e);
  for (cudaEvent_t e : c->gev) cudaEventDestroy(e);
  if (c->side) {
    cudaStreamSynchronize(c->side);
    cudaStreamDestroy(c->side);
    cudaEventDestroy(c->fork_ev);
    cudaEventDestroy(c->join_ev);
  }
  if (c->own_stream && c->stream) cudaStreamDestroy(c->stream);
  if (c->ws) cudaFree(c->ws);
  delete c;
}

extern "C" jepa_status jepa_context_set_stream(jepa_context* c, void* stream) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_context_set_stream: null context");
  CUDA_TRY(cudaSetDevice(c->m->device));
  CUDA_TRY(cudaStreamSynchronize(c->stream));
  if (c->own_stream) cudaStreamDestroy(c->stream);
  c->stream = reinterpret_cast<cudaStream_t>(stream);
  c->own_stream = false;
  if (c->gexec) {  // a graph recorded for another stream is dropped
    cudaGraphExecDestroy(c->gexec);
    c->gexec = nullptr;
  }
  return JEPA_OK;
}

extern "C" jepa_status jepa_context_set_graph(jepa_context* c, int32_t enable) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_context_set_graph: null context");
  c->use_graph = enable != 0;
  return JEPA_OK;
}

extern "C" jepa_status jepa_context_set_pdl(jepa_context* c, int32_t enable) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_context_set_pdl: null context");
  c->use_pdl = enable != 0;
  return JEPA_OK;
}

extern "C" jepa_status jepa_context_workspace_bytes(const jepa_context* c, size_t* out) {
  if (!c || !out) return fail(JEPA_E_INVALID_ARG, "jepa_context_workspace_bytes: null argument");
  *out = c->ws_bytes;
  return JEPA_OK;
}

extern "C" jepa_status jepa_context_max_batch(const jepa_context* c, int32_t* out) {
  if (!c || !out) return fail(JEPA_E_INVALID_ARG, "jepa_context_max_batch: null argument");
  *out = c->max_B;
  return JEPA_OK;
}

namespace {
int launches_per_encode(const jepa_model* m) {
  return 2 + (m->hp.cls_token ? 1 : 0) + 7 * m->hp.n_layer + 1;
}

jepa_status check_shape(jepa_context* c, const float* pix, int B, int T, int H, int W, int layout, const void* tok,
                        Geo* g) {
  if (!pix || !tok) return fail(JEPA_E_INVALID_ARG, "jepa_encode: null pixel or token pointer");
  if (layout != JEPA_LAYOUT_TCHW && layout != JEPA_LAYOUT_CTHW) return fail(JEPA_E_INVALID_ARG, "layout %d unknown", layout);
  if (B <= 0) return fail(JEPA_E_INVALID_ARG, "batch %d must be positive", B);
  jepa_status st = geometry(&c->m->hp, T, H, W, g);
  if (st != JEPA_OK) return st;
  if (B > c->max_B || T > c->max_T || H > c->max_H || W > c->max_W || (long long)B * g->N > c->max_rows ||
      (long long)B * g->Np > c->max_prows)
    return fail(JEPA_E_BUDGET, "clip batch %d x %dx%dx%d exceeds the context's maximum %d x %dx%dx%d", B, T, H, W,
                c->max_B, c->max_T, c->max_H, c->max_W);
  if (c->m->hp.pos_type == JEPA_POS_LEARNED && g->N != c->m->hp.n_pos_rows)
    return fail(JEPA_E_UNSUPPORTED, "learned position table has %d rows, the clip has %d tokens", c->m->hp.n_pos_rows,
                g->N);
  if (c->m->hp.pos_type == JEPA_POS_SINCOS2D && g->gt != 1)
    return fail(JEPA_E_UNSUPPORTED, "a 2-D sin-cos table serves single-frame clips (the clip has %d)", g->gt);
  return JEPA_OK;
}

// Per-shape set-up: tensor maps over the workspace, GEMM tile widths, the RoPE table.
// The rows of items [item0, item0 + B) in every workspace buffer, tensor maps over them and the
// GEMM tile widths for their row count.
bool build_lane(jepa_context* c, jepa_context::Lane* ln, int item0, int B, const Geo& g) {
  const jepa_model* m = c->m;
  const int D = m->hp.embed_dim, F = m->hp.ffn_dim;
  const size_t es = m->dtype == JEPA_BF16 ? 2 : 4;
  const long long r0 = (long long)item0 * g.N, p0 = (long long)item0 * g.Np;
  const long long M = (long long)B * g.N, Mp = (long long)B * g.Np;
  ln->item0 = item0;
  ln->B = B;
  ln->X = c->X + r0 * D;
  ln->Xn = static_cast<uint8_t*>(c->Xn) + r0 * D * es;
  ln->qkv = static_cast<uint8_t*>(c->qkv) + r0 * 3 * D * es;
  ln->ao = static_cast<uint8_t*>(c->ao) + r0 * D * es;
  ln->Hh = static_cast<uint8_t*>(c->Hh) + r0 * F * es;
  ln->Pm = static_cast<uint8_t*>(c->Pm) + p0 * m->K * es;
  if (m->dtype != JEPA_BF16) return true;
  bool ok = true;
  ok &= make_tmap_2d_bf16(&ln->tm_Pm, ln->Pm, Mp, m->K, 128);
  ok &= make_tmap_2d_bf16(&ln->tm_Xn, ln->Xn, M, D, 128);
  ok &= make_tmap_2d_bf16(&ln->tm_ao, ln->ao, M, D, 128);
  ok &= make_tmap_2d_bf16(&ln->tm_Hh, ln->Hh, M, F, 128);
  ok &= make_tmap_3d_bf16(&ln->tm_qkv3, ln->qkv, B, g.N, 3 * D, 128);
  ok &= make_tmap_2d_out(&ln->tm_o_qkv, ln->qkv, M, 3 * D, 2);
  ok &= make_tmap_2d_out(&ln->tm_o_hh, ln->Hh, M, F, 2);
  ok &= make_tmap_2d_out(&ln->tm_o_x, ln->X, M, D, 4);
  ln->bn_patch = gemm_tc_pick_bn((int)Mp, D);
  ln->bn_qkv = gemm_tc_pick_bn((int)M, 3 * D);
  ln->bn_out = gemm_tc_pick_bn((int)M, D);
  ln->bn_up = gemm_tc_pick_bn((int)M, F);
  ln->bn_down = gemm_tc_pick_bn((int)M, D);
  return ok;
}

jepa_status prepare_shape(jepa_context* c, int B, int T, int H, int W, const Geo& g) {
  if (c->kB == B && c->kT == T && c->kH == H && c->kW == W) return JEPA_OK;
  const jepa_model* m = c->m;
  const jepa_hparams& hp = m->hp;
  const int D = hp.embed_dim;
  c->kB = -1;  // set again once everything below has succeeded
  bool ok = build_lane(c, &c->lanes[0], 0, B, g);
  c->halves = m->dtype == JEPA_BF16 && c->side != nullptr && B >= kSplitMin;
  if (c->halves) {
    const int B1 = (B + 1) / 2;
    ok &= build_lane(c, &c->lanes[1], 0, B1, g);
    ok &= build_lane(c, &c->lanes[2], B1, B - B1, g);
  }
  if (!ok) return fail(JEPA_E_CUDA, "cuTensorMapEncodeTiled refused a workspace tensor map");
  if (hp.pos_type == JEPA_POS_ROPE3D) {
    CUDA_TRY(rope_axes_launch(g.gt, g.gh, g.gw, D / hp.n_head, hp.rope_theta, hp.rope_interpolate,
                              hp.rope_ref_grid, c->rope, c->stream));
  }
  c->pos_clip = m->pos;
  if (is_sincos(hp)) {  // the training-grid table, resized when the clip's grid differs
    int gt0, gh0, gw0;
    sincos_train_grid(hp, &gt0, &gh0, &gw0);
    if (g.gt != gt0 || g.gh != gh0 || g.gw != gw0) {
      const int mode = hp.pos_type == JEPA_POS_SINCOS3D ? JEPA_RESIZE_TRILINEAR : JEPA_RESIZE_BICUBIC;
      CUDA_TRY(pos_resize_launch(m->pos, gt0, gh0, gw0, D, mode, c->pos_buf, g.gt, g.gh, g.gw, c->stream));
      c->pos_clip = c->pos_buf;
    }
  }
  c->kB = B;
  c->kT = T;
  c->kH = H;
  c->kW = W;
  return JEPA_OK;
}

EpiArgs make_epi(int kind, int M, int N, const float* bias, void* out) {
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

// Kernel classes of the profiling hook.
enum ProfClass { kPPatchify, kPGemmPatch, kPPrefix, kPLn, kPGemmQkv, kPAttention, kPGemmOut, kPGemmUp, kPGemmDown,
                 kPLnFinal, kPClasses };
const char* kProfNames[kPClasses] = {"patchify", "gemm_patch", "prefix_rows", "layernorm", "gemm_qkv",
                                     "attention", "gemm_out", "gemm_up", "gemm_down", "layernorm_final"};

size_t prof_event(jepa_context* c) {
  if (c->capturing) return c->gev_used < c->gev.size() ? c->gev_used++ : (size_t)-1;  // created before capture
  if (c->ev_used == c->ev_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return (size_t)-1;
    c->ev_pool.push_back(e);
  }
  return c->ev_used++;
}

// Runs `launch`, bracketed by two events when profiling is on.
template <class F>
cudaError_t prof(jepa_context* c, int cls, double flops, double bytes, F&& launch) {
  if (!c->profiling) return launch();
  const size_t e0 = prof_event(c), e1 = prof_event(c);
  if (e0 == (size_t)-1 || e1 == (size_t)-1) return cudaErrorMemoryAllocation;
  std::vector<cudaEvent_t>& pool = c->capturing ? c->gev : c->ev_pool;
  // inside a capture the records become external event nodes, re-recorded by every replay
  const unsigned flags = c->capturing ? cudaEventRecordExternal : cudaEventRecordDefault;
  cudaEventRecordWithFlags(pool[e0], c->stream, flags);
  const cudaError_t r = launch();
  cudaEventRecordWithFlags(pool[e1], c->stream, flags);
  (c->capturing ? c->grecs : c->recs).push_back({cls, e0, e1, flops, bytes});
  return r;
}

// Adds the durations of the last graph replay's recorded events to the accumulators.
cudaError_t fold_graph_events(jepa_context* c) {
  if (!c->gpending) return cudaSuccess;
  c->gpending = false;  // folded at most once, even when the driver refuses the timing
  cudaError_t e = cudaStreamSynchronize(c->stream);
  if (e != cudaSuccess) return e;
  for (const auto& r : c->grecs) {
    float ms = 0.0f;
    e = cudaEventElapsedTime(&ms, c->gev[r.e0], c->gev[r.e1]);
    if (e != cudaSuccess) return e;
    c->prof_launches[r.cls] += 1;
    c->prof_ms[r.cls] += ms;
    c->prof_flops[r.cls] += r.flops;
    c->prof_bytes[r.cls] += r.bytes;
  }
  c->gpending = false;
  return cudaSuccess;
}

// Visible (query, key) pairs of one item: N^2 for full attention; for block-causal, every
// patch query of frame f sees the (f + 1) frame_tokens patch keys before it, a prefix row sees N.
double visible_pairs(int attn_mode, int prefix, int frames, int frame_tokens, int N) {
  if (attn_mode == 0) return (double)N * N;
  double v = (double)prefix * N;
  for (int f = 0; f < frames; ++f) v += (double)frame_tokens * (f + 1) * frame_tokens;
  return v;
}

// The launch sequence of one encode (no host synchronisation inside: graph-capturable).
// The encode of one lane (its items' pixels in, their tokens out) on stream s.
jepa_status encode_lane(jepa_context* c, const jepa_context::Lane& ln, cudaStream_t s, const float* pix, int T, int H,
                        int W, int layout, float* tok, const Geo& g) {
  const jepa_model* m = c->m;
  const int B = ln.B;
  const jepa_hparams& hp = m->hp;
  const bool bf = m->dtype == JEPA_BF16;
  const int D = hp.embed_dim, F = hp.ffn_dim, L = hp.n_layer, NH = hp.n_head, hd = D / NH;
  const int M = B * g.N, Mp = B * g.Np;
  const uint64_t lim = default_wait_limit_ns();
  const double es = bf ? 2.0 : 4.0;                       // bytes of a GEMM operand element
  const double dM = M, dMp = Mp, dD = D, dF = F, dK = m->K;
  const double ln_bytes = dM * dD * (4.0 + es);           // read X fp32, write the normalised rows
  const double attn_flops = 4.0 * hd * NH * B *
                            visible_pairs(hp.attn_mode, g.prefix, g.gt, g.gh * g.gw, g.N);

  CUDA_TRY(prof(c, kPPatchify, 0.0, (double)B * T * hp.in_chans * H * W * 4.0 + dMp * dK * es, [&] {
    return patchify_launch(pix, B, T, hp.in_chans, H, W, hp.tubelet_size, hp.patch_size, layout, bf, ln.Pm, s);
  }));
  EpiArgs pe = make_epi(kEpiPatch, Mp, D, m->b_patch, ln.X);
  pe.patches_per_item = g.Np;
  pe.rows_per_item = g.N;
  pe.prefix = g.prefix;
  pe.pos = c->pos_clip;
  pe.vec = m->mod;
  CUDA_TRY(prof(c, kPGemmPatch, 2.0 * dMp * dD * dK, 0.0, [&] {
    return bf ? gemm_tc_launch(ln.tm_Pm, m->tm_patch[bn_slot(ln.bn_patch)], ln.tm_o_x, ln.bn_patch, pe, Mp, D, m->K, c->err, lim, s)
              : gemm_simt_launch(reinterpret_cast<const float*>(ln.Pm), reinterpret_cast<const float*>(m->w_patch), pe,
                                 Mp, D, m->K, s);
  }));
  if (g.prefix)
    CUDA_TRY(prof(c, kPPrefix, 0.0, (double)B * D * 4.0,
                  [&] { return prefix_rows_launch(ln.X, B, g.N, D, m->cls, m->pos, m->mod, s); }));

  AttnParams ap;
  ap.B = B;
  ap.N = g.N;
  ap.H = NH;
  ap.head_dim = hd;
  ap.attn_mode = hp.attn_mode;
  ap.prefix = g.prefix;
  ap.frame_tokens = g.gh * g.gw;
  ap.out = ln.ao;
  ap.qkv = ln.qkv;

  for (int l = 0; l < L; ++l) {
    const LayerW& w = m->layers[l];
    CUDA_TRY(prof(c, kPLn, 0.0, ln_bytes,
                  [&] { return layernorm_launch(ln.X, M, D, w.ln1_w, w.ln1_b, hp.ln_eps, bf, ln.Xn, s); }));
    EpiArgs qe = make_epi(kEpiQkvRope, M, 3 * D, w.b_qkv, ln.qkv);
    qe.rows_per_item = g.N;
    qe.prefix = g.prefix;
    qe.n_head = NH;
    qe.head_dim = hd;
    qe.rope_layout = hp.rope_layout;
    qe.rope_d = rope_d(hd);
    qe.rope_axes = hp.pos_type == JEPA_POS_ROPE3D ? c->rope : nullptr;
    qe.rope_gt = g.gt;
    qe.rope_gh = g.gh;
    qe.rope_gw = g.gw;
    EpiArgs oe = make_epi(kEpiResidual, M, D, w.b_out, ln.X);
    EpiArgs ue = make_epi(kEpiGelu, M, F, w.b_up, ln.Hh);
    EpiArgs de = make_epi(kEpiResidual, M, D, w.b_down, ln.X);
    const float* Xn = reinterpret_cast<const float*>(ln.Xn);
    CUDA_TRY(prof(c, kPGemmQkv, 2.0 * dM * 3.0 * dD * dD, 0.0, [&] {
      return bf ? gemm_tc_launch(ln.tm_Xn, w.tm_qkv[bn_slot(ln.bn_qkv)], ln.tm_o_qkv, ln.bn_qkv, qe, M, 3 * D, D, c->err, lim, s)
                : gemm_simt_launch(Xn, reinterpret_cast<const float*>(w.w_qkv), qe, M, 3 * D, D, s);
    }));
    CUDA_TRY(prof(c, kPAttention, attn_flops, 0.0, [&] {
      return bf ? attention_tc_launch(ln.tm_qkv3, ap, c->err, lim, s)
                : attention_simt_launch(reinterpret_cast<const float*>(ln.qkv), ap, s);
    }));
    CUDA_TRY(prof(c, kPGemmOut, 2.0 * dM * dD * dD, 0.0, [&] {
      return bf ? gemm_tc_launch(ln.tm_ao, w.tm_out[bn_slot(ln.bn_out)], ln.tm_o_x, ln.bn_out, oe, M, D, D, c->err, lim, s)
                : gemm_simt_launch(reinterpret_cast<const float*>(ln.ao), reinterpret_cast<const float*>(w.w_out), oe,
                                   M, D, D, s);
    }));
    CUDA_TRY(prof(c, kPLn, 0.0, ln_bytes,
                  [&] { return layernorm_launch(ln.X, M, D, w.ln2_w, w.ln2_b, hp.ln_eps, bf, ln.Xn, s); }));
    CUDA_TRY(prof(c, kPGemmUp, 2.0 * dM * dF * dD, 0.0, [&] {
      return bf ? gemm_tc_launch(ln.tm_Xn, w.tm_up[bn_slot(ln.bn_up)], ln.tm_o_hh, ln.bn_up, ue, M, F, D, c->err, lim, s)
                : gemm_simt_launch(Xn, reinterpret_cast<const float*>(w.w_up), ue, M, F, D, s);
    }));
    CUDA_TRY(prof(c, kPGemmDown, 2.0 * dM * dD * dF, 0.0, [&] {
      return bf ? gemm_tc_launch(ln.tm_Hh, w.tm_down[bn_slot(ln.bn_down)], ln.tm_o_x, ln.bn_down, de, M, D, F, c->err, lim, s)
                : gemm_simt_launch(reinterpret_cast<const float*>(ln.Hh), reinterpret_cast<const float*>(w.w_down), de,
                                   M, D, F, s);
    }));
  }
  CUDA_TRY(prof(c, kPLnFinal, 0.0, dM * dD * 8.0,
                [&] { return layernorm_launch(ln.X, M, D, m->norm_w, m->norm_b, hp.ln_eps, false, tok, s); }));
  return JEPA_OK;
}

jepa_status launch_encode(jepa_context* c, const float* pix, int B, int T, int H, int W, int layout, float* tok,
                          const Geo& g) {
  // programmatic launches for this sequence (not between profiling events)
  struct PdlScope {
    bool prev;
    explicit PdlScope(bool on) : prev(pdl_launches()) { pdl_launches() = on; }
    ~PdlScope() { pdl_launches() = prev; }
  } pdl_scope(c->use_pdl && !c->profiling);
  (void)B;  // the lanes were set up for this batch by prepare_shape
  if (!c->halves || c->profiling) return encode_lane(c, c->lanes[0], c->stream, pix, T, H, W, layout, tok, g);
  // two halves: the second on the side stream, forked from and joined back into the context
  // stream (inside a capture the side stream joins the capture through the fork event)
  const size_t pix_item = (size_t)T * c->m->hp.in_chans * H * W;
  const size_t tok_item = (size_t)g.N * c->m->hp.embed_dim;
  const jepa_context::Lane& b = c->lanes[2];
  CUDA_TRY(cudaEventRecord(c->fork_ev, c->stream));
  CUDA_TRY(cudaStreamWaitEvent(c->side, c->fork_ev, 0));
  jepa_status st = encode_lane(c, c->lanes[1], c->stream, pix, T, H, W, layout, tok, g);
  const jepa_status st2 =
      encode_lane(c, b, c->side, pix + b.item0 * pix_item, T, H, W, layout, tok + b.item0 * tok_item, g);
  // join even after a failed launch, so that a capture in progress can end
  CUDA_TRY(cudaEventRecord(c->join_ev, c->side));
  CUDA_TRY(cudaStreamWaitEvent(c->stream, c->join_ev, 0));
  return st != JEPA_OK ? st : st2;
}

}  // namespace

extern "C" jepa_status jepa_context_launches(const jepa_context* c, int32_t B, int32_t T, int32_t H, int32_t W,
                                             int32_t* n_out) {
  if (!c || !n_out) return fail(JEPA_E_INVALID_ARG, "jepa_context_launches: null argument");
  if (B <= 0) return fail(JEPA_E_INVALID_ARG, "batch %d must be positive", B);
  Geo g;
  jepa_status st = geometry(&c->m->hp, T, H, W, &g);
  if (st != JEPA_OK) return st;
  // a batch that runs as two halves launches every kernel of the sequence once per half
  const bool halves = c->m->dtype == JEPA_BF16 && c->side != nullptr && B >= kSplitMin && !c->profiling;
  *n_out = launches_per_encode(c->m) * (halves ? 2 : 1);
  return JEPA_OK;
}

extern "C" jepa_status jepa_encode(jepa_context* c, const float* d_pixels, int32_t B, int32_t T, int32_t H,
                                   int32_t W, int32_t layout, float* d_tokens) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_encode: null context");
  Geo g;
  jepa_status st = check_shape(c, d_pixels, B, T, H, W, layout, d_tokens, &g);
  if (st != JEPA_OK) return st;
  CUDA_TRY(cudaSetDevice(c->m->device));
  st = prepare_shape(c, B, T, H, W, g);
  if (st != JEPA_OK) return st;
  if (!c->use_graph) return launch_encode(c, d_pixels, B, T, H, W, layout, d_tokens, g);

  CUDA_TRY(fold_graph_events(c));  // the previous replay's events are about to be re-recorded
  const bool hit = c->gexec && c->gB == B && c->gT == T && c->gH == H && c->gW == W && c->glayout == layout &&
                   c->gpix == d_pixels && c->gtok == d_tokens && c->gprof == c->profiling && c->gpdl == c->use_pdl;
  if (!hit) {
    if (c->gexec) {
      cudaGraphExecDestroy(c->gexec);
      c->gexec = nullptr;
    }
    c->grecs.clear();
    c->gev_used = 0;
    if (c->profiling) {  // two events per launch, created outside the capture
      const size_t need = 2 * (size_t)launches_per_encode(c->m);
      while (c->gev.size() < need) {
        cudaEvent_t e;
        CUDA_TRY(cudaEventCreate(&e));
        c->gev.push_back(e);
      }
    }
    cudaGraph_t graph = nullptr;
    CUDA_TRY(cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal));
    c->capturing = true;
    st = launch_encode(c, d_pixels, B, T, H, W, layout, d_tokens, g);
    c->capturing = false;
    cudaError_t e = cudaStreamEndCapture(c->stream, &graph);
    if (st != JEPA_OK) {
      if (graph) cudaGraphDestroy(graph);
      return st;
    }
    if (e != cudaSuccess) return fail(JEPA_E_CUDA, "graph capture: %s", cudaGetErrorString(e));
    e = cudaGraphInstantiate(&c->gexec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return fail(JEPA_E_CUDA, "graph instantiate: %s", cudaGetErrorString(e));
    c->gB = B;
    c->gT = T;
    c->gH = H;
    c->gW = W;
    c->glayout = layout;
    c->gpix = d_pixels;
    c->gtok = d_tokens;
    c->gprof = c->profiling;
    c->gpdl = c->use_pdl;
  }
  CUDA_TRY(cudaGraphLaunch(c->gexec, c->stream));
  c->gpending = c->gprof;
  return JEPA_OK;
}

extern "C" jepa_status jepa_encode_host(jepa_context* c, const float* h_pixels, int32_t B, int32_t T, int32_t H,
                                        int32_t W, int32_t layout, float* h_tokens) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_encode_host: null context");
  Geo g;
  jepa_status st = check_shape(c, h_pixels, B, T, H, W, layout, h_tokens, &g);
  if (st != JEPA_OK) return st;
  CUDA_TRY(cudaSetDevice(c->m->device));
  const size_t pix_bytes = (size_t)B * T * c->m->hp.in_chans * H * W * sizeof(float);
  const size_t tok_bytes = (size_t)B * g.N * c->m->hp.embed_dim * sizeof(float);
  CUDA_TRY(cudaMemcpyAsync(c->pix_stage, h_pixels, pix_bytes, cudaMemcpyHostToDevice, c->stream));
  st = jepa_encode(c, c->pix_stage, B, T, H, W, layout, c->tok_stage);
  if (st != JEPA_OK) return st;
  CUDA_TRY(cudaMemcpyAsync(h_tokens, c->tok_stage, tok_bytes, cudaMemcpyDeviceToHost, c->stream));
  return jepa_context_sync(c);
}

namespace {
jepa_status host_pipeline_init(jepa_context* c) {
  if (c->hp_ready) return JEPA_OK;
  const size_t pix_bytes = (size_t)c->max_pix * sizeof(float);
  const size_t tok_bytes = (size_t)c->max_rows * c->m->hp.embed_dim * sizeof(float);
  for (int s = 0; s < 2; ++s) {
    if (cudaMalloc(&c->hp_pix[s], pix_bytes) != cudaSuccess || cudaMalloc(&c->hp_tok[s], tok_bytes) != cudaSuccess) {
      cudaGetLastError();
      for (int t = 0; t <= s; ++t) {
        cudaFree(c->hp_pix[t]);
        cudaFree(c->hp_tok[t]);
        c->hp_pix[t] = c->hp_tok[t] = nullptr;
      }
      return fail(JEPA_E_OOM, "pipelined host encode: cudaMalloc of 2 x (%zu + %zu) bytes failed", pix_bytes,
                  tok_bytes);
    }
  }
  CUDA_TRY(cudaStreamCreateWithFlags(&c->hp_up, cudaStreamNonBlocking));
  CUDA_TRY(cudaStreamCreateWithFlags(&c->hp_down, cudaStreamNonBlocking));
  for (int s = 0; s < 2; ++s) {
    CUDA_TRY(cudaEventCreateWithFlags(&c->hp_uploaded[s], cudaEventDisableTiming));
    CUDA_TRY(cudaEventCreateWithFlags(&c->hp_pix_free[s], cudaEventDisableTiming));
    CUDA_TRY(cudaEventCreateWithFlags(&c->hp_tok_ready[s], cudaEventDisableTiming));
    CUDA_TRY(cudaEventCreateWithFlags(&c->hp_downloaded[s], cudaEventDisableTiming));
    // recorded once on the idle streams so that the first waits on them pass
    CUDA_TRY(cudaEventRecord(c->hp_pix_free[s], c->stream));
    CUDA_TRY(cudaEventRecord(c->hp_downloaded[s], c->hp_down));
  }
  c->hp_ready = true;
  return JEPA_OK;
}
}  // namespace

extern "C" jepa_status jepa_encode_host_async(jepa_context* c, const float* h_pixels, int32_t B, int32_t T,
                                              int32_t H, int32_t W, int32_t layout, float* h_tokens) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_encode_host_async: null context");
  Geo g;
  jepa_status st = check_shape(c, h_pixels, B, T, H, W, layout, h_tokens, &g);
  if (st != JEPA_OK) return st;
  CUDA_TRY(cudaSetDevice(c->m->device));
  st = host_pipeline_init(c);
  if (st != JEPA_OK) return st;
  const int s = (int)(c->hp_step & 1);
  const size_t pix_bytes = (size_t)B * T * c->m->hp.in_chans * H * W * sizeof(float);
  const size_t tok_bytes = (size_t)B * g.N * c->m->hp.embed_dim * sizeof(float);
  // upload into slot s once the encode two steps back has taken its pixels out of it
  CUDA_TRY(cudaStreamWaitEvent(c->hp_up, c->hp_pix_free[s], 0));
  CUDA_TRY(cudaMemcpyAsync(c->hp_pix[s], h_pixels, pix_bytes, cudaMemcpyHostToDevice, c->hp_up));
  CUDA_TRY(cudaEventRecord(c->hp_uploaded[s], c->hp_up));
  // the encode reads its own staging buffers (one captured graph serves every step)
  CUDA_TRY(cudaStreamWaitEvent(c->stream, c->hp_uploaded[s], 0));
  CUDA_TRY(cudaMemcpyAsync(c->pix_stage, c->hp_pix[s], pix_bytes, cudaMemcpyDeviceToDevice, c->stream));
  CUDA_TRY(cudaEventRecord(c->hp_pix_free[s], c->stream));
  st = jepa_encode(c, c->pix_stage, B, T, H, W, layout, c->tok_stage);
  if (st != JEPA_OK) return st;
  CUDA_TRY(cudaStreamWaitEvent(c->stream, c->hp_downloaded[s], 0));  // slot s's last download is done
  CUDA_TRY(cudaMemcpyAsync(c->hp_tok[s], c->tok_stage, tok_bytes, cudaMemcpyDeviceToDevice, c->stream));
  CUDA_TRY(cudaEventRecord(c->hp_tok_ready[s], c->stream));
  CUDA_TRY(cudaStreamWaitEvent(c->hp_down, c->hp_tok_ready[s], 0));
  CUDA_TRY(cudaMemcpyAsync(h_tokens, c->hp_tok[s], tok_bytes, cudaMemcpyDeviceToHost, c->hp_down));
  CUDA_TRY(cudaEventRecord(c->hp_downloaded[s], c->hp_down));
  ++c->hp_step;
  return JEPA_OK;
}

extern "C" jepa_status jepa_context_sync(jepa_context* c) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_context_sync: null context");
  CUDA_TRY(cudaSetDevice(c->m->device));
  CUDA_TRY(cudaStreamSynchronize(c->stream));
  if (c->hp_ready) {
    CUDA_TRY(cudaStreamSynchronize(c->hp_up));
    CUDA_TRY(cudaStreamSynchronize(c->hp_down));
  }
  int h_err = 0;
  CUDA_TRY(cudaMemcpy(&h_err, c->err, sizeof(int), cudaMemcpyDeviceToHost));
  if (h_err) {
    CUDA_TRY(cudaMemset(c->err, 0, sizeof(int)));
    return fail(JEPA_E_TIMEOUT, "a device-side wait gave up (error word %d)", h_err);
  }
  return JEPA_OK;
}

extern "C" jepa_status jepa_context_set_profiling(jepa_context* c, int32_t enable) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_context_set_profiling: null context");
  c->profiling = enable != 0;
  return JEPA_OK;
}

extern "C" jepa_status jepa_context_profile(jepa_context* c, jepa_kernel_stat* out, int32_t max, int32_t* n_out,
                                            int32_t reset) {
  if (!c || !n_out || (max > 0 && !out)) return fail(JEPA_E_INVALID_ARG, "jepa_context_profile: null argument");
  CUDA_TRY(cudaSetDevice(c->m->device));
  CUDA_TRY(cudaStreamSynchronize(c->stream));
  CUDA_TRY(fold_graph_events(c));
  for (const auto& r : c->recs) {
    float ms = 0.0f;
    CUDA_TRY(cudaEventElapsedTime(&ms, c->ev_pool[r.e0], c->ev_pool[r.e1]));
    c->prof_launches[r.cls] += 1;
    c->prof_ms[r.cls] += ms;
    c->prof_flops[r.cls] += r.flops;
    c->prof_bytes[r.cls] += r.bytes;
  }
  c->recs.clear();
  c->ev_used = 0;
  int n = 0;
  for (int k = 0; k < kPClasses; ++k) {
    if (!c->prof_launches[k]) continue;
    if (n < max) {
      jepa_kernel_stat& st = out[n];
      memset(&st, 0, sizeof st);
      snprintf(st.name, sizeof st.name, "%s", kProfNames[k]);
      st.launches = c->prof_launches[k];
      st.total_ms = (float)c->prof_ms[k];
      st.flops = c->prof_flops[k];
      st.bytes = c->prof_bytes[k];
    }
    ++n;
  }
  *n_out = n;
  if (reset) {
    for (int k = 0; k < kPClasses; ++k) {
      c->prof_launches[k] = 0;
      c->prof_ms[k] = c->prof_flops[k] = c->prof_bytes[k] = 0.0;
    }
  }
  return JEPA_OK;
}

// ------------------------------------------------------------------ stage entry points
namespace {
std::mutex g_op_mu;
int* g_op_err = nullptr;  // device error word of the stage entry points (one per process)

jepa_status op_err_word(int** out) {
  std::lock_guard<std::mutex> lk(g_op_mu);
  if (!g_op_err) {
    CUDA_TRY(cudaMalloc(&g_op_err, sizeof(int)));
    CUDA_TRY(cudaMemset(g_op_err, 0, sizeof(int)));
  }
  *out = g_op_err;
  return JEPA_OK;
}
}  // namespace

extern "C" jepa_status jepa_op_patchify(const float* d_pixels, int32_t B, int32_t T, int32_t C, int32_t H, int32_t W,
                                        int32_t tubelet, int32_t patch, int32_t layout, int32_t out_dtype, void* d_out,
                                        void* stream) {
  if (!d_pixels || !d_out) return fail(JEPA_E_INVALID_ARG, "jepa_op_patchify: null pointer");
  if (B <= 0 || T <= 0 || C <= 0 || H <= 0 || W <= 0 || tubelet <= 0 || patch <= 0)
    return fail(JEPA_E_INVALID_ARG, "jepa_op_patchify: non-positive size");
  if (T % tubelet || H % patch || W % patch) return fail(JEPA_E_INVALID_ARG, "jepa_op_patchify: sizes not divisible");
  if (layout != 0 && layout != 1) return fail(JEPA_E_INVALID_ARG, "layout %d unknown", layout);
  CUDA_TRY(patchify_launch(d_pixels, B, T, C, H, W, tubelet, patch, layout, out_dtype == JEPA_BF16, d_out,
                           reinterpret_cast<cudaStream_t>(stream)));
  return JEPA_OK;
}

extern "C" jepa_status jepa_op_layernorm(const float* d_x, int32_t M, int32_t D, const float* d_gamma,
                                         const float* d_beta, float eps, int32_t out_dtype, void* d_y, void* stream) {
  if (!d_x || !d_gamma || !d_beta || !d_y) return fail(JEPA_E_INVALID_ARG, "jepa_op_layernorm: null pointer");
  if (M < 0 || D <= 0 || D % 4 || D > 2048) return fail(JEPA_E_INVALID_ARG, "jepa_op_layernorm: bad size M %d D %d", M, D);
  CUDA_TRY(layernorm_launch(d_x, M, D, d_gamma, d_beta, eps, out_dtype == JEPA_BF16, d_y,
                            reinterpret_cast<cudaStream_t>(stream)));
  return JEPA_OK;
}

extern "C" jepa_status jepa_op_linear(int32_t dtype, const void* d_x, int32_t M, int32_t K, const void* d_w, int32_t N,
                                      const jepa_epilogue* epi, void* stream) {
  if (!d_x || !d_w || !epi || !epi->d_bias || !epi->d_out) return fail(JEPA_E_INVALID_ARG, "jepa_op_linear: null pointer");
  if (M < 0 || K <= 0 || N <= 0) return fail(JEPA_E_INVALID_ARG, "jepa_op_linear: bad size %d x %d x %d", M, K, N);
  if (epi->kind < 0 || epi->kind > JEPA_EPI_PATCH_EMBED) return fail(JEPA_E_INVALID_ARG, "epilogue kind %d", epi->kind);
  EpiArgs e = make_epi(epi->kind, M, N, epi->d_bias, epi->d_out);
  if (epi->kind == JEPA_EPI_QKV_ROPE) {
    if (epi->n_head <= 0 || epi->head_dim <= 0 || 3 * epi->n_head * epi->head_dim != N || epi->head_dim % 2 ||
        epi->rows_per_item <= 0 || epi->prefix < 0)
      return fail(JEPA_E_INVALID_ARG, "QKV_ROPE epilogue: inconsistent heads/rows");
    e.rope = reinterpret_cast<const float2*>(epi->d_rope);
    e.rope_ids = epi->d_rope_ids;
    e.rows_per_item = epi->rows_per_item;
    e.prefix = epi->prefix;
    e.n_head = epi->n_head;
    e.head_dim = epi->head_dim;
    e.rope_layout = epi->rope_layout;
    e.rope_d = rope_d(epi->head_dim);
  }
  if (epi->kind == JEPA_EPI_PATCH_EMBED) {
    if (epi->patches_per_item <= 0 || epi->rows_per_item < epi->patches_per_item + epi->prefix || epi->prefix < 0)
      return fail(JEPA_E_INVALID_ARG, "PATCH_EMBED epilogue: inconsistent rows");
    e.patches_per_item = epi->patches_per_item;
    e.rows_per_item = epi->rows_per_item;
    e.prefix = epi->prefix;
    e.pos = epi->d_pos;
    e.vec = epi->d_vec;
  }
  if (N % 4) return fail(JEPA_E_INVALID_ARG, "GEMM epilogues need N %% 4 == 0 (N %d)", N);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == JEPA_FP32) {
    CUDA_TRY(gemm_simt_launch(reinterpret_cast<const float*>(d_x), reinterpret_cast<const float*>(d_w), e, M, N, K, s));
    return JEPA_OK;
  }
  if (dtype != JEPA_BF16) return fail(JEPA_E_INVALID_ARG, "dtype %d unknown", dtype);
  if (K % 64 || N % 64) return fail(JEPA_E_UNSUPPORTED, "bf16 GEMM needs K %% 64 == 0 and N %% 64 == 0 (K %d, N %d)", K, N);
  if ((reinterpret_cast<uintptr_t>(d_x) | reinterpret_cast<uintptr_t>(d_w)) & 15)
    return fail(JEPA_E_INVALID_ARG, "bf16 GEMM operands must be 16-byte aligned");
  if (M == 0) return JEPA_OK;
  CUDA_TRY(tc_kernels_init());
  int* err = nullptr;
  jepa_status st = op_err_word(&err);
  if (st != JEPA_OK) return st;
  const int bn = gemm_tc_pick_bn(M, N);
  CUtensorMap ta, tb, to;
  if (!make_tmap_2d_bf16(&ta, d_x, M, K, 128) ||
      !make_tmap_2d_bf16(&tb, d_w, N, K, gemm_tc_b_box(bn)))
    return fail(JEPA_E_CUDA, "cuTensorMapEncodeTiled refused an operand");
  memset(&to, 0, sizeof to);
  // the patch embedding stores through TMA too when its rows are the patch rows themselves
  const bool patch_tma = e.kind == kEpiPatch && e.prefix == 0 && e.rows_per_item == e.patches_per_item;
  if (e.kind != kEpiPatch || patch_tma) {
    if (reinterpret_cast<uintptr_t>(e.out) & 15) return fail(JEPA_E_INVALID_ARG, "bf16 GEMM output must be 16-byte aligned");
    if (!make_tmap_2d_out(&to, e.out, M, N, (e.kind == kEpiResidual || e.kind == kEpiPatch) ? 4 : 2))
      return fail(JEPA_E_CUDA, "cuTensorMapEncodeTiled refused the output");
  }
  CUDA_TRY(gemm_tc_launch(ta, tb, to, bn, e, M, N, K, err, default_wait_limit_ns(), s));
  return JEPA_OK;
}

extern "C" jepa_status jepa_op_rope_table(const jepa_hparams* hp, int32_t T, int32_t H, int32_t W, float* d_table,
                                          void* stream) {
  if (!hp || !d_table) return fail(JEPA_E_INVALID_ARG, "jepa_op_rope_table: null pointer");
  jepa_status st = jepa_hparams_validate(hp);
  if (st != JEPA_OK) return st;
  Geo g;
  st = geometry(hp, T, H, W, &g);
  if (st != JEPA_OK) return st;
  CUDA_TRY(rope_table_launch(g.gt, g.gh, g.gw, hp->embed_dim / hp->n_head, hp->rope_theta, hp->rope_interpolate,
                             hp->rope_ref_grid, reinterpret_cast<float2*>(d_table), reinterpret_cast<cudaStream_t>(stream)));
  return JEPA_OK;
}

extern "C" jepa_status jepa_op_sincos_table(int32_t kind, int32_t gt, int32_t gh, int32_t gw, int32_t D,
                                            int32_t w_first, int32_t uniform_power, float* d_table, void* stream) {
  if (!d_table) return fail(JEPA_E_INVALID_ARG, "jepa_op_sincos_table: null pointer");
  if (kind != JEPA_POS_SINCOS2D && kind != JEPA_POS_SINCOS3D)
    return fail(JEPA_E_INVALID_ARG, "jepa_op_sincos_table: kind %d is not a sin-cos table", kind);
  const int k = kind == JEPA_POS_SINCOS3D ? 1 : 0;
  if (gt <= 0 || gh <= 0 || gw <= 0 || (k == 0 && gt != 1) || (long long)gt * gh * gw > (1ll << 22))
    return fail(JEPA_E_INVALID_ARG, "jepa_op_sincos_table: grid %dx%dx%d", gt, gh, gw);
  int d0, d1, d2;
  if (!sincos_widths(k, D, uniform_power, &d0, &d1, &d2))
    return fail(JEPA_E_INVALID_ARG, "jepa_op_sincos_table: width %d cannot be split", D);
  CUDA_TRY(sincos_table_launch(k, gt, gh, gw, D, w_first, uniform_power, d_table, reinterpret_cast<cudaStream_t>(stream)));
  return JEPA_OK;
}

extern "C" jepa_status jepa_op_pos_resize(const float* d_src, int32_t st, int32_t sh, int32_t sw, int32_t D,
                                          int32_t mode, float* d_dst, int32_t dt, int32_t dh, int32_t dw, void* stream) {
  if (!d_src || !d_dst) return fail(JEPA_E_INVALID_ARG, "jepa_op_pos_resize: null pointer");
  if (mode != JEPA_RESIZE_TRILINEAR && mode != JEPA_RESIZE_BICUBIC)
    return fail(JEPA_E_INVALID_ARG, "jepa_op_pos_resize: mode %d unknown", mode);
  if (st <= 0 || sh <= 0 || sw <= 0 || dt <= 0 || dh <= 0 || dw <= 0 || D <= 0 || D % 4)
    return fail(JEPA_E_INVALID_ARG, "jepa_op_pos_resize: bad size (%dx%dx%d -> %dx%dx%d, D %d)", st, sh, sw, dt, dh,
                dw, D);
  if (mode == JEPA_RESIZE_BICUBIC && st != dt)
    return fail(JEPA_E_INVALID_ARG, "jepa_op_pos_resize: bicubic resizes each frame (st %d != dt %d)", st, dt);
  if ((reinterpret_cast<uintptr_t>(d_src) | reinterpret_cast<uintptr_t>(d_dst)) & 15)
    return fail(JEPA_E_INVALID_ARG, "jepa_op_pos_resize: tables must be 16-byte aligned");
  const size_t sb = (size_t)st * sh * sw * D * 4, db = (size_t)dt * dh * dw * D * 4;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(d_src), d0 = reinterpret_cast<uintptr_t>(d_dst);
  if (s0 < d0 + db && d0 < s0 + sb) return fail(JEPA_E_INVALID_ARG, "jepa_op_pos_resize: source and output overlap");
  CUDA_TRY(pos_resize_launch(d_src, st, sh, sw, D, mode, d_dst, dt, dh, dw, reinterpret_cast<cudaStream_t>(stream)));
  return JEPA_OK;
}

extern "C" jepa_status jepa_op_attention(int32_t dtype, const void* d_qkv, int32_t B, int32_t N, int32_t n_head,
                                         int32_t head_dim, int32_t attn_mode, int32_t prefix, int32_t frame_tokens,
                                         void* d_out, void* stream) {
  if (!d_qkv || !d_out) return fail(JEPA_E_INVALID_ARG, "jepa_op_attention: null pointer");
  if (B <= 0 || N <= 0 || n_head <= 0) return fail(JEPA_E_INVALID_ARG, "jepa_op_attention: bad size");
  if (attn_mode != 0 && attn_mode != 1) return fail(JEPA_E_INVALID_ARG, "attn_mode %d unknown", attn_mode);
  if (attn_mode == 1 && (frame_tokens <= 0 || prefix < 0)) return fail(JEPA_E_INVALID_ARG, "block-causal needs frame_tokens > 0");
  if (head_dim != 64 && !(head_dim == 32 && dtype == JEPA_BF16))
    return fail(JEPA_E_UNSUPPORTED, "attention kernels are built for head_dim 64 (and 32 in bf16; got %d)", head_dim);
  AttnParams p;
  p.B = B;
  p.N = N;
  p.H = n_head;
  p.head_dim = head_dim;
  p.attn_mode = attn_mode;
  p.prefix = prefix;
  p.frame_tokens = frame_tokens;
  p.out = d_out;
  p.qkv = d_qkv;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == JEPA_FP32) {
    if ((reinterpret_cast<uintptr_t>(d_qkv) | reinterpret_cast<uintptr_t>(d_out)) & 15)
      return fail(JEPA_E_INVALID_ARG, "fp32 attention: qkv and out must be 16-byte aligned");
    CUDA_TRY(attention_simt_launch(reinterpret_cast<const float*>(d_qkv), p, s));
    return JEPA_OK;
  }
  if (dtype != JEPA_BF16) return fail(JEPA_E_INVALID_ARG, "dtype %d unknown", dtype);
  if (reinterpret_cast<uintptr_t>(d_qkv) & 15) return fail(JEPA_E_INVALID_ARG, "qkv must be 16-byte aligned");
  CUDA_TRY(tc_kernels_init());
  int* err = nullptr;
  jepa_status st = op_err_word(&err);
  if (st != JEPA_OK) return st;
  CUtensorMap tm;
  if (!make_tmap_3d_bf16(&tm, d_qkv, B, N, 3 * n_head * head_dim, 128, head_dim))
    return fail(JEPA_E_CUDA, "cuTensorMapEncodeTiled refused qkv");
  CUDA_TRY(attention_tc_launch(tm, p, err, default_wait_limit_ns(), s));
  return JEPA_OK;
}

extern "C" jepa_status jepa_device_status(void) {
  CUDA_TRY(cudaDeviceSynchronize());
  int* err = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_op_mu);
    err = g_op_err;
  }
  if (!err) return JEPA_OK;
  int h = 0;
  CUDA_TRY(cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost));
  if (h) {
    CUDA_TRY(cudaMemset(err, 0, sizeof(int)));
    return fail(JEPA_E_TIMEOUT, "a device-side wait gave up (error word %d)", h);
  }
  return JEPA_OK;
}

extern "C" jepa_status jepa_debug_wait_timeout(int32_t limit_us) {
  if (limit_us <= 0 || limit_us > 1000000) return fail(JEPA_E_INVALID_ARG, "limit_us %d outside (0, 1e6]", limit_us);
  int* err = nullptr;
  jepa_status st = op_err_word(&err);
  if (st != JEPA_OK) return st;
  CUDA_TRY(wait_timeout_probe_launch(err, (uint64_t)limit_us * 1000ull, nullptr));
  return jepa_device_status();
}

// ------------------------------------------------------------------ allocation-free encode
// For callers that cannot allocate device memory: the encode workspace lives in one fixed
// scratch array of this file instead of a context's cudaMalloc'd arena. The launch sequence is
// the one jepa_encode runs, over a jepa_context that only views the array.
namespace {
static __device__ __align__(256) uint8_t g_noalloc_scratch[JEPA_NOALLOC_SCRATCH_BYTES];
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
uint8_t* g_noalloc_base[kNoAllocMaxDevices] = {};  // the array's device address, per device

// Set-up, once per device with that device current: the host-side name of the array is only a
// stand-in, so its device address is looked up and kept.
jepa_status noalloc_scratch(int device, uint8_t** out) {
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_base[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return fail(JEPA_E_CUDA, "jepa_encode_noalloc: scratch array address on device %d: %s", device,
                  cudaGetErrorString(e));
    g_noalloc_base[device] = reinterpret_cast<uint8_t*>(p);
  }
  *out = g_noalloc_base[device];
  return JEPA_OK;
}
}  // namespace

extern "C" jepa_status jepa_encode_noalloc(const jepa_model* m, const float* d_pixels, int32_t B, int32_t T,
                                           int32_t H, int32_t W, int32_t layout, float* d_tokens, void* stream) {
  if (!m) return fail(JEPA_E_INVALID_ARG, "jepa_encode_noalloc: null model");
  if (!d_pixels || !d_tokens) return fail(JEPA_E_INVALID_ARG, "jepa_encode_noalloc: null pixel or token pointer");
  if (layout != JEPA_LAYOUT_TCHW && layout != JEPA_LAYOUT_CTHW) return fail(JEPA_E_INVALID_ARG, "layout %d unknown", layout);
  if (B <= 0) return fail(JEPA_E_INVALID_ARG, "batch %d must be positive", B);
  Geo g;
  jepa_status st = geometry(&m->hp, T, H, W, &g);
  if (st != JEPA_OK) return st;
  if (m->hp.pos_type == JEPA_POS_LEARNED && g.N != m->hp.n_pos_rows)
    return fail(JEPA_E_UNSUPPORTED, "learned position table has %d rows, the clip has %d tokens", m->hp.n_pos_rows, g.N);
  if (m->hp.pos_type == JEPA_POS_SINCOS2D && g.gt != 1)
    return fail(JEPA_E_UNSUPPORTED, "a 2-D sin-cos table serves single-frame clips (the clip has %d)", g.gt);
  if (m->device < 0 || m->device >= kNoAllocMaxDevices)
    return fail(JEPA_E_UNSUPPORTED, "jepa_encode_noalloc: device %d beyond %d", m->device, kNoAllocMaxDevices);
  const long long rows = (long long)B * g.N, prows = (long long)B * g.Np;
  const size_t need = ws_layout(m, rows, prows, g.Np, 0, nullptr);
  if (need > JEPA_NOALLOC_SCRATCH_BYTES)
    return fail(JEPA_E_BUDGET, "jepa_encode_noalloc: %d x %dx%dx%d needs %zu bytes of scratch, the array holds %llu",
                B, T, H, W, need, (unsigned long long)JEPA_NOALLOC_SCRATCH_BYTES);
  CUDA_TRY(cudaSetDevice(m->device));
  uint8_t* base = nullptr;
  st = noalloc_scratch(m->device, &base);
  if (st != JEPA_OK) return st;
  if (m->dtype == JEPA_BF16) CUDA_TRY(tc_kernels_init());

  jepa_context c;  // a view over the scratch array: owns nothing, frees nothing
  c.m = m;
  c.stream = reinterpret_cast<cudaStream_t>(stream);
  c.own_stream = false;
  c.max_B = B;
  c.max_T = T;
  c.max_H = H;
  c.max_W = W;
  c.max_rows = rows;
  c.max_prows = prows;
  c.max_np = g.Np;
  c.max_pix = 0;
  c.ws = base;
  c.ws_bytes = need;
  ws_layout(m, rows, prows, g.Np, 0, &c);
  CUDA_TRY(cudaMemsetAsync(c.err, 0, sizeof(int), c.stream));  // the array keeps the last call's word
  st = prepare_shape(&c, B, T, H, W, g);
  if (st != JEPA_OK) return st;
  st = launch_encode(&c, d_pixels, B, T, H, W, layout, d_tokens, g);
  if (st != JEPA_OK) return st;
  int h_err = 0;
  CUDA_TRY(cudaMemcpyAsync(&h_err, c.err, sizeof(int), cudaMemcpyDeviceToHost, c.stream));
  CUDA_TRY(cudaStreamSynchronize(c.stream));
  if (h_err) return fail(JEPA_E_TIMEOUT, "jepa_encode_noalloc: a device-side wait gave up (error word %d)", h_err);
  return JEPA_OK;
}
