// head.cu -- the attentive-pool head and classifier of the V-JEPA 2 video classifiers behind the
// jepa_head_* entry points, and token pooling (jepa_op_pool). ("GGUF schema (v1)", Head: head.*
// tensors; the SkyVision V-JEPA 2 notes, attentive pooler and classifier.) Launch sequence of one
// jepa_head_forward over B items of N encoder tokens:
//
//   per pooler layer (on a copy of the tokens): the encoder block without RoPE -- LN1 -> QKV GEMM
//              (+bias) -> attention -> out GEMM (+=X) -> LN2 -> up GEMM (GELU) -> down GEMM (+=X)
//   ln_kv LN -> K|V GEMM (the two projections as one [2D, D] weight)
//   query projection (one row) -> cross attention of the query over each item's tokens, + query
//   ln2 LN -> MLP up (GELU) -> MLP down (+ residual) = pooled -> classifier -> logits
//
// After the self-attention layers everything works on one row per item: those steps run on
// small SIMT kernels (a warp per output feature, the rows staged in shared memory, so the weights
// and the rows are read once per CTA), in fp32 with bf16 weights; the cross attention splits each
// item's keys over CTAs and merges their partial softmax sums.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"
#include "jepa.h"
#include "jepa_synth.h"
#include "kernels.h"
#include "ptx.cuh"
#include "seq.h"

using namespace jepa;

namespace {

__device__ __forceinline__ void bf16x8_to_f32(const uint4 w, float (&f)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
  }
}

// y[r, n] = act(sum_k x[r, k] W[n, k] + b[n]) (+ res[r, n]) for the R rows of x: a CTA of 8 warps
// takes 8 output features (warp w: feature n0 + w) and stages x in shared memory, 8 rows by 1024
// columns at a time, so each weight row is read once and x once per CTA. x fp32 [R, K], W bf16
// [N, K], K % 8 == 0; res may be y itself (each element is read and written by the same lane).
constexpr int kRvWarps = 8, kRvRows = 8, kRvChunk = 1024;
template <bool GELU>
__global__ void __launch_bounds__(32 * kRvWarps) rowvec_linear_kernel(const float* __restrict__ x, int R, int K,
                                                                      const __nv_bfloat16* __restrict__ W, int N,
                                                                      const float* __restrict__ bias, const float* res,
                                                                      float* y) {
  pdl_trigger();
  pdl_wait();
  __shared__ __align__(16) float xs[kRvRows][kRvChunk];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int n0 = blockIdx.x * kRvWarps; n0 < N; n0 += gridDim.x * kRvWarps) {  // uniform across the CTA
    const int n = n0 + warp;
    for (int r0 = 0; r0 < R; r0 += kRvRows) {
      const int rows = min(kRvRows, R - r0);
      float acc[kRvRows];
#pragma unroll
      for (int r = 0; r < kRvRows; ++r) acc[r] = 0.0f;
      for (int k0 = 0; k0 < K; k0 += kRvChunk) {
        const int kc = min(kRvChunk, K - k0), kc4 = kc / 4;
        __syncthreads();  // the previous chunk is no longer read
        for (int i = threadIdx.x; i < rows * kc4; i += blockDim.x) {
          const int r = i / kc4, c4 = i - r * kc4;
          reinterpret_cast<float4*>(xs[r])[c4] = __ldg(reinterpret_cast<const float4*>(x + (size_t)(r0 + r) * K + k0) + c4);
        }
        __syncthreads();
        if (n < N) {
          const __nv_bfloat16* w = W + (size_t)n * K + k0;
#pragma unroll 4  // several weight loads in flight per warp (one CTA per SM: latency-bound otherwise)
          for (int k = lane * 8; k < kc; k += 256) {
            float wf[8];
            bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(w + k)), wf);
#pragma unroll
            for (int r = 0; r < kRvRows; ++r) {
              if (r < rows) {
                const float4 a = *reinterpret_cast<const float4*>(&xs[r][k]);
                const float4 c = *reinterpret_cast<const float4*>(&xs[r][k + 4]);
                float t = acc[r];
                t = fmaf(a.x, wf[0], t);
                t = fmaf(a.y, wf[1], t);
                t = fmaf(a.z, wf[2], t);
                t = fmaf(a.w, wf[3], t);
                t = fmaf(c.x, wf[4], t);
                t = fmaf(c.y, wf[5], t);
                t = fmaf(c.z, wf[6], t);
                acc[r] = fmaf(c.w, wf[7], t);
              }
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kRvRows; ++r)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
      if (lane == 0 && n < N) {
        const float bn = __ldg(bias + n);
#pragma unroll
        for (int r = 0; r < kRvRows; ++r) {
          if (r < rows) {
            float v = acc[r] + bn;
            if (GELU) v = gelu_erf(v);
            if (res) v += res[(size_t)(r0 + r) * N + n];
            y[(size_t)(r0 + r) * N + n] = v;
          }
        }
      }
    }
  }
}

// Cross attention of one query row per head over the N tokens of each item, in two kernels. Part:
// CTA (h, b, s) takes keys [256 s, 256 s + 256) of item b: scores (eight lanes per key row, 16
// bytes each, so a warp reads four whole rows per load), their max m, p = exp(score - m), the sum
// l and o = sum p v; it writes (m, l, o[hd]). Combine: CTA (h, b) merges the S parts,
// O = sum_s o_s exp(m_s - M) / sum_s l_s exp(m_s - M) with M = max_s m_s, and writes
// out[b, h*hd + d] = query[h*hd + d] + O[d] (no output projection: the raw query is the residual).
// q fp32 [D] (projected query), kv bf16 [B*N, 2D] (keys in columns [0, D), values in [D, 2D)),
// hd in {32, 64, 128}.
constexpr int kXThreads = 256, kXKeys = 256;
__global__ void __launch_bounds__(kXThreads) xattn_part_kernel(const float* __restrict__ q,
                                                               const __nv_bfloat16* __restrict__ kv, int N, int D,
                                                               int hd, float* __restrict__ part) {
  pdl_trigger();
  pdl_wait();
  __shared__ float qh[128];
  __shared__ float sc[kXKeys];
  __shared__ float red[kXThreads];
  const int h = blockIdx.x, b = blockIdx.y, sidx = blockIdx.z, S = gridDim.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j0 = sidx * kXKeys, cnt = min(kXKeys, N - j0);
  if (tid < hd) qh[tid] = q[h * hd + tid] * rsqrtf((float)hd);
  __syncthreads();
  const __nv_bfloat16* base = kv + ((size_t)b * N + j0) * 2 * D + (size_t)h * hd;
  const int c = lane & 7;  // 16-byte chunk of the row: dims [8c, 8c + 8) (+ 64 for hd 128)
  for (int j = warp * 4 + (lane >> 3); j < kXKeys; j += kXThreads / 8) {
    float acc = 0.0f;
    if (j < cnt) {
      const uint4* kr = reinterpret_cast<const uint4*>(base + (size_t)j * 2 * D);
      for (int cc = c; cc * 8 < hd; cc += 8) {
        float kf[8];
        bf16x8_to_f32(__ldg(kr + cc), kf);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(qh[cc * 8 + e], kf[e], acc);
      }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    if (c == 0) sc[j] = j < cnt ? acc : -INFINITY;
  }
  __syncthreads();
  // max, then p = exp(s - m) and its sum, over the 256 slots (one per thread)
  float v = sc[tid], mx = v;
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  float m = red[0];
  for (int w = 1; w < kXThreads / 32; ++w) m = fmaxf(m, red[w]);
  const float p = tid < cnt ? expf(v - m) : 0.0f;
  float sum = p;
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  __syncthreads();  // red[] read by every thread above before it is reused
  sc[tid] = p;
  if (lane == 0) red[warp] = sum;
  __syncthreads();
  float l = 0.0f;
  for (int w = 0; w < kXThreads / 32; ++w) l += red[w];
  __syncthreads();
  // o = sum p v: thread (g, d) takes keys g, g + G, ... for value dim d (a row's dims are adjacent)
  const int G = kXThreads / hd, g = tid / hd, d = tid - g * hd;
  float acc = 0.0f;
  for (int j = g; j < cnt; j += G) acc = fmaf(sc[j], __bfloat162float(base[(size_t)j * 2 * D + D + d]), acc);
  red[tid] = acc;
  __syncthreads();
  float* out = part + (((size_t)b * gridDim.x + h) * S + sidx) * (hd + 2);
  if (tid < hd) {
    float o = 0.0f;
    for (int k = 0; k < G; ++k) o += red[k * hd + tid];
    out[2 + tid] = o;
  }
  if (tid == 0) {
    out[0] = m;
    out[1] = l;
  }
}

__global__ void xattn_combine_kernel(const float* __restrict__ part, int S, int hd, int D,
                                     const float* __restrict__ query, float* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const float* pp = part + ((size_t)b * gridDim.x + h) * S * (hd + 2);
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, pp[(size_t)s * (hd + 2)]);
  float L = 0.0f, O = 0.0f;
  for (int s = 0; s < S; ++s) {
    const float* ps = pp + (size_t)s * (hd + 2);
    const float w = expf(ps[0] - M);
    L = fmaf(ps[1], w, L);
    O = fmaf(ps[2 + d], w, O);
  }
  out[(size_t)b * D + h * hd + d] = query[h * hd + d] + O / L;
}

// out[b, :] = mean of rows [prefix, N) of item b (mode 0) or row 0 (mode 1); CTA (column block of
// 128, item b): 8 row groups x 32 column quads, partial sums added in shared memory (fixed order).
__global__ void pool_kernel(const float* __restrict__ x, int N, int D, int prefix, int mode, float* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  __shared__ float4 part[8][32];
  const int b = blockIdx.y, c4 = blockIdx.x * 32 + (threadIdx.x & 31), rg = threadIdx.x >> 5;
  const int D4 = D / 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (c4 < D4) {
    const float4* xb = reinterpret_cast<const float4*>(x + (size_t)b * N * D) + c4;
    if (mode == 1) {
      if (rg == 0) acc = __ldg(xb);
    } else {
      for (int n = prefix + rg; n < N; n += 8) {
        const float4 v = __ldg(xb + (size_t)n * D4);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
    }
  }
  part[rg][threadIdx.x & 31] = acc;
  __syncthreads();
  if (rg == 0 && c4 < D4) {
    float4 t = part[0][threadIdx.x];
    for (int k = 1; k < 8; ++k) {
      const float4 v = part[k][threadIdx.x];
      t.x += v.x;
      t.y += v.y;
      t.z += v.z;
      t.w += v.w;
    }
    const float sc = mode == 1 ? 1.0f : 1.0f / (float)(N - prefix);
    reinterpret_cast<float4*>(out + (size_t)b * D)[c4] = make_float4(t.x * sc, t.y * sc, t.z * sc, t.w * sc);
  }
}

cudaError_t rowvec_launch(const float* x, int R, int K, const void* W, int N, const float* bias, const float* res,
                          float* y, bool gelu, cudaStream_t s) {
  const int grid = std::max(1, std::min((N + kRvWarps - 1) / kRvWarps, num_sms() * 8));
  const __nv_bfloat16* w = reinterpret_cast<const __nv_bfloat16*>(W);
  return gelu ? launch_kernel(rowvec_linear_kernel<true>, dim3(grid), dim3(32 * kRvWarps), 0, s, x, R, K, w, N, bias,
                              res, y)
              : launch_kernel(rowvec_linear_kernel<false>, dim3(grid), dim3(32 * kRvWarps), 0, s, x, R, K, w, N, bias,
                              res, y);
}

constexpr int kXMaxTokens = 32768;
int xattn_splits(int N) { return (N + kXKeys - 1) / kXKeys; }

struct Rec {
  std::string name;
  size_t offset, n;
  bool bf16;
};
struct HeadLayer {
  const float *ln1_w, *ln1_b, *b_qkv, *b_out, *ln2_w, *ln2_b, *b_up, *b_down;
  const void *w_qkv, *w_out, *w_up, *w_down;
  CUtensorMap tm_qkv[3], tm_out[3], tm_up[3], tm_down[3];
};
int slot(int bn) { return bn == 64 ? 0 : ((bn == 128 || bn == kPairTile) ? 1 : 2); }

enum HeadClass { kHLn, kHQkv, kHAttn, kHOut, kHUp, kHDown, kHLnKv, kHKv, kHQuery, kHXattn, kHLn2, kHMlpUp, kHMlpDown,
                 kHCls, kHClasses };
const char* kHNames[kHClasses] = {"layernorm", "gemm_qkv", "attention", "gemm_out", "gemm_up", "gemm_down",
                                  "layernorm_kv", "gemm_kv", "query_proj", "cross_attention", "layernorm_q",
                                  "mlp_up", "mlp_down", "classifier"};
}  // namespace

struct jepa_head {
  jepa_head_hparams hp;
  int device = 0;
  uint8_t* arena = nullptr;
  std::vector<Rec> tensors;
  std::vector<HeadLayer> layers;
  const float *query = nullptr, *lkv_w = nullptr, *lkv_b = nullptr, *b_q = nullptr, *b_kv = nullptr, *l2_w = nullptr,
              *l2_b = nullptr, *b_up = nullptr, *b_down = nullptr, *b_cls = nullptr;
  const void *w_q = nullptr, *w_kv = nullptr, *w_up = nullptr, *w_down = nullptr, *w_cls = nullptr;
  CUtensorMap tm_kv[3];
  const Rec* find(const char* name) const {
    for (const auto& t : tensors)
      if (t.name == name) return &t;
    return nullptr;
  }
};

struct jepa_head_context {
  const jepa_head* h = nullptr;
  SeqRunner run;
  int max_B = 0, max_N = 0;
  uint8_t* ws = nullptr;
  size_t ws_bytes = 0;
  float *X = nullptr, *qv = nullptr, *x1 = nullptr, *y = nullptr, *u = nullptr, *pooled = nullptr, *part = nullptr;
  void *Xn = nullptr, *qkv = nullptr, *ao = nullptr, *Hh = nullptr;
  int* err = nullptr;
  int kB = -1, kN = -1;
  CUtensorMap tm_Xn, tm_ao, tm_Hh, tm_qkv3, tm_o_qkv, tm_o_kv, tm_o_hh, tm_o_x;
  int bn_qkv = 0, bn_out = 0, bn_up = 0, bn_down = 0, bn_kv = 0;
};

// ------------------------------------------------------------------ hyper-parameters
extern "C" jepa_status jepa_head_preset(const char* name, jepa_head_hparams* out) {
  if (!name || !out) return fail(JEPA_E_INVALID_ARG, "jepa_head_preset: null argument");
  jepa_head_hparams h;
  memset(&h, 0, sizeof h);
  if (std::string(name) == "vjepa2_vitl16_ssv2") {
    h.embed_dim = 1024; h.n_head = 16; h.ffn_dim = 4096; h.n_pool_layers = 3; h.n_classes = 174; h.ln_eps = 1e-6f;
  } else {
    return fail(JEPA_E_INVALID_ARG, "jepa_head_preset: unknown preset '%s'", name);
  }
  *out = h;
  return JEPA_OK;
}

extern "C" jepa_status jepa_head_hparams_validate(const jepa_head_hparams* hp) {
  if (!hp) return fail(JEPA_E_INVALID_ARG, "head hparams: null");
  auto in = [](int v, int lo, int hi) { return v >= lo && v <= hi; };
  if (!in(hp->embed_dim, 1, 65536)) return fail(JEPA_E_INVALID_ARG, "head embed_dim %d outside [1, 65536]", hp->embed_dim);
  if (!in(hp->n_head, 1, 1024)) return fail(JEPA_E_INVALID_ARG, "head n_head %d outside [1, 1024]", hp->n_head);
  if (!in(hp->ffn_dim, 1, 1 << 20)) return fail(JEPA_E_INVALID_ARG, "head ffn_dim %d outside [1, 2^20]", hp->ffn_dim);
  if (!in(hp->n_pool_layers, 0, 64)) return fail(JEPA_E_INVALID_ARG, "head n_pool_layers %d outside [0, 64]", hp->n_pool_layers);
  if (!in(hp->n_classes, 1, 1 << 20)) return fail(JEPA_E_INVALID_ARG, "head n_classes %d outside [1, 2^20]", hp->n_classes);
  if (!std::isfinite(hp->ln_eps) || hp->ln_eps < 0.0f || hp->ln_eps > 1.0f)
    return fail(JEPA_E_INVALID_ARG, "head ln_eps %g not finite in [0, 1]", (double)hp->ln_eps);
  if (hp->embed_dim % hp->n_head)
    return fail(JEPA_E_INVALID_ARG, "head embed_dim %d not divisible by n_head %d", hp->embed_dim, hp->n_head);
  return JEPA_OK;
}

// ------------------------------------------------------------------ weights
extern "C" void jepa_head_free(jepa_head* h) {
  if (!h) return;
  if (h->arena) {
    cudaSetDevice(h->device);
    cudaFree(h->arena);
  }
  delete h;
}

extern "C" jepa_status jepa_head_load(const jepa_head_hparams* hp, uint64_t seed, int32_t dtype, int32_t device,
                                      jepa_head** out) {
  if (!hp || !out) return fail(JEPA_E_INVALID_ARG, "jepa_head_load: null argument");
  *out = nullptr;
  jepa_status st = jepa_head_hparams_validate(hp);
  if (st != JEPA_OK) return st;
  if (dtype != JEPA_BF16) return fail(JEPA_E_UNSUPPORTED, "the head runs in bf16 only (dtype %d)", dtype);
  const int D = hp->embed_dim, F = hp->ffn_dim, C = hp->n_classes, L = hp->n_pool_layers, hd = D / hp->n_head;
  if (D % 64 || F % 64 || D > 2048)
    return fail(JEPA_E_UNSUPPORTED, "head widths (embed %d, ffn %d) must be multiples of 64, embed at most 2048", D, F);
  if (hd != 32 && hd != 64 && hd != 128) return fail(JEPA_E_UNSUPPORTED, "head head_dim %d: 32, 64 or 128 only", hd);
  if (L > 0 && hd != 64) return fail(JEPA_E_UNSUPPORTED, "pooler self-attention layers need head_dim 64 (got %d)", hd);
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
    return fail(JEPA_E_CUDA, "CUDA device %d not available (%d devices)", device, ndev);
  CUDA_TRY(cudaSetDevice(device));
  jepa_head* h = new jepa_head();
  h->hp = *hp;
  h->device = device;
  auto add = [&](const std::string& name, size_t n, bool matrix) { h->tensors.push_back({name, 0, n, matrix}); };
  for (int l = 0; l < L; ++l) {
    const std::string s = "head.blk." + std::to_string(l) + ".";
    add(s + "ln1.weight", D, false);
    add(s + "ln1.bias", D, false);
    add(s + "attn_qkv.weight", (size_t)3 * D * D, true);
    add(s + "attn_qkv.bias", (size_t)3 * D, false);
    add(s + "attn_out.weight", (size_t)D * D, true);
    add(s + "attn_out.bias", D, false);
    add(s + "ln2.weight", D, false);
    add(s + "ln2.bias", D, false);
    add(s + "ffn_up.weight", (size_t)F * D, true);
    add(s + "ffn_up.bias", F, false);
    add(s + "ffn_down.weight", (size_t)D * F, true);
    add(s + "ffn_down.bias", D, false);
  }
  add("head.query", D, false);
  add("head.xattn.ln_kv.weight", D, false);
  add("head.xattn.ln_kv.bias", D, false);
  add("head.xattn.q.weight", (size_t)D * D, true);
  add("head.xattn.q.bias", D, false);
  // k then v, weights and biases each adjacent: one [2D, D] projection
  add("head.xattn.k.weight", (size_t)D * D, true);
  add("head.xattn.v.weight", (size_t)D * D, true);
  add("head.xattn.k.bias", D, false);
  add("head.xattn.v.bias", D, false);
  add("head.xattn.ln2.weight", D, false);
  add("head.xattn.ln2.bias", D, false);
  add("head.xattn.ffn_up.weight", (size_t)F * D, true);
  add("head.xattn.ffn_up.bias", F, false);
  add("head.xattn.ffn_down.weight", (size_t)D * F, true);
  add("head.xattn.ffn_down.bias", D, false);
  add("head.cls.weight", (size_t)C * D, true);
  add("head.cls.bias", C, false);
  size_t off = 0, largest = 0;
  for (auto& t : h->tensors) {
    t.offset = off;
    off = align256(off + t.n * (t.bf16 ? 2 : 4));
    largest = std::max(largest, t.n);
  }
  cudaError_t e = cudaMalloc(&h->arena, off);
  if (e != cudaSuccess) {
    delete h;
    return fail(JEPA_E_OOM, "head weights: cudaMalloc(%zu bytes) failed: %s", off, cudaGetErrorString(e));
  }
  std::vector<float> host(largest);
  std::vector<uint16_t> bits;
  for (const auto& t : h->tensors) {
    synth_parallel(seed, t.name, 1, t.n, host.data());
    if (t.bf16) {
      bits.resize(t.n);
      for (size_t i = 0; i < t.n; ++i) bits[i] = jsynth_f32_to_bf16_bits(host[i]);
      e = cudaMemcpy(h->arena + t.offset, bits.data(), t.n * 2, cudaMemcpyHostToDevice);
    } else {
      e = cudaMemcpy(h->arena + t.offset, host.data(), t.n * 4, cudaMemcpyHostToDevice);
    }
    if (e != cudaSuccess) {
      jepa_head_free(h);
      return fail(JEPA_E_CUDA, "head weights upload: %s", cudaGetErrorString(e));
    }
  }
  auto ptr = [&](const std::string& n) -> uint8_t* { return h->arena + h->find(n.c_str())->offset; };
  auto fptr = [&](const std::string& n) -> const float* { return reinterpret_cast<const float*>(ptr(n)); };
  if (ptr("head.xattn.v.weight") != ptr("head.xattn.k.weight") + (size_t)D * D * 2 ||
      ptr("head.xattn.v.bias") != ptr("head.xattn.k.bias") + (size_t)D * 4) {
    jepa_head_free(h);
    return fail(JEPA_E_UNSUPPORTED, "head key / value tensors are not adjacent (embed %d)", D);
  }
  h->query = fptr("head.query");
  h->lkv_w = fptr("head.xattn.ln_kv.weight");
  h->lkv_b = fptr("head.xattn.ln_kv.bias");
  h->w_q = ptr("head.xattn.q.weight");
  h->b_q = fptr("head.xattn.q.bias");
  h->w_kv = ptr("head.xattn.k.weight");
  h->b_kv = fptr("head.xattn.k.bias");
  h->l2_w = fptr("head.xattn.ln2.weight");
  h->l2_b = fptr("head.xattn.ln2.bias");
  h->w_up = ptr("head.xattn.ffn_up.weight");
  h->b_up = fptr("head.xattn.ffn_up.bias");
  h->w_down = ptr("head.xattn.ffn_down.weight");
  h->b_down = fptr("head.xattn.ffn_down.bias");
  h->w_cls = ptr("head.cls.weight");
  h->b_cls = fptr("head.cls.bias");
  const uint32_t boxes[3] = {64, 128, 256};
  bool ok = true;
  for (int s = 0; s < 3; ++s) ok &= make_tmap_2d_bf16(&h->tm_kv[s], h->w_kv, 2 * D, D, boxes[s]);
  h->layers.resize(L);
  for (int l = 0; l < L; ++l) {
    const std::string s = "head.blk." + std::to_string(l) + ".";
    HeadLayer& w = h->layers[l];
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
      ok &= make_tmap_2d_bf16(&w.tm_qkv[b], w.w_qkv, 3 * D, D, boxes[b]);
      ok &= make_tmap_2d_bf16(&w.tm_out[b], w.w_out, D, D, boxes[b]);
      ok &= make_tmap_2d_bf16(&w.tm_up[b], w.w_up, F, D, boxes[b]);
      ok &= make_tmap_2d_bf16(&w.tm_down[b], w.w_down, D, F, boxes[b]);
    }
  }
  if (!ok) {
    jepa_head_free(h);
    return fail(JEPA_E_CUDA, "cuTensorMapEncodeTiled refused a head weight map");
  }
  *out = h;
  return JEPA_OK;
}

extern "C" jepa_status jepa_head_tensor(const jepa_head* h, const char* name, float* h_dst, size_t n_elems) {
  if (!h || !name || !h_dst) return fail(JEPA_E_INVALID_ARG, "jepa_head_tensor: null argument");
  const Rec* t = h->find(name);
  if (!t) return fail(JEPA_E_INVALID_ARG, "jepa_head_tensor: no tensor named '%s'", name);
  if (t->n != n_elems) return fail(JEPA_E_INVALID_ARG, "tensor '%s' has %zu elements, not %zu", name, t->n, n_elems);
  CUDA_TRY(cudaSetDevice(h->device));
  if (t->bf16) {
    std::vector<uint16_t> bits(t->n);
    CUDA_TRY(cudaMemcpy(bits.data(), h->arena + t->offset, t->n * 2, cudaMemcpyDeviceToHost));
    for (size_t i = 0; i < t->n; ++i) h_dst[i] = jsynth_bf16_bits_to_f32(bits[i]);
  } else {
    CUDA_TRY(cudaMemcpy(h_dst, h->arena + t->offset, t->n * 4, cudaMemcpyDeviceToHost));
  }
  return JEPA_OK;
}

// ------------------------------------------------------------------ context
namespace {
size_t head_ws_layout(const jepa_head* h, long long B, long long N, jepa_head_context* c) {
  const size_t D = h->hp.embed_dim, F = h->hp.ffn_dim;
  const size_t rows = (size_t)(B * N);
  const bool blocks = h->hp.n_pool_layers > 0;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const size_t oX = take(blocks ? rows * D * 4 : 0), oXn = take(rows * D * 2), oQ = take(rows * 3 * D * 2),
               oA = take(blocks ? rows * D * 2 : 0), oH = take(blocks ? rows * F * 2 : 0), oq = take(D * 4),
               o1 = take((size_t)B * D * 4), oy = take((size_t)B * D * 4), ou = take((size_t)B * F * 4),
               op = take((size_t)B * D * 4),
               oP = take((size_t)B * h->hp.n_head * xattn_splits((int)N) * (D / h->hp.n_head + 2) * 4),
               oE = take(sizeof(int));
  if (c) {
    c->X = reinterpret_cast<float*>(c->ws + oX);
    c->Xn = c->ws + oXn;
    c->qkv = c->ws + oQ;
    c->ao = c->ws + oA;
    c->Hh = c->ws + oH;
    c->qv = reinterpret_cast<float*>(c->ws + oq);
    c->x1 = reinterpret_cast<float*>(c->ws + o1);
    c->y = reinterpret_cast<float*>(c->ws + oy);
    c->u = reinterpret_cast<float*>(c->ws + ou);
    c->pooled = reinterpret_cast<float*>(c->ws + op);
    c->part = reinterpret_cast<float*>(c->ws + oP);
    c->err = reinterpret_cast<int*>(c->ws + oE);
  }
  return off;
}

// kernels of one forward: 7 per pooler layer; ln_kv, K|V GEMM, query, cross attention (two), ln2, up, down;
// the classifier when logits are asked for (the token copy before the layers is not a kernel)
int head_launches(const jepa_head_hparams& hp, bool logits) { return 7 * hp.n_pool_layers + 8 + (logits ? 1 : 0); }
}  // namespace

extern "C" jepa_status jepa_head_context_new(const jepa_head* h, int32_t max_batch, int32_t max_tokens,
                                             size_t max_workspace_bytes, jepa_head_context** out) {
  if (!h || !out) return fail(JEPA_E_INVALID_ARG, "jepa_head_context_new: null argument");
  *out = nullptr;
  if (max_batch <= 0 || max_tokens <= 0 || max_tokens > kXMaxTokens)
    return fail(JEPA_E_INVALID_ARG, "head context %d x %d tokens out of range (tokens at most %d)", max_batch, max_tokens,
                kXMaxTokens);
  const size_t need = head_ws_layout(h, max_batch, max_tokens, nullptr);
  const size_t budget = max_workspace_bytes ? max_workspace_bytes : kDefaultBudget;
  if (need > budget)
    return fail(JEPA_E_BUDGET, "head workspace of %zu bytes for %d x %d tokens exceeds the budget of %zu bytes", need,
                max_batch, max_tokens, budget);
  CUDA_TRY(cudaSetDevice(h->device));
  CUDA_TRY(tc_kernels_init());
  jepa_head_context* c = new jepa_head_context();
  c->h = h;
  c->max_B = max_batch;
  c->max_N = max_tokens;
  cudaError_t e = cudaMalloc(&c->ws, need);
  if (e != cudaSuccess) {
    delete c;
    return fail(JEPA_E_OOM, "head workspace: cudaMalloc(%zu bytes) failed: %s", need, cudaGetErrorString(e));
  }
  c->ws_bytes = need;
  head_ws_layout(h, max_batch, max_tokens, c);
  e = cudaMemset(c->err, 0, sizeof(int));
  const jepa_status st = e == cudaSuccess ? c->run.init(kHClasses) : JEPA_E_CUDA;
  if (st != JEPA_OK) {
    cudaFree(c->ws);
    delete c;
    return st == JEPA_E_CUDA && e != cudaSuccess ? fail(JEPA_E_CUDA, "head context: %s", cudaGetErrorString(e)) : st;
  }
  *out = c;
  return JEPA_OK;
}

extern "C" void jepa_head_context_free(jepa_head_context* c) {
  if (!c) return;
  cudaSetDevice(c->h->device);
  c->run.destroy();
  if (c->ws) cudaFree(c->ws);
  delete c;
}

extern "C" jepa_status jepa_head_context_set_stream(jepa_head_context* c, void* stream) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_head_context_set_stream: null context");
  CUDA_TRY(cudaSetDevice(c->h->device));
  return c->run.set_stream(stream);
}

extern "C" jepa_status jepa_head_context_set_graph(jepa_head_context* c, int32_t enable) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_head_context_set_graph: null context");
  c->run.use_graph = enable != 0;
  return JEPA_OK;
}

extern "C" jepa_status jepa_head_context_set_profiling(jepa_head_context* c, int32_t enable) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_head_context_set_profiling: null context");
  c->run.profiling = enable != 0;
  return JEPA_OK;
}

extern "C" jepa_status jepa_head_context_launches(const jepa_head_context* c, int32_t with_logits, int32_t* n_out) {
  if (!c || !n_out) return fail(JEPA_E_INVALID_ARG, "jepa_head_context_launches: null argument");
  *n_out = head_launches(c->h->hp, with_logits != 0);
  return JEPA_OK;
}

namespace {
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

jepa_status head_prepare(jepa_head_context* c, int B, int N) {
  if (c->kB == B && c->kN == N) return JEPA_OK;
  const jepa_head_hparams& hp = c->h->hp;
  const int D = hp.embed_dim, F = hp.ffn_dim;
  const long long M = (long long)B * N;
  bool ok = true;
  ok &= make_tmap_2d_bf16(&c->tm_Xn, c->Xn, M, D, 128);
  ok &= make_tmap_2d_out(&c->tm_o_kv, c->qkv, M, 2 * D, 2);
  if (hp.n_pool_layers > 0) {
    ok &= make_tmap_2d_bf16(&c->tm_ao, c->ao, M, D, 128);
    ok &= make_tmap_2d_bf16(&c->tm_Hh, c->Hh, M, F, 128);
    ok &= make_tmap_3d_bf16(&c->tm_qkv3, c->qkv, B, N, 3 * D, 128);
    ok &= make_tmap_2d_out(&c->tm_o_qkv, c->qkv, M, 3 * D, 2);
    ok &= make_tmap_2d_out(&c->tm_o_hh, c->Hh, M, F, 2);
    ok &= make_tmap_2d_out(&c->tm_o_x, c->X, M, D, 4);
  }
  if (!ok) return fail(JEPA_E_CUDA, "cuTensorMapEncodeTiled refused a head workspace map");
  c->bn_qkv = gemm_tc_pick_bn((int)M, 3 * D);
  c->bn_out = gemm_tc_pick_bn((int)M, D);
  c->bn_up = gemm_tc_pick_bn((int)M, F);
  c->bn_down = gemm_tc_pick_bn((int)M, D);
  c->bn_kv = gemm_tc_pick_bn((int)M, 2 * D);
  c->kB = B;
  c->kN = N;
  return JEPA_OK;
}

jepa_status head_launch(jepa_head_context* c, const float* tokens, int B, int N, float* pooled, float* logits) {
  const jepa_head* h = c->h;
  const jepa_head_hparams& hp = h->hp;
  const int D = hp.embed_dim, F = hp.ffn_dim, NH = hp.n_head, hd = D / NH, C = hp.n_classes;
  const int M = B * N;
  cudaStream_t s = c->run.stream;
  const uint64_t lim = default_wait_limit_ns();
  PdlScope pdl_scope(!c->run.profiling);
  auto timed = [c](int cls, double fl, double by, auto&& launch) { return c->run.timed(cls, fl, by, launch); };
  const double dM = M, dD = D, dF = F;
  const double ln_bytes = dM * dD * 6.0;
  const float* src = tokens;
  if (hp.n_pool_layers > 0) {
    CUDA_TRY(cudaMemcpyAsync(c->X, tokens, (size_t)M * D * 4, cudaMemcpyDeviceToDevice, s));
    src = c->X;
    AttnParams ap;
    ap.B = B;
    ap.N = N;
    ap.H = NH;
    ap.head_dim = 64;
    ap.attn_mode = 0;
    ap.prefix = 0;
    ap.frame_tokens = 1;
    ap.out = c->ao;
    const double attn_flops = 4.0 * hd * NH * B * (double)N * N;
    for (int l = 0; l < hp.n_pool_layers; ++l) {
      const HeadLayer& w = h->layers[l];
      EpiArgs qe = epi_of(kEpiBias, M, 3 * D, w.b_qkv, c->qkv);
      EpiArgs oe = epi_of(kEpiResidual, M, D, w.b_out, c->X);
      EpiArgs ue = epi_of(kEpiGelu, M, F, w.b_up, c->Hh);
      EpiArgs de = epi_of(kEpiResidual, M, D, w.b_down, c->X);
      CUDA_TRY(timed(kHLn, 0.0, ln_bytes,
                     [&] { return layernorm_launch(c->X, M, D, w.ln1_w, w.ln1_b, hp.ln_eps, true, c->Xn, s); }));
      CUDA_TRY(timed(kHQkv, 2.0 * dM * 3.0 * dD * dD, 0.0, [&] {
        return gemm_tc_launch(c->tm_Xn, w.tm_qkv[slot(c->bn_qkv)], c->tm_o_qkv, c->bn_qkv, qe, M, 3 * D, D, c->err, lim, s);
      }));
      CUDA_TRY(timed(kHAttn, attn_flops, 0.0, [&] { return attention_tc_launch(c->tm_qkv3, ap, c->err, lim, s); }));
      CUDA_TRY(timed(kHOut, 2.0 * dM * dD * dD, 0.0, [&] {
        return gemm_tc_launch(c->tm_ao, w.tm_out[slot(c->bn_out)], c->tm_o_x, c->bn_out, oe, M, D, D, c->err, lim, s);
      }));
      CUDA_TRY(timed(kHLn, 0.0, ln_bytes,
                     [&] { return layernorm_launch(c->X, M, D, w.ln2_w, w.ln2_b, hp.ln_eps, true, c->Xn, s); }));
      CUDA_TRY(timed(kHUp, 2.0 * dM * dF * dD, 0.0, [&] {
        return gemm_tc_launch(c->tm_Xn, w.tm_up[slot(c->bn_up)], c->tm_o_hh, c->bn_up, ue, M, F, D, c->err, lim, s);
      }));
      CUDA_TRY(timed(kHDown, 2.0 * dM * dD * dF, 0.0, [&] {
        return gemm_tc_launch(c->tm_Hh, w.tm_down[slot(c->bn_down)], c->tm_o_x, c->bn_down, de, M, D, F, c->err, lim, s);
      }));
    }
  }
  // cross attention: keys / values from the normalised tokens, the query from the raw query token
  CUDA_TRY(timed(kHLnKv, 0.0, ln_bytes,
                 [&] { return layernorm_launch(src, M, D, h->lkv_w, h->lkv_b, hp.ln_eps, true, c->Xn, s); }));
  EpiArgs ke = epi_of(kEpiBias, M, 2 * D, h->b_kv, c->qkv);
  CUDA_TRY(timed(kHKv, 2.0 * dM * 2.0 * dD * dD, 0.0, [&] {
    return gemm_tc_launch(c->tm_Xn, h->tm_kv[slot(c->bn_kv)], c->tm_o_kv, c->bn_kv, ke, M, 2 * D, D, c->err, lim, s);
  }));
  CUDA_TRY(timed(kHQuery, 2.0 * dD * dD, dD * dD * 2.0,
                 [&] { return rowvec_launch(h->query, 1, D, h->w_q, D, h->b_q, nullptr, c->qv, false, s); }));
  const int S = xattn_splits(N);
  CUDA_TRY(timed(kHXattn, 4.0 * dD * B * N, (double)M * 2 * D * 2.0, [&] {
    return launch_kernel(xattn_part_kernel, dim3(NH, B, S), dim3(kXThreads), 0, s, (const float*)c->qv,
                         reinterpret_cast<const __nv_bfloat16*>(c->qkv), N, D, hd, c->part);
  }));
  CUDA_TRY(timed(kHXattn, 0.0, (double)B * NH * S * (hd + 2) * 4.0, [&] {
    return launch_kernel(xattn_combine_kernel, dim3(NH, B), dim3(hd), 0, s, (const float*)c->part, S, hd, D, h->query,
                         c->x1);
  }));
  CUDA_TRY(timed(kHLn2, 0.0, (double)B * D * 8.0,
                 [&] { return layernorm_launch(c->x1, B, D, h->l2_w, h->l2_b, hp.ln_eps, false, c->y, s); }));
  CUDA_TRY(timed(kHMlpUp, 2.0 * B * dF * dD, dF * dD * 2.0,
                 [&] { return rowvec_launch(c->y, B, D, h->w_up, F, h->b_up, nullptr, c->u, true, s); }));
  float* pout = pooled ? pooled : c->pooled;
  CUDA_TRY(timed(kHMlpDown, 2.0 * B * dD * dF, dD * dF * 2.0,
                 [&] { return rowvec_launch(c->u, B, F, h->w_down, D, h->b_down, c->x1, pout, false, s); }));
  if (logits)
    CUDA_TRY(timed(kHCls, 2.0 * B * (double)C * dD, (double)C * dD * 2.0,
                   [&] { return rowvec_launch(pout, B, D, h->w_cls, C, h->b_cls, nullptr, logits, false, s); }));
  return JEPA_OK;
}
}  // namespace

extern "C" jepa_status jepa_head_forward(jepa_head_context* c, const float* d_tokens, int32_t B, int32_t N,
                                         float* d_pooled, float* d_logits) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_head_forward: null context");
  if (!d_tokens || (!d_pooled && !d_logits)) return fail(JEPA_E_INVALID_ARG, "jepa_head_forward: null pointer");
  if (B <= 0 || N <= 0) return fail(JEPA_E_INVALID_ARG, "jepa_head_forward: sizes B %d, N %d", B, N);
  if (B > c->max_B || N > c->max_N)
    return fail(JEPA_E_BUDGET, "jepa_head_forward: %d x %d tokens exceed the context's %d x %d", B, N, c->max_B, c->max_N);
  if (reinterpret_cast<uintptr_t>(d_tokens) & 15) return fail(JEPA_E_INVALID_ARG, "jepa_head_forward: tokens must be 16-byte aligned");
  CUDA_TRY(cudaSetDevice(c->h->device));
  jepa_status st = head_prepare(c, B, N);
  if (st != JEPA_OK) return st;
  const std::vector<uintptr_t> key = {(uintptr_t)B, (uintptr_t)N, (uintptr_t)d_tokens, (uintptr_t)d_pooled,
                                     (uintptr_t)d_logits};
  return c->run.run(key, [&] { return head_launch(c, d_tokens, B, N, d_pooled, d_logits); }, "jepa_head_forward");
}

extern "C" jepa_status jepa_head_context_sync(jepa_head_context* c) {
  if (!c) return fail(JEPA_E_INVALID_ARG, "jepa_head_context_sync: null context");
  CUDA_TRY(cudaSetDevice(c->h->device));
  return c->run.sync(c->err, "jepa_head_forward");
}

extern "C" jepa_status jepa_head_context_profile(jepa_head_context* c, jepa_kernel_stat* out, int32_t max,
                                                 int32_t* n_out, int32_t reset) {
  if (!c || !n_out || (max > 0 && !out)) return fail(JEPA_E_INVALID_ARG, "jepa_head_context_profile: null argument");
  CUDA_TRY(cudaSetDevice(c->h->device));
  return c->run.profile(kHNames, out, max, n_out, reset);
}

extern "C" jepa_status jepa_op_pool(int32_t mode, const float* d_tokens, int32_t B, int32_t N, int32_t D, int32_t prefix,
                                    float* d_out, void* stream) {
  if (!d_tokens || !d_out) return fail(JEPA_E_INVALID_ARG, "jepa_op_pool: null pointer");
  if (mode != JEPA_POOL_MEAN && mode != JEPA_POOL_CLS) return fail(JEPA_E_INVALID_ARG, "jepa_op_pool: mode %d unknown", mode);
  if (B <= 0 || N <= 0 || D <= 0 || D % 4 || prefix < 0 || prefix >= N || (mode == JEPA_POOL_CLS && prefix < 1))
    return fail(JEPA_E_INVALID_ARG, "jepa_op_pool: B %d, N %d, D %d, prefix %d (mode %d)", B, N, D, prefix, mode);
  if ((reinterpret_cast<uintptr_t>(d_tokens) | reinterpret_cast<uintptr_t>(d_out)) & 15)
    return fail(JEPA_E_INVALID_ARG, "jepa_op_pool: tokens and output must be 16-byte aligned");
  CUDA_TRY(launch_kernel(pool_kernel, dim3((D / 4 + 31) / 32, B), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream),
                         d_tokens, N, D, prefix, mode, d_out));
  return JEPA_OK;
}
