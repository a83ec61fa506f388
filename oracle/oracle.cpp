// oracle.cpp -- plain fp64 CPU reference of the shared ViT encoder forward.
//
// TEST INFRASTRUCTURE ONLY: used by tests/, the smoke check and the bench's CPU
// baseline; never by the product path. Shares nothing with the GPU library
// except the seeded input generator (synth/jepa_synth.h).
//
// Each step is written from the jepa.cpp pages (see oracle.h for the page tags),
// with no fusion and no reordering of the method's steps. OpenMP only splits
// independent rows / heads across threads; the row blocking of oracle_linear and
// the vectorised dot products change nothing but the rounding order of the sums.
#include "oracle.h"

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

#include "../synth/jepa_synth.h"

namespace {

struct Geometry {
  int C, t, P, gt, gh, gw, Np, prefix, N, K;
};

bool geometry(const oracle_hparams* hp, int T, int H, int W, Geometry* g) {
  if (!hp || T <= 0 || H <= 0 || W <= 0) return false;
  const int t = hp->tubelet_size, P = hp->patch_size;
  if (t <= 0 || P <= 0 || T % t || H % P || W % P) return false;
  g->C = hp->in_chans;
  g->t = t;
  g->P = P;
  g->gt = T / t;
  g->gh = H / P;
  g->gw = W / P;
  g->Np = g->gt * g->gh * g->gw;
  g->prefix = hp->cls_token ? 1 : 0;
  g->N = g->Np + g->prefix;
  g->K = g->C * t * P * P;
  return true;
}

// pixel (b, frame, c, y, x) of a [B,T,C,H,W] (layout 0) or [B,C,T,H,W] (layout 1) array.
inline float pixel_at(const float* pix, int layout, int T, int C, int H, int W, int b, int f, int c, int y,
                      int x) {
  size_t idx;
  if (layout == 0)
    idx = ((((size_t)b * T + f) * C + c) * H + y) * (size_t)W + x;
  else
    idx = ((((size_t)b * C + c) * T + f) * H + y) * (size_t)W + x;
  return pix[idx];
}

// Synthetic parameter tensor, generated in parallel chunks (the generator is counter-based).
void gen_param(uint64_t seed, const std::string& name, int bf16, size_t n, std::vector<double>& dst) {
  dst.assign(n, 0.0);
  int kind, is_matrix;
  double a, b;
  jsynth_param_init(name.c_str(), &kind, &a, &b, &is_matrix);
  const int round = (bf16 && is_matrix) ? 1 : 0;
  const size_t chunk = 4096;
  const long nchunks = (long)((n + chunk - 1) / chunk);
#pragma omp parallel
  {
    std::vector<float> tmp(chunk);
#pragma omp for schedule(static)
    for (long c = 0; c < nchunks; ++c) {
      size_t first = (size_t)c * chunk;
      size_t len = std::min(chunk, n - first);
      jsynth_fill(seed, name.c_str(), kind, a, b, round, first, len, tmp.data());
      for (size_t j = 0; j < len; ++j) dst[first + j] = (double)tmp[j];
    }
  }
}

}  // namespace

extern "C" {

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

int oracle_n_tokens(const oracle_hparams* hp, int T, int H, int W) {
  Geometry g;
  if (!geometry(hp, T, H, W, &g)) return -1;
  return g.N;
}

// [A] "The shared ViT graph": rows [N, C*T*P*P]; [S] "Token order": i = t*gh*gw + h*gw + w;
// [C] flatten_patch_conv: C-T-H-W element order; [K]: element order (c, dt, dh, dw).
int oracle_patchify(const oracle_hparams* hp, const float* pix, int B, int T, int H, int W, int layout,
                    double* out) {
  Geometry g;
  if (!geometry(hp, T, H, W, &g) || B <= 0) return -1;
#pragma omp parallel for collapse(2) schedule(static)
  for (int b = 0; b < B; ++b)
    for (int i = 0; i < g.Np; ++i) {
      const int tt = i / (g.gh * g.gw), hh = (i % (g.gh * g.gw)) / g.gw, ww = i % g.gw;
      double* row = out + ((size_t)b * g.Np + i) * g.K;
      for (int c = 0; c < g.C; ++c)
        for (int dt = 0; dt < g.t; ++dt)
          for (int dy = 0; dy < g.P; ++dy)
            for (int dx = 0; dx < g.P; ++dx) {
              const int k = ((c * g.t + dt) * g.P + dy) * g.P + dx;
              row[k] = pixel_at(pix, layout, T, g.C, H, W, b, tt * g.t + dt, c, hh * g.P + dy, ww * g.P + dx);
            }
    }
  return 0;
}

// The strided Conv3d the patch embedding replaces ([A] "The shared ViT graph"; [K]):
// kernel = stride = (t, P, P), no padding.
int oracle_conv3d(const oracle_hparams* hp, const float* pix, int B, int T, int H, int W, int layout,
                  const double* w, const double* bias, double* out) {
  Geometry g;
  if (!geometry(hp, T, H, W, &g) || B <= 0) return -1;
  const int D = hp->embed_dim;
#pragma omp parallel for collapse(4) schedule(static)
  for (int b = 0; b < B; ++b)
    for (int ot = 0; ot < g.gt; ++ot)
      for (int oy = 0; oy < g.gh; ++oy)
        for (int ox = 0; ox < g.gw; ++ox)
          for (int d = 0; d < D; ++d) {
            double acc = bias ? bias[d] : 0.0;
            for (int c = 0; c < g.C; ++c)
              for (int kt = 0; kt < g.t; ++kt)
                for (int ky = 0; ky < g.P; ++ky)
                  for (int kx = 0; kx < g.P; ++kx) {
                    const double wv = w[((((size_t)d * g.C + c) * g.t + kt) * g.P + ky) * g.P + kx];
                    acc += wv * (double)pixel_at(pix, layout, T, g.C, H, W, b, ot * g.t + kt, c, oy * g.P + ky,
                                                 ox * g.P + kx);
                  }
            out[((((size_t)b * g.gt + ot) * g.gh + oy) * g.gw + ox) * D + d] = acc;
          }
  return 0;
}

// y = x w^T + b, the ggml_mul_mat of every linear layer ([S] weights stored [out, in]).
void oracle_linear(const double* x, int M, int K, const double* w, const double* b, int N, double* y) {
  const int IB = 16;  // rows of x sharing one pass over w (cache reuse only; same sums)
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int i0 = 0; i0 < M; i0 += IB)
    for (int j0 = 0; j0 < N; j0 += 64) {
      const int i1 = std::min(M, i0 + IB), j1 = std::min(N, j0 + 64);
      for (int j = j0; j < j1; ++j) {
        const double* wr = w + (size_t)j * K;
        for (int i = i0; i < i1; ++i) {
          const double* xr = x + (size_t)i * K;
          double acc = 0.0;
#pragma omp simd reduction(+ : acc)
          for (int k = 0; k < K; ++k) acc += xr[k] * wr[k];
          y[(size_t)i * N + j] = acc + (b ? b[j] : 0.0);
        }
      }
    }
}

// LayerNorm: mean, centred biased variance, (x - mu) / sqrt(var + eps) * gamma + beta.
void oracle_layernorm(const double* x, int M, int D, const double* gamma, const double* beta, double eps,
                      double* y) {
#pragma omp parallel for schedule(static)
  for (int i = 0; i < M; ++i) {
    const double* xr = x + (size_t)i * D;
    double mu = 0.0;
    for (int j = 0; j < D; ++j) mu += xr[j];
    mu /= D;
    double var = 0.0;
    for (int j = 0; j < D; ++j) var += (xr[j] - mu) * (xr[j] - mu);
    var /= D;
    const double rstd = 1.0 / std::sqrt(var + eps);
    for (int j = 0; j < D; ++j) y[(size_t)i * D + j] = (xr[j] - mu) * rstd * gamma[j] + beta[j];
  }
}

void oracle_gelu(const double* x, size_t n, double* y) {
#pragma omp parallel for schedule(static)
  for (long i = 0; i < (long)n; ++i) y[i] = 0.5 * x[i] * (1.0 + std::erf(x[i] / std::sqrt(2.0)));
}

// [A] "3-D RoPE": t = i // (gh gw), h = (i % (gh gw)) // gw, w = i % gw; V-JEPA 2.1 rescales
// h and w (not t) by (rope_ref_grid - 1) / (grid - 1). A grid of one row keeps its position.
int oracle_rope_positions(const oracle_hparams* hp, int T, int H, int W, double* pos) {
  Geometry g;
  if (!geometry(hp, T, H, W, &g)) return -1;
  const double sh = (hp->rope_interpolate && g.gh > 1) ? (double)(hp->rope_ref_grid - 1) / (double)(g.gh - 1) : 1.0;
  const double sw = (hp->rope_interpolate && g.gw > 1) ? (double)(hp->rope_ref_grid - 1) / (double)(g.gw - 1) : 1.0;
  for (int i = 0; i < g.Np; ++i) {
    pos[3 * i + 0] = (double)(i / (g.gh * g.gw));
    pos[3 * i + 1] = (double)((i % (g.gh * g.gw)) / g.gw) * sh;
    pos[3 * i + 2] = (double)(i % g.gw) * sw;
  }
  return 0;
}

// [A] "3-D RoPE": per axis d = 2*((hd//3)//2) dims; omega_k = 1/theta^(2k/d), k < d/2;
// tiled table[j] = f(pos * omega_{j mod d/2}) (V-JEPA 2), interleaved table[2k] = table[2k+1]
// = f(pos * omega_k) (V-JEPA 2.1); x cos + rot90(x) sin with rot90(y1, y2) = (-y2, y1), the
// sign carried in the sin table; prefix (CLS) rows are identity ([S] levjepa note).
void oracle_rope_tables_pos(int hd, double theta, int layout, const double* pos, int n, double* cos_t,
                            double* sin_t) {
  const int d = 2 * ((hd / 3) / 2);
  for (int i = 0; i < n; ++i) {
    double* cr = cos_t + (size_t)i * hd;
    double* sr = sin_t + (size_t)i * hd;
    for (int j = 0; j < hd; ++j) { cr[j] = 1.0; sr[j] = 0.0; }
    for (int a = 0; a < 3; ++a)
      for (int jj = 0; jj < d; ++jj) {
        const int kidx = (layout == 0) ? (jj % (d / 2)) : (jj / 2);
        const double omega = 1.0 / std::pow(theta, 2.0 * kidx / d);
        const double th = pos[3 * i + a] * omega;
        cr[a * d + jj] = std::cos(th);
        sr[a * d + jj] = ((jj % 2 == 0) ? -1.0 : 1.0) * std::sin(th);
      }
  }
}

int oracle_rope_tables(const oracle_hparams* hp, int T, int H, int W, double* cos_t, double* sin_t) {
  Geometry g;
  if (!geometry(hp, T, H, W, &g)) return -1;
  const int hd = hp->embed_dim / hp->n_head;
  std::vector<double> pos((size_t)g.Np * 3);
  oracle_rope_positions(hp, T, H, W, pos.data());
  for (int n = 0; n < g.prefix; ++n)  // prefix (CLS) rows: identity
    for (int j = 0; j < hd; ++j) {
      cos_t[(size_t)n * hd + j] = 1.0;
      sin_t[(size_t)n * hd + j] = 0.0;
    }
  oracle_rope_tables_pos(hd, hp->rope_theta, hp->rope_layout, pos.data(), g.Np, cos_t + (size_t)g.prefix * hd,
                         sin_t + (size_t)g.prefix * hd);
  return 0;
}

void oracle_rope_apply(const double* x, int N, int n_head, int hd, const double* cos_t, const double* sin_t,
                       double* out) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n)
    for (int h = 0; h < n_head; ++h) {
      const double* xr = x + ((size_t)n * n_head + h) * hd;
      double* orow = out + ((size_t)n * n_head + h) * hd;
      const double* cr = cos_t + (size_t)n * hd;
      const double* sr = sin_t + (size_t)n * hd;
      for (int j = 0; j < hd; ++j) orow[j] = xr[j] * cr[j] + ((j ^ 1) < hd ? xr[j ^ 1] * sr[j] : 0.0);
    }
}

// ---- fixed sin-cos position tables ([S] "Encoder": sincos2d / sincos3d; [R] sincos_2d, sincos_3d) ----

// One axis of even width d: column k < d/2 is sin(p w_k), column d/2 + k is cos(p w_k), with the
// d/2 frequencies w_k = 10000^(-k / (d/2)) falling geometrically from 1 towards 1/10000.
static void sincos_axis(int d, double p, double* out) {
  const int half = d / 2;
  for (int k = 0; k < half; ++k) {
    const double w = std::pow(10000.0, -(double)k / (double)half);
    out[k] = std::sin(p * w);
    out[half + k] = std::cos(p * w);
  }
}

int oracle_sincos_2d(int gh, int gw, int D, int w_first, double* out) {
  if (gh <= 0 || gw <= 0 || D <= 0 || D % 4) return -1;
  const int half = D / 2;
  for (int i = 0; i < gh * gw; ++i) {
    const int h = i / gw, w = i % gw;
    double* row = out + (size_t)i * D;
    sincos_axis(half, w_first ? w : h, row);
    sincos_axis(half, w_first ? h : w, row + half);
  }
  return 0;
}

int oracle_sincos_3d(int gt, int gh, int gw, int D, int uniform_power, double* out) {
  if (gt <= 0 || gh <= 0 || gw <= 0 || D <= 0) return -1;
  int dt, dh, dw;
  if (uniform_power) {
    dt = dh = dw = 2 * ((D + 5) / 6);  // 2 ceil(D / 6)
  } else {
    if (D % 8) return -1;
    dt = D / 2;
    dh = dw = D / 4;
  }
  std::vector<double> full((size_t)(dt + dh + dw));
  for (int i = 0; i < gt * gh * gw; ++i) {
    const int t = i / (gh * gw), h = (i / gw) % gh, w = i % gw;
    sincos_axis(dt, t, full.data());
    sincos_axis(dh, h, full.data() + dt);
    sincos_axis(dw, w, full.data() + dt + dh);
    std::memcpy(out + (size_t)i * D, full.data(), (size_t)D * sizeof(double));  // cut to D columns
  }
  return 0;
}

// Pixel-centre source coordinate of output index o on an axis resized from n_in to n_out samples.
static double resize_coord(int o, int n_in, int n_out) { return (o + 0.5) * ((double)n_in / (double)n_out) - 0.5; }

// Linear blend on one axis: the two input indices and their weights.
static void linear_taps(int o, int n_in, int n_out, int idx[2], double wt[2]) {
  double c = resize_coord(o, n_in, n_out);
  if (c < 0.0) c = 0.0;
  int i0 = (int)std::floor(c);
  if (i0 > n_in - 1) i0 = n_in - 1;
  const double l1 = c - i0;
  idx[0] = i0;
  idx[1] = std::min(i0 + 1, n_in - 1);
  wt[0] = 1.0 - l1;
  wt[1] = l1;
}

// Keys' cubic convolution kernel with a = -0.75.
static double keys_cubic(double x) {
  const double a = -0.75;
  x = std::fabs(x);
  if (x <= 1.0) return ((a + 2.0) * x - (a + 3.0)) * x * x + 1.0;
  if (x < 2.0) return ((a * x - 5.0 * a) * x + 8.0 * a) * x - 4.0 * a;
  return 0.0;
}

// Cubic taps on one axis: samples floor(c)-1 .. floor(c)+2, clamped to the axis.
static void cubic_taps(int o, int n_in, int n_out, int idx[4], double wt[4]) {
  const double c = resize_coord(o, n_in, n_out);
  const int i0 = (int)std::floor(c);
  for (int j = 0; j < 4; ++j) {
    const int s = i0 - 1 + j;
    idx[j] = std::min(std::max(s, 0), n_in - 1);
    wt[j] = keys_cubic(c - s);
  }
}

int oracle_interp_trilinear(const double* src, int st, int sh, int sw, int D, int dt, int dh, int dw, double* dst) {
  if (st <= 0 || sh <= 0 || sw <= 0 || D <= 0 || dt <= 0 || dh <= 0 || dw <= 0) return -1;
#pragma omp parallel for collapse(3) schedule(static)
  for (int t = 0; t < dt; ++t)
    for (int h = 0; h < dh; ++h)
      for (int w = 0; w < dw; ++w) {
        int it[2], ih[2], iw[2];
        double at[2], ah[2], aw[2];
        linear_taps(t, st, dt, it, at);
        linear_taps(h, sh, dh, ih, ah);
        linear_taps(w, sw, dw, iw, aw);
        double* out = dst + (((size_t)t * dh + h) * dw + w) * D;
        for (int c = 0; c < D; ++c) out[c] = 0.0;
        for (int a = 0; a < 2; ++a)
          for (int b = 0; b < 2; ++b)
            for (int e = 0; e < 2; ++e) {
              const double wt = at[a] * ah[b] * aw[e];
              const double* in = src + (((size_t)it[a] * sh + ih[b]) * sw + iw[e]) * D;
              for (int c = 0; c < D; ++c) out[c] += wt * in[c];
            }
      }
  return 0;
}

int oracle_interp_bicubic(const double* src, int sh, int sw, int D, int dh, int dw, double* dst) {
  if (sh <= 0 || sw <= 0 || D <= 0 || dh <= 0 || dw <= 0) return -1;
#pragma omp parallel for collapse(2) schedule(static)
  for (int h = 0; h < dh; ++h)
    for (int w = 0; w < dw; ++w) {
      int ih[4], iw[4];
      double ah[4], aw[4];
      cubic_taps(h, sh, dh, ih, ah);
      cubic_taps(w, sw, dw, iw, aw);
      double* out = dst + ((size_t)h * dw + w) * D;
      for (int c = 0; c < D; ++c) out[c] = 0.0;
      for (int a = 0; a < 4; ++a)
        for (int b = 0; b < 4; ++b) {
          const double wt = ah[a] * aw[b];
          const double* in = src + ((size_t)ih[a] * sw + iw[b]) * D;
          for (int c = 0; c < D; ++c) out[c] += wt * in[c];
        }
    }
  return 0;
}

// [S] "Encoder": the table is baked for the training grid; other grids get it resized (bicubic for
// the 2-D image table, trilinear for the 3-D video table).
int oracle_pos_table(const oracle_hparams* hp, int T, int H, int W, double* out) {
  Geometry g;
  if (!geometry(hp, T, H, W, &g)) return -1;
  const int D = hp->embed_dim;
  if (hp->pos_type != 3 && hp->pos_type != 4) return -1;
  if (hp->img_size <= 0 || hp->img_size % hp->patch_size) return -1;
  const int gh0 = hp->img_size / hp->patch_size, gw0 = gh0;
  if (hp->pos_type == 3) {
    if (g.gt != 1) return -2;  // a 2-D table has no time axis
    std::vector<double> t0((size_t)gh0 * gw0 * D);
    if (oracle_sincos_2d(gh0, gw0, D, hp->sincos_w_first, t0.data())) return -1;
    if (g.gh == gh0 && g.gw == gw0) {
      std::memcpy(out, t0.data(), t0.size() * sizeof(double));
      return 0;
    }
    return oracle_interp_bicubic(t0.data(), gh0, gw0, D, g.gh, g.gw, out);
  }
  if (hp->n_frames <= 0 || hp->n_frames % hp->tubelet_size) return -1;
  const int gt0 = hp->n_frames / hp->tubelet_size;
  std::vector<double> t0((size_t)gt0 * gh0 * gw0 * D);
  if (oracle_sincos_3d(gt0, gh0, gw0, D, hp->sincos_uniform_power, t0.data())) return -1;
  if (g.gt == gt0 && g.gh == gh0 && g.gw == gw0) {
    std::memcpy(out, t0.data(), t0.size() * sizeof(double));
    return 0;
  }
  return oracle_interp_trilinear(t0.data(), gt0, gh0, gw0, D, g.gt, g.gh, g.gw, out);
}

// [S] levjepa note; [A] "Block-causal attention": key j visible to query i iff
// frame_id(i) >= frame_id(j), frame_id = id // (gh gw) of the patch token; CLS row open,
// CLS column closed to patch queries.
int oracle_mask_allow(int attn_mode, int prefix, int frame_tokens, int N, int q, int k) {
  if (k < 0 || k >= N || q < 0 || q >= N) return 0;
  if (attn_mode == 0) return 1;
  if (q < prefix) return 1;
  if (k < prefix) return 0;
  return ((q - prefix) / frame_tokens) >= ((k - prefix) / frame_tokens);
}

// softmax(q k^T / sqrt(hd) + mask) v per head, in fp64, masked keys excluded.
void oracle_attention(const double* q, const double* k, const double* v, int N, int n_head, int hd,
                      int attn_mode, int prefix, int frame_tokens, double* o) {
  const size_t ld = (size_t)n_head * hd;
  const double scale = 1.0 / std::sqrt((double)hd);
  for (int h = 0; h < n_head; ++h) {
#pragma omp parallel
    {
      std::vector<double> s(N);
#pragma omp for schedule(static)
      for (int i = 0; i < N; ++i) {
        const double* qi = q + (size_t)i * ld + (size_t)h * hd;
        double mx = -INFINITY;
        for (int j = 0; j < N; ++j) {
          if (!oracle_mask_allow(attn_mode, prefix, frame_tokens, N, i, j)) { s[j] = -INFINITY; continue; }
          const double* kj = k + (size_t)j * ld + (size_t)h * hd;
          double acc = 0.0;
#pragma omp simd reduction(+ : acc)
          for (int c = 0; c < hd; ++c) acc += qi[c] * kj[c];
          s[j] = acc * scale;
          if (s[j] > mx) mx = s[j];
        }
        double sum = 0.0;
        for (int j = 0; j < N; ++j) {
          s[j] = (s[j] == -INFINITY) ? 0.0 : std::exp(s[j] - mx);
          sum += s[j];
        }
        double* oi = o + (size_t)i * ld + (size_t)h * hd;
        for (int c = 0; c < hd; ++c) oi[c] = 0.0;
        for (int j = 0; j < N; ++j) {
          if (s[j] == 0.0) continue;
          const double p = s[j] / sum;
          const double* vj = v + (size_t)j * ld + (size_t)h * hd;
          for (int c = 0; c < hd; ++c) oi[c] += p * vj[c];
        }
      }
    }
  }
}

}  // extern "C"

namespace {
// The weights of one pre-LN block under `prefix` ("enc.blk.{l}." or "pred.blk.{l}.": [S] the
// predictor blocks have the encoder's layout).
struct BlockW {
  std::vector<double> ln1w, ln1b, wqkv, bqkv, wout, bout, ln2w, ln2b, wup, bup, wdn, bdn;
  void gen(uint64_t seed, const std::string& p, int bf16_weights, int D, int F, double q_scale = 1.0,
           double k_scale = 1.0) {
    gen_param(seed, p + "ln1.weight", bf16_weights, D, ln1w);
    gen_param(seed, p + "ln1.bias", bf16_weights, D, ln1b);
    gen_param(seed, p + "attn_qkv.weight", bf16_weights, (size_t)3 * D * D, wqkv);
    // test input option (oracle.h): scaled q and k rows; with bf16 weights the scaled value is
    // rounded to bf16 again (exact for powers of two), as a bf16 model holds a file's f32 value
    if (q_scale != 1.0 || k_scale != 1.0) {
      for (size_t i = 0; i < (size_t)2 * D * D; ++i) {
        const float v = (float)(wqkv[i] * (i < (size_t)D * D ? q_scale : k_scale));
        wqkv[i] = bf16_weights ? (double)jsynth_round_bf16(v) : (double)v;
      }
    }
    gen_param(seed, p + "attn_qkv.bias", bf16_weights, (size_t)3 * D, bqkv);
    gen_param(seed, p + "attn_out.weight", bf16_weights, (size_t)D * D, wout);
    gen_param(seed, p + "attn_out.bias", bf16_weights, D, bout);
    gen_param(seed, p + "ln2.weight", bf16_weights, D, ln2w);
    gen_param(seed, p + "ln2.bias", bf16_weights, D, ln2b);
    gen_param(seed, p + "ffn_up.weight", bf16_weights, (size_t)F * D, wup);
    gen_param(seed, p + "ffn_up.bias", bf16_weights, F, bup);
    gen_param(seed, p + "ffn_down.weight", bf16_weights, (size_t)D * F, wdn);
    gen_param(seed, p + "ffn_down.bias", bf16_weights, D, bdn);
  }
};

struct BlockScratch {
  std::vector<double> h, qkv, q, k, v, o, tmp, u;
  BlockScratch(int N, int D, int F)
      : h((size_t)N * D), qkv((size_t)N * 3 * D), q((size_t)N * D), k((size_t)N * D), v((size_t)N * D),
        o((size_t)N * D), tmp((size_t)N * D), u((size_t)N * F) {}
};

// One block on the N rows x [N, D] of one item, in place ([A] "The shared ViT graph"):
// x += out(attn(rope(qkv(ln1(x))))); x += down(GELU(up(ln2(x)))). rc / rs: RoPE tables [N, hd]
// applied to q and k (not v) after the projection and before scaling, or null for none.
void block_forward(const BlockW& w, double* x, int N, int D, int NH, int F, double eps, const double* rc,
                   const double* rs, int attn_mode, int prefix, int frame_tokens, BlockScratch& s) {
  const int hd = D / NH;
  const size_t MD = (size_t)N * D;
  // x += attn(ln1(x)): fused qkv rows [q; k; v] ([S] attn_qkv), heads contiguous in each.
  oracle_layernorm(x, N, D, w.ln1w.data(), w.ln1b.data(), eps, s.h.data());
  oracle_linear(s.h.data(), N, D, w.wqkv.data(), w.bqkv.data(), 3 * D, s.qkv.data());
  for (int n = 0; n < N; ++n)
    for (int c = 0; c < D; ++c) {
      s.q[(size_t)n * D + c] = s.qkv[(size_t)n * 3 * D + c];
      s.k[(size_t)n * D + c] = s.qkv[(size_t)n * 3 * D + D + c];
      s.v[(size_t)n * D + c] = s.qkv[(size_t)n * 3 * D + 2 * D + c];
    }
  if (rc) {
    oracle_rope_apply(s.q.data(), N, NH, hd, rc, rs, s.tmp.data());
    s.q.swap(s.tmp);
    oracle_rope_apply(s.k.data(), N, NH, hd, rc, rs, s.tmp.data());
    s.k.swap(s.tmp);
  }
  oracle_attention(s.q.data(), s.k.data(), s.v.data(), N, NH, hd, attn_mode, prefix, frame_tokens, s.o.data());
  oracle_linear(s.o.data(), N, D, w.wout.data(), w.bout.data(), D, s.tmp.data());
  for (size_t i = 0; i < MD; ++i) x[i] += s.tmp[i];
  // x += ffn(ln2(x)) with GELU(erf)
  oracle_layernorm(x, N, D, w.ln2w.data(), w.ln2b.data(), eps, s.h.data());
  oracle_linear(s.h.data(), N, D, w.wup.data(), w.bup.data(), F, s.u.data());
  oracle_gelu(s.u.data(), (size_t)N * F, s.u.data());
  oracle_linear(s.u.data(), N, F, w.wdn.data(), w.bdn.data(), D, s.tmp.data());
  for (size_t i = 0; i < MD; ++i) x[i] += s.tmp[i];
}
}  // namespace

extern "C" {

// [A] "The shared ViT graph":
//   tokens = patch_embed(rearranged pixels) [+ pos_embed] [+ cls] [+ modality vec]
//   for each block: x += attn(ln1(x)); x += ffn(ln2(x))   (pre-LN, GELU(erf), qkv bias)
//   x = norm(x)
int oracle_encode(const oracle_hparams* hp, uint64_t seed, int bf16_weights, const float* pix, int B, int T,
                  int H, int W, int layout, int final_norm, double* out) {
  Geometry g;
  if (!geometry(hp, T, H, W, &g) || B <= 0) return -1;
  const int D = hp->embed_dim, F = hp->ffn_dim, NH = hp->n_head;
  if (NH <= 0 || D % NH) return -1;
  const int hd = D / NH;
  const int N = g.N, Np = g.Np, prefix = g.prefix;
  if (hp->pos_type == 1 && hp->n_pos_rows != N) return -2;  // learned table must cover every token
  if ((hp->pos_type == 3 || hp->pos_type == 4) && prefix) return -2;  // sin-cos tables cover patch rows only
  const size_t MD = (size_t)N * D;

  // ---- patch embedding, prefix and position/modality terms ----
  std::vector<double> patches((size_t)B * Np * g.K);
  oracle_patchify(hp, pix, B, T, H, W, layout, patches.data());
  std::vector<double> wpe, bpe;
  gen_param(seed, "enc.patch_embed.weight", bf16_weights, (size_t)D * g.K, wpe);
  gen_param(seed, "enc.patch_embed.bias", bf16_weights, D, bpe);
  std::vector<double> emb((size_t)B * Np * D);
  oracle_linear(patches.data(), B * Np, g.K, wpe.data(), bpe.data(), D, emb.data());
  patches.clear();
  patches.shrink_to_fit();

  std::vector<double> X((size_t)B * MD, 0.0);
  std::vector<double> cls, pos, mod;
  if (hp->cls_token) gen_param(seed, "enc.cls_token", bf16_weights, D, cls);
  if (hp->pos_type == 1) gen_param(seed, "enc.pos_embed", bf16_weights, (size_t)hp->n_pos_rows * D, pos);
  if (hp->pos_type == 3 || hp->pos_type == 4) {
    pos.resize((size_t)Np * D);
    const int rc = oracle_pos_table(hp, T, H, W, pos.data());
    if (rc) return rc;
  }
  if (hp->modality_embed) gen_param(seed, "enc.mod_embed_video", bf16_weights, D, mod);
  for (int b = 0; b < B; ++b)
    for (int n = 0; n < N; ++n) {
      double* xr = X.data() + (size_t)b * MD + (size_t)n * D;
      for (int c = 0; c < D; ++c) {
        double v = (n < prefix) ? cls[c] : emb[((size_t)b * Np + (n - prefix)) * D + c];
        if (hp->pos_type == 1) v += pos[(size_t)n * D + c];  // rows = [CLS?; patches]
        if (hp->pos_type == 3 || hp->pos_type == 4) v += pos[(size_t)n * D + c];  // patch rows, no prefix
        if (hp->modality_embed) v += mod[c];
        xr[c] = v;
      }
    }
  emb.clear();
  emb.shrink_to_fit();

  // ---- RoPE tables (shared by all layers and heads) ----
  std::vector<double> rc, rs;
  if (hp->pos_type == 2) {
    rc.resize((size_t)N * hd);
    rs.resize((size_t)N * hd);
    oracle_rope_tables(hp, T, H, W, rc.data(), rs.data());
  }
  const int frame_tokens = g.gh * g.gw;

  BlockScratch sc(N, D, F);
  for (int l = 0; l < hp->n_layer; ++l) {
    BlockW w;
    w.gen(seed, "enc.blk." + std::to_string(l) + ".", bf16_weights, D, F, hp->q_weight_scale, hp->k_weight_scale);
    for (int b = 0; b < B; ++b)
      block_forward(w, X.data() + (size_t)b * MD, N, D, NH, F, hp->ln_eps, hp->pos_type == 2 ? rc.data() : nullptr,
                    rs.data(), hp->attn_mode, prefix, frame_tokens, sc);
  }

  if (final_norm) {
    std::vector<double> nw, nb;
    gen_param(seed, "enc.norm.weight", bf16_weights, D, nw);
    gen_param(seed, "enc.norm.bias", bf16_weights, D, nb);
    for (int b = 0; b < B; ++b)
      oracle_layernorm(X.data() + (size_t)b * MD, N, D, nw.data(), nb.data(), hp->ln_eps, out + (size_t)b * MD);
  } else {
    std::memcpy(out, X.data(), X.size() * sizeof(double));
  }
  return 0;
}

// [S] "Predictor": pred.embed [pred_dim, enc_dim], pred.mask_tokens [n, pred_dim], pred.blk.{i}
// (the encoder block layout), pred.norm, pred.proj [out_dim, pred_dim]. [K] masked-latent
// predictor: context features -> embed -> append mask tokens -> order by position -> stack (own
// RoPE table) -> LN -> restore order, take the targets -> proj.
int oracle_predict(const oracle_pred_hparams* hp, uint64_t seed, int bf16_weights, const double* enc, int B,
                   int n_enc, const int* ctx_ids, int n_ctx, const int* tgt_ids, int n_tgt, int gh, int gw,
                   double* out) {
  if (!hp || B <= 0 || n_ctx < 0 || n_tgt <= 0 || n_enc <= 0 || gh <= 0 || gw <= 0) return -1;
  const int P = hp->embed_dim, E = hp->enc_dim, O = hp->out_dim, NH = hp->n_head, F = hp->ffn_dim;
  if (NH <= 0 || P % NH || hp->n_mask_tokens <= 0 || hp->mask_index < 0) return -1;
  const int hd = P / NH, N = n_ctx + n_tgt;
  for (int i = 0; i < B * n_ctx; ++i)
    if (ctx_ids[i] < 0 || ctx_ids[i] >= n_enc) return -1;
  for (int i = 0; i < B * n_tgt; ++i)
    if (tgt_ids[i] < 0) return -1;

  std::vector<double> we, be, mt, nw, nb, wp, bp;
  gen_param(seed, "pred.embed.weight", bf16_weights, (size_t)P * E, we);
  gen_param(seed, "pred.embed.bias", bf16_weights, P, be);
  gen_param(seed, "pred.mask_tokens", bf16_weights, (size_t)hp->n_mask_tokens * P, mt);
  const double* mask_tok = mt.data() + (size_t)(hp->mask_index % hp->n_mask_tokens) * P;

  // per item: the token rows in position order, the order itself, and the RoPE tables
  std::vector<double> X((size_t)B * N * P), rc((size_t)B * N * hd), rs((size_t)B * N * hd);
  std::vector<int> order((size_t)B * N);
  for (int b = 0; b < B; ++b) {
    std::vector<double> ctx((size_t)n_ctx * E), emb((size_t)n_ctx * P);
    for (int s = 0; s < n_ctx; ++s)
      std::memcpy(&ctx[(size_t)s * E], enc + ((size_t)b * n_enc + ctx_ids[b * n_ctx + s]) * E, E * sizeof(double));
    if (n_ctx) oracle_linear(ctx.data(), n_ctx, E, we.data(), be.data(), P, emb.data());
    std::vector<int> ids(N);
    for (int s = 0; s < N; ++s) ids[s] = s < n_ctx ? ctx_ids[b * n_ctx + s] : tgt_ids[b * n_tgt + (s - n_ctx)];
    int* ord = order.data() + (size_t)b * N;
    for (int s = 0; s < N; ++s) ord[s] = s;
    std::stable_sort(ord, ord + N, [&](int a, int c) { return ids[a] < ids[c]; });
    std::vector<double> pos((size_t)N * 3);
    for (int r = 0; r < N; ++r) {
      const int s = ord[r], id = ids[s];
      const double* src = s < n_ctx ? &emb[(size_t)s * P] : mask_tok;
      std::memcpy(&X[((size_t)b * N + r) * P], src, P * sizeof(double));
      pos[3 * r + 0] = (double)(id / (gh * gw));
      pos[3 * r + 1] = (double)((id % (gh * gw)) / gw);
      pos[3 * r + 2] = (double)(id % gw);
    }
    oracle_rope_tables_pos(hd, hp->rope_theta, hp->rope_layout, pos.data(), N, rc.data() + (size_t)b * N * hd,
                           rs.data() + (size_t)b * N * hd);
  }

  BlockScratch sc(N, P, F);
  for (int l = 0; l < hp->n_layer; ++l) {
    BlockW w;
    w.gen(seed, "pred.blk." + std::to_string(l) + ".", bf16_weights, P, F);
    for (int b = 0; b < B; ++b)
      block_forward(w, X.data() + (size_t)b * N * P, N, P, NH, F, hp->ln_eps, rc.data() + (size_t)b * N * hd,
                    rs.data() + (size_t)b * N * hd, 0, 0, 1, sc);
  }

  gen_param(seed, "pred.norm.weight", bf16_weights, P, nw);
  gen_param(seed, "pred.norm.bias", bf16_weights, P, nb);
  gen_param(seed, "pred.proj.weight", bf16_weights, (size_t)O * P, wp);
  gen_param(seed, "pred.proj.bias", bf16_weights, O, bp);
  for (int b = 0; b < B; ++b) {
    std::vector<double> y((size_t)N * P), back((size_t)N * P), tgt((size_t)n_tgt * P);
    oracle_layernorm(X.data() + (size_t)b * N * P, N, P, nw.data(), nb.data(), hp->ln_eps, y.data());
    const int* ord = order.data() + (size_t)b * N;
    for (int r = 0; r < N; ++r) std::memcpy(&back[(size_t)ord[r] * P], &y[(size_t)r * P], P * sizeof(double));
    std::memcpy(tgt.data(), &back[(size_t)n_ctx * P], (size_t)n_tgt * P * sizeof(double));
    oracle_linear(tgt.data(), n_tgt, P, wp.data(), bp.data(), O, out + (size_t)b * n_tgt * O);
  }
  return 0;
}

void oracle_cross_attention(const double* q, int Nq, const double* k, const double* v, int Nk, int n_head, int hd,
                            double* o) {
  const int D = n_head * hd;
  const double scale = 1.0 / std::sqrt((double)hd);
#pragma omp parallel for collapse(2) schedule(static)
  for (int h = 0; h < n_head; ++h)
    for (int i = 0; i < Nq; ++i) {
      std::vector<double> s(Nk);
      const double* qi = q + (size_t)i * D + (size_t)h * hd;
      double mx = -INFINITY;
      for (int j = 0; j < Nk; ++j) {
        const double* kj = k + (size_t)j * D + (size_t)h * hd;
        double acc = 0.0;
        for (int c = 0; c < hd; ++c) acc += qi[c] * kj[c];
        s[j] = acc * scale;
        mx = std::max(mx, s[j]);
      }
      double sum = 0.0;
      for (int j = 0; j < Nk; ++j) {
        s[j] = std::exp(s[j] - mx);
        sum += s[j];
      }
      double* oi = o + (size_t)i * D + (size_t)h * hd;
      for (int c = 0; c < hd; ++c) oi[c] = 0.0;
      for (int j = 0; j < Nk; ++j) {
        const double p = s[j] / sum;
        const double* vj = v + (size_t)j * D + (size_t)h * hd;
        for (int c = 0; c < hd; ++c) oi[c] += p * vj[c];
      }
    }
}

// [S] "Head": head.blk.{i} (encoder block layout, run first), head.query [1, D], head.xattn.ln_kv
// (keys / values only), head.xattn.q / k / v with bias (no output projection), head.xattn.ln2,
// head.xattn.ffn_up / ffn_down, head.cls [n_classes, D] (no final norm). [K] attentive pooler:
// pre-norm self-attention layers without RoPE or mask over the whole token stream, then the
// learned query's cross attention, query residual + MLP; the classifier on the pooled token.
int oracle_attentive_head(const oracle_head_hparams* hp, uint64_t seed, int bf16_weights, const double* tokens, int B,
                          int N, double* pooled, double* logits) {
  if (!hp || B <= 0 || N <= 0 || hp->n_head <= 0 || hp->embed_dim % hp->n_head || hp->n_pool_layers < 0 ||
      hp->n_classes <= 0)
    return -1;
  const int D = hp->embed_dim, F = hp->ffn_dim, NH = hp->n_head, C = hp->n_classes;
  const int hd = D / NH;
  const size_t MD = (size_t)N * D;
  std::vector<double> X(tokens, tokens + (size_t)B * MD);
  BlockScratch sc(N, D, F);
  for (int l = 0; l < hp->n_pool_layers; ++l) {
    BlockW w;
    w.gen(seed, "head.blk." + std::to_string(l) + ".", bf16_weights, D, F);
    for (int b = 0; b < B; ++b)
      block_forward(w, X.data() + (size_t)b * MD, N, D, NH, F, hp->ln_eps, nullptr, nullptr, 0, 0, 1, sc);
  }
  std::vector<double> query, lkw, lkb, wq, bq, wk, bk, wv, bv, l2w, l2b, wup, bup, wdn, bdn, wc, bc;
  gen_param(seed, "head.query", bf16_weights, D, query);
  gen_param(seed, "head.xattn.ln_kv.weight", bf16_weights, D, lkw);
  gen_param(seed, "head.xattn.ln_kv.bias", bf16_weights, D, lkb);
  gen_param(seed, "head.xattn.q.weight", bf16_weights, (size_t)D * D, wq);
  gen_param(seed, "head.xattn.q.bias", bf16_weights, D, bq);
  gen_param(seed, "head.xattn.k.weight", bf16_weights, (size_t)D * D, wk);
  gen_param(seed, "head.xattn.k.bias", bf16_weights, D, bk);
  gen_param(seed, "head.xattn.v.weight", bf16_weights, (size_t)D * D, wv);
  gen_param(seed, "head.xattn.v.bias", bf16_weights, D, bv);
  gen_param(seed, "head.xattn.ln2.weight", bf16_weights, D, l2w);
  gen_param(seed, "head.xattn.ln2.bias", bf16_weights, D, l2b);
  gen_param(seed, "head.xattn.ffn_up.weight", bf16_weights, (size_t)F * D, wup);
  gen_param(seed, "head.xattn.ffn_up.bias", bf16_weights, F, bup);
  gen_param(seed, "head.xattn.ffn_down.weight", bf16_weights, (size_t)D * F, wdn);
  gen_param(seed, "head.xattn.ffn_down.bias", bf16_weights, D, bdn);
  gen_param(seed, "head.cls.weight", bf16_weights, (size_t)C * D, wc);
  gen_param(seed, "head.cls.bias", bf16_weights, C, bc);
  std::vector<double> q(D), kv(MD), k(MD), v(MD), o(D), x(D), h(D), u(F), t(D);
  oracle_linear(query.data(), 1, D, wq.data(), bq.data(), D, q.data());  // the raw query token, no LN
  for (int b = 0; b < B; ++b) {
    oracle_layernorm(X.data() + (size_t)b * MD, N, D, lkw.data(), lkb.data(), hp->ln_eps, kv.data());
    oracle_linear(kv.data(), N, D, wk.data(), bk.data(), D, k.data());
    oracle_linear(kv.data(), N, D, wv.data(), bv.data(), D, v.data());
    oracle_cross_attention(q.data(), 1, k.data(), v.data(), N, NH, hd, o.data());
    for (int c = 0; c < D; ++c) x[c] = query[c] + o[c];  // no output projection; the query is the residual
    oracle_layernorm(x.data(), 1, D, l2w.data(), l2b.data(), hp->ln_eps, h.data());
    oracle_linear(h.data(), 1, D, wup.data(), bup.data(), F, u.data());
    oracle_gelu(u.data(), F, u.data());
    oracle_linear(u.data(), 1, F, wdn.data(), bdn.data(), D, t.data());
    for (int c = 0; c < D; ++c) x[c] += t[c];
    if (pooled) std::memcpy(pooled + (size_t)b * D, x.data(), D * sizeof(double));
    if (logits) oracle_linear(x.data(), 1, D, wc.data(), bc.data(), C, logits + (size_t)b * C);
  }
  return 0;
}

int oracle_pool(const double* tokens, int B, int N, int D, int prefix, int mode, double* out) {
  if (B <= 0 || N <= 0 || D <= 0 || prefix < 0 || prefix >= N) return -1;
  if (mode == 1 && prefix < 1) return -1;
  if (mode != 0 && mode != 1) return -1;
  for (int b = 0; b < B; ++b) {
    const double* t = tokens + (size_t)b * N * D;
    double* o = out + (size_t)b * D;
    if (mode == 1) {
      std::memcpy(o, t, D * sizeof(double));
      continue;
    }
    for (int c = 0; c < D; ++c) o[c] = 0.0;
    for (int n = prefix; n < N; ++n)
      for (int c = 0; c < D; ++c) o[c] += t[(size_t)n * D + c];
    for (int c = 0; c < D; ++c) o[c] /= (double)(N - prefix);
  }
  return 0;
}

}  // extern "C"
