// postab.cu -- fixed sin-cos position tables and their resizing to a clip's grid.
//
// Both run once per model (the table of the training grid) or once per clip shape (the resized
// table); neither is part of the per-call launch sequence. The encode then adds the table in the
// patch-embedding GEMM's epilogue, like a learned table.
#include <cuda_runtime.h>

#include <cmath>

#include "kernels.h"

namespace jepa {
namespace {

int blocks_for(long long work, int threads) {
  long long b = (work + threads - 1) / threads;
  const long long cap = (long long)num_sms() * 16;
  if (b > cap) b = cap;
  return (int)(b < 1 ? 1 : b);
}

// ------------------------------------------------------------------ sin-cos tables
// ("GGUF schema (v1)", Encoder: sincos2d / sincos3d tables baked for the training grid;
// "Converter", sincos_2d / sincos_3d.) One axis of even width d maps position p to
// [sin(p w_0) .. sin(p w_{d/2-1}), cos(p w_0) .. cos(p w_{d/2-1})], w_k = 10000^(-k/(d/2)).
// One thread per table element, computed in double and stored as float.
__global__ void sincos_table_kernel(int kind, int gt, int gh, int gw, int D, int w_first, int d0, int d1, int d2,
                                    float* __restrict__ out) {
  const long long total = (long long)gt * gh * gw * D;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int row = (int)(idx / D), col = (int)(idx % D);
    const int t = row / (gh * gw), h = (row / gw) % gh, w = row % gw;
    int d, j, p;
    if (kind == 0) {  // 2-D: [axis(h) | axis(w)] or [axis(w) | axis(h)], each d0 = D/2 wide
      const bool first = col < d0;
      d = d0;
      j = first ? col : col - d0;
      p = (first != (w_first != 0)) ? h : w;
    } else {          // 3-D: [axis(t) | axis(h) | axis(w)] of widths d0, d1, d2, cut to D
      if (col < d0) {
        d = d0; j = col; p = t;
      } else if (col < d0 + d1) {
        d = d1; j = col - d0; p = h;
      } else {
        d = d2; j = col - d0 - d1; p = w;
      }
    }
    const int half = d / 2;
    const int k = j < half ? j : j - half;
    const double omega = pow(10000.0, -(double)k / (double)half);
    const double a = (double)p * omega;
    out[idx] = (float)(j < half ? sin(a) : cos(a));
  }
}

// ------------------------------------------------------------------ resizing
// Pixel-centre alignment: output index o of an axis of n_in -> n_out samples reads c =
// (o + 1/2) n_in/n_out - 1/2 ("as HF does": align_corners off). Float arithmetic.
__device__ __forceinline__ float resize_coord(int o, int n_in, int n_out) {
  return ((float)n_in / (float)n_out) * ((float)o + 0.5f) - 0.5f;
}

__device__ __forceinline__ void linear_taps(int o, int n_in, int n_out, int idx[2], float wt[2]) {
  const float c = fmaxf(resize_coord(o, n_in, n_out), 0.0f);
  const int i0 = min((int)c, n_in - 1);
  const float l1 = c - (float)i0;
  idx[0] = i0;
  idx[1] = min(i0 + 1, n_in - 1);
  wt[0] = 1.0f - l1;
  wt[1] = l1;
}

// Keys' cubic convolution kernel, a = -0.75, at the four distances 1+x, x, 1-x, 2-x.
__device__ __forceinline__ void cubic_taps(int o, int n_in, int n_out, int idx[4], float wt[4]) {
  const float c = resize_coord(o, n_in, n_out);
  const float fl = floorf(c);
  const int i0 = (int)fl;
  const float x = c - fl;
  const float a = -0.75f;
  const float near0 = x, near1 = 1.0f - x;             // |distance| <= 1
  const float far0 = 1.0f + x, far1 = 2.0f - x;        // 1 <= |distance| <= 2
  wt[0] = ((a * far0 - 5.0f * a) * far0 + 8.0f * a) * far0 - 4.0f * a;
  wt[1] = ((a + 2.0f) * near0 - (a + 3.0f)) * near0 * near0 + 1.0f;
  wt[2] = ((a + 2.0f) * near1 - (a + 3.0f)) * near1 * near1 + 1.0f;
  wt[3] = ((a * far1 - 5.0f * a) * far1 + 8.0f * a) * far1 - 4.0f * a;
  for (int j = 0; j < 4; ++j) idx[j] = min(max(i0 - 1 + j, 0), n_in - 1);
}

__device__ __forceinline__ void fma4(float4& acc, float w, const float4 v) {
  acc.x = fmaf(w, v.x, acc.x);
  acc.y = fmaf(w, v.y, acc.y);
  acc.z = fmaf(w, v.z, acc.z);
  acc.w = fmaf(w, v.w, acc.w);
}

// One thread per (output row, 4 columns); the taps are recomputed per thread (a handful of
// float operations against 8 or 16 loads that mostly hit L2).
__global__ void pos_resize_kernel(const float4* __restrict__ src, int st, int sh, int sw, int D4, int mode,
                                  float4* __restrict__ dst, int dt, int dh, int dw) {
  const long long total = (long long)dt * dh * dw * D4;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int row = (int)(idx / D4), c4 = (int)(idx % D4);
    const int t = row / (dh * dw), h = (row / dw) % dh, w = row % dw;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (mode == 0) {
      int it[2], ih[2], iw[2];
      float at[2], ah[2], aw[2];
      linear_taps(t, st, dt, it, at);
      linear_taps(h, sh, dh, ih, ah);
      linear_taps(w, sw, dw, iw, aw);
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            fma4(acc, at[a] * ah[b] * aw[e], __ldg(src + (((size_t)it[a] * sh + ih[b]) * sw + iw[e]) * D4 + c4));
    } else {
      int ih[4], iw[4];
      float ah[4], aw[4];
      cubic_taps(h, sh, dh, ih, ah);
      cubic_taps(w, sw, dw, iw, aw);
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);  // along w first, then along h
#pragma unroll
        for (int b = 0; b < 4; ++b) fma4(r, aw[b], __ldg(src + (((size_t)t * sh + ih[a]) * sw + iw[b]) * D4 + c4));
        fma4(acc, ah[a], r);
      }
    }
    dst[idx] = acc;
  }
}

}  // namespace

bool sincos_widths(int kind, int D, int uniform_power, int* d0, int* d1, int* d2) {
  if (D <= 0) return false;
  if (kind == 0) {
    if (D % 4) return false;
    *d0 = D / 2;
    *d1 = *d2 = 0;
    return true;
  }
  if (uniform_power) {
    *d0 = *d1 = *d2 = 2 * ((D + 5) / 6);
    return true;
  }
  if (D % 8) return false;
  *d0 = D / 2;
  *d1 = *d2 = D / 4;
  return true;
}

cudaError_t sincos_table_launch(int kind, int gt, int gh, int gw, int D, int w_first, int uniform_power, float* out,
                                cudaStream_t s) {
  int d0, d1, d2;
  if (!sincos_widths(kind, D, uniform_power, &d0, &d1, &d2) || gt <= 0 || gh <= 0 || gw <= 0)
    return cudaErrorInvalidValue;
  const long long total = (long long)gt * gh * gw * D;
  sincos_table_kernel<<<blocks_for(total, 256), 256, 0, s>>>(kind, gt, gh, gw, D, w_first, d0, d1, d2, out);
  return cudaGetLastError();
}

cudaError_t pos_resize_launch(const float* src, int st, int sh, int sw, int D, int mode, float* dst, int dt, int dh,
                              int dw, cudaStream_t s) {
  if (D % 4 || st <= 0 || sh <= 0 || sw <= 0 || dt <= 0 || dh <= 0 || dw <= 0 || (mode == 1 && st != dt))
    return cudaErrorInvalidValue;
  const long long total = (long long)dt * dh * dw * (D / 4);
  pos_resize_kernel<<<blocks_for(total, 256), 256, 0, s>>>(reinterpret_cast<const float4*>(src), st, sh, sw, D / 4,
                                                           mode, reinterpret_cast<float4*>(dst), dt, dh, dw);
  return cudaGetLastError();
}

}  // namespace jepa
