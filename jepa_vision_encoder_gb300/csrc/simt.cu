// simt.cu -- the fp32 path: a tiled FFMA GEMM with the shared epilogues and an fp32 flash
// attention (online softmax). Used when the model is loaded in fp32 (the hfvit Ti/14 image
// encoder workload), where every operation keeps fp32 precision end to end.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace jepa {

namespace {

// C[M,N] = A[M,K] B[N,K]^T. 64x64 tile, BK 16, 256 threads, a 4x4 micro-tile per thread
// (4 consecutive columns, so RoPE pairs stay inside one thread's fragment).
constexpr int kTM = 64, kTN = 64, kTK = 16;

__global__ void __launch_bounds__(256) gemm_simt_kernel(const float* __restrict__ A, const float* __restrict__ Bw,
                                                        EpiArgs epi, int M, int N, int K) {
  __shared__ float As[kTK][kTM + 4];
  __shared__ float Bs[kTK][kTN + 4];
  pdl_trigger();
  pdl_wait();
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * kTM, n0 = blockIdx.x * kTN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kTK) {
    // 64 rows x 16 k of A and of B: 1024 floats each, 4 per thread
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int idx = threadIdx.x + t * 256;
      const int row = idx / kTK, kk = idx % kTK;
      const int gm = m0 + row, gn = n0 + row, gk = k0 + kk;
      As[kk][row] = (gm < M && gk < K) ? A[(size_t)gm * K + gk] : 0.0f;
      Bs[kk][row] = (gn < N && gk < K) ? Bw[(size_t)gn * K + gk] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kTK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    const int n = n0 + tx * 4;
    if (m < M && n < N) epi_fragment<4, false>(epi, m, n, acc[i]);
  }
}

// fp32 attention: one thread per query row, K/V tiles of 64 keys staged in shared memory.
constexpr int kSQ = 128, kSK = 64, kSHD = 64;

__global__ void __launch_bounds__(kSQ) attn_simt_kernel(const float* __restrict__ qkv, AttnParams p) {
  __shared__ float Ks[kSK][kSHD];
  __shared__ float Vs[kSK][kSHD];
  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.y, b = blockIdx.z;
  const int D = p.H * kSHD, ld = 3 * D;
  const int q = blockIdx.x * kSQ + threadIdx.x;
  const bool valid = q < p.N;
  float qv[kSHD], o[kSHD];
  const float* qrow = qkv + ((size_t)b * p.N + (valid ? q : 0)) * ld + h * kSHD;
#pragma unroll
  for (int c = 0; c < kSHD; ++c) {
    qv[c] = qrow[c] * 0.125f;  // 1/sqrt(64), exact
    o[c] = 0.0f;
  }
  int lo = 0, hi = p.N;
  if (p.attn_mode == 1 && q >= p.prefix) {
    lo = p.prefix;
    hi = min(p.N, p.prefix + ((q - p.prefix) / p.frame_tokens + 1) * p.frame_tokens);
  }
  // keys the whole block needs
  int kv_end = p.N;
  const int q0 = blockIdx.x * kSQ;
  if (p.attn_mode == 1 && q0 >= p.prefix) {
    const int q_last = min(q0 + kSQ - 1, p.N - 1);
    kv_end = min(p.N, p.prefix + ((q_last - p.prefix) / p.frame_tokens + 1) * p.frame_tokens);
  }
  float m = -INFINITY, l = 0.0f;
  for (int k0 = 0; k0 < kv_end; k0 += kSK) {
    for (int idx = threadIdx.x; idx < kSK * kSHD; idx += kSQ) {
      const int kr = idx / kSHD, c = idx % kSHD;
      const int key = k0 + kr;
      const float* base = qkv + ((size_t)b * p.N + (key < p.N ? key : 0)) * ld + h * kSHD + c;
      Ks[kr][c] = key < p.N ? base[D] : 0.0f;
      Vs[kr][c] = key < p.N ? base[2 * D] : 0.0f;
    }
    __syncthreads();
    const int kn = min(kSK, kv_end - k0);
    for (int kr = 0; kr < kn; ++kr) {
      const int key = k0 + kr;
      if (key < lo || key >= hi) continue;
      float s = 0.0f;
#pragma unroll
      for (int c = 0; c < kSHD; ++c) s = fmaf(qv[c], Ks[kr][c], s);
      if (s > m) {
        const float alpha = expf(m - s);  // 0 on the first visible key (m = -inf)
        l *= alpha;
#pragma unroll
        for (int c = 0; c < kSHD; ++c) o[c] *= alpha;
        m = s;
      }
      const float pw = expf(s - m);
      l += pw;
#pragma unroll
      for (int c = 0; c < kSHD; ++c) o[c] = fmaf(pw, Vs[kr][c], o[c]);
    }
    __syncthreads();
  }
  if (valid) {
    float* dst = reinterpret_cast<float*>(p.out) + ((size_t)b * p.N + q) * D + h * kSHD;
    const float inv = 1.0f / l;
#pragma unroll
    for (int c = 0; c < kSHD; c += 4)
      *reinterpret_cast<float4*>(dst + c) = make_float4(o[c] * inv, o[c + 1] * inv, o[c + 2] * inv, o[c + 3] * inv);
  }
}

}  // namespace

cudaError_t gemm_simt_launch(const float* A, const float* Bw, const EpiArgs& epi, int M, int N, int K,
                             cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  dim3 grid((N + kTN - 1) / kTN, (M + kTM - 1) / kTM);
  return launch_kernel(gemm_simt_kernel, grid, dim3(256), 0, s, A, Bw, epi, M, N, K);
}

cudaError_t attention_simt_launch(const float* qkv, const AttnParams& p, cudaStream_t s) {
  if (p.head_dim != kSHD) return cudaErrorInvalidValue;
  if (p.B <= 0 || p.N <= 0) return cudaSuccess;
  AttnParams q = p;
  if (q.frame_tokens <= 0) q.frame_tokens = 1;
  dim3 grid((p.N + kSQ - 1) / kSQ, p.H, p.B);
  return launch_kernel(attn_simt_kernel, grid, dim3(kSQ), 0, s, qkv, q);
}

}  // namespace jepa
