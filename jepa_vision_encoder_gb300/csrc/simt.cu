// simt.cu -- the fp32 path: a split-K tiled FFMA GEMM with the shared epilogues and an fp32 flash
// attention (online softmax). Used when the model is loaded in fp32 (the hfvit Ti/14 image
// encoder workload), where every operation keeps fp32 precision end to end.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace jepa {

namespace {

// C[M,N] = A[M,K] B[N,K]^T for the small fp32 shapes (one image of 257 tokens: every GEMM has a
// few dozen 32 x 32 output tiles). A CTA of 8 warps computes one 32 x 32 tile; each warp takes
// one eighth of the K steps (so a CTA's dependent chain of global loads is K / 8 long), stages
// its 32 x 16 slices of A and B in its own shared memory with the next step's loads in flight, and
// accumulates a 4 x 8 micro-tile per lane; the eight partial tiles are then summed in a fixed
// order (the same order for every batch size) and passed to the epilogue four columns at a time.
constexpr int kTM = 32, kTN = 32, kTK = 16, kKS = 8, kLd = 36;  // kLd: padded row (16-byte aligned)

__global__ void __launch_bounds__(256) gemm_simt_kernel(const float* __restrict__ A, const float* __restrict__ Bw,
                                                        EpiArgs epi, int M, int N, int K) {
  __shared__ __align__(16) float sm[kKS * 2 * kTK * kLd];  // per warp A and B slices; then the partial tiles
  static_assert(kKS * 2 * kTK * kLd >= kKS * kTM * kTN, "partial tiles fit the staging area");
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * kTM, n0 = blockIdx.x * kTN;
  float* As = sm + warp * 2 * kTK * kLd;  // [kTK][kLd]: As[kk][row]
  float* Bs = As + kTK * kLd;             // [kTK][kLd]: Bs[kk][col]
  const int steps = (K + kTK - 1) / kTK, per = (steps + kKS - 1) / kKS;
  const int s_begin = warp * per, s_end = min(steps, s_begin + per);
  const int r0 = (lane >> 2) * 4, c0 = (lane & 3) * 8;  // this lane's 4 x 8 outputs
  float acc[4][8] = {};
  float ra[16], rb[16];  // one step of A and B (32 x 16 each), 16 values per lane
  auto load_a = [&](int st) {
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const int idx = lane + 32 * t, row = idx / kTK, kk = idx % kTK, gk = st * kTK + kk;
      ra[t] = (m0 + row < M && gk < K) ? __ldg(A + (size_t)(m0 + row) * K + gk) : 0.0f;
    }
  };
  auto load_b = [&](int st) {
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const int idx = lane + 32 * t, row = idx / kTK, kk = idx % kTK, gk = st * kTK + kk;
      rb[t] = (n0 + row < N && gk < K) ? __ldg(Bw + (size_t)(n0 + row) * K + gk) : 0.0f;
    }
  };
  // B holds weights, written by no kernel of the sequence: its first step is requested before
  // waiting for the kernel that produced A
  if (s_begin < s_end) load_b(s_begin);
  pdl_wait();
  if (s_begin < s_end) load_a(s_begin);
  for (int st = s_begin; st < s_end; ++st) {
    __syncwarp();  // the previous step's shared-memory reads are done
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const int idx = lane + 32 * t, row = idx / kTK, kk = idx % kTK;
      As[kk * kLd + row] = ra[t];
      Bs[kk * kLd + row] = rb[t];
    }
    __syncwarp();
    if (st + 1 < s_end) {  // in flight during this step's FMAs
      load_a(st + 1);
      load_b(st + 1);
    }
#pragma unroll
    for (int kk = 0; kk < kTK; ++kk) {
      const float4 a4 = *reinterpret_cast<const float4*>(As + kk * kLd + r0);
      const float4 b0 = *reinterpret_cast<const float4*>(Bs + kk * kLd + c0);
      const float4 b1 = *reinterpret_cast<const float4*>(Bs + kk * kLd + c0 + 4);
      const float a[4] = {a4.x, a4.y, a4.z, a4.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
  }
  __syncthreads();  // every warp is done with its staging area
  float* red = sm;  // [kKS][kTM * kTN]
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; j += 4)
      *reinterpret_cast<float4*>(red + warp * kTM * kTN + (r0 + i) * kTN + c0 + j) =
          make_float4(acc[i][j], acc[i][j + 1], acc[i][j + 2], acc[i][j + 3]);
  __syncthreads();
  const int o = threadIdx.x * 4, row = o / kTN, col = o % kTN;
  float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int w = 0; w < kKS; ++w) {
    const float4 x = *reinterpret_cast<const float4*>(red + w * kTM * kTN + o);
    v[0] += x.x;
    v[1] += x.y;
    v[2] += x.z;
    v[3] += x.w;
  }
  const int m = m0 + row, n = n0 + col;
  if (m < M && n < N) epi_fragment<4, false>(epi, m, n, v);
}

// fp32 attention ("Architecture", attention): a CTA per (8 query rows, head, item), kTpr threads
// per query row, the row's scaled q in registers. Keys come in chunks of 32 staged in shared memory
// (the next chunk's loads in flight while one is scored); thread `sub` of a row scores keys sub,
// sub + kTpr, ... of the chunk (64-wide dot products from 16-byte shared-memory reads), the row's
// threads combine the chunk maximum and sum by shuffles (online softmax: earlier sums and outputs
// rescaled when the maximum moves), and each accumulates 64 / kTpr of the row's output columns.
constexpr int kSQ = 8, kSK = 32, kSHD = 64, kKLd = kSHD + 4, kTpr = 16;
constexpr int kAThreads = kSQ * kTpr, kALoads = kSK * (kSHD / 4) / kAThreads;  // float4 of K (and of V) per thread
constexpr int kKpt = kSK / kTpr, kOpt = kSHD / kTpr;  // keys scored, output columns per thread

__global__ void __launch_bounds__(kAThreads) attn_simt_kernel(const float* __restrict__ qkv, AttnParams p) {
  __shared__ __align__(16) float Ks[kSK][kKLd];
  __shared__ __align__(16) float Vs[kSK][kSHD];
  __shared__ float Ps[kSQ][kSK + 1];
  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.y, b = blockIdx.z;
  const int D = p.H * kSHD, ld = 3 * D;
  const int q0 = blockIdx.x * kSQ;
  const int r = threadIdx.x / kTpr, sub = threadIdx.x % kTpr;  // query row of the CTA, its share
  const int q = q0 + r;
  const float* base = qkv + (size_t)b * p.N * ld + h * kSHD;
  float qv[kSHD];
  {
    const float4* qr = reinterpret_cast<const float4*>(base + (size_t)(q < p.N ? q : 0) * ld);
#pragma unroll
    for (int c = 0; c < kSHD; c += 4) {
      const float4 x = __ldg(qr + c / 4);
      qv[c] = x.x * 0.125f;  // 1/sqrt(64), exact
      qv[c + 1] = x.y * 0.125f;
      qv[c + 2] = x.z * 0.125f;
      qv[c + 3] = x.w * 0.125f;
    }
  }
  int lo = 0, hi = p.N;  // visible keys of this row
  if (p.attn_mode == 1 && q >= p.prefix) {
    lo = p.prefix;
    hi = min(p.N, p.prefix + ((q - p.prefix) / p.frame_tokens + 1) * p.frame_tokens);
  }
  int kv_end = p.N;  // keys any row of the CTA sees
  if (p.attn_mode == 1 && q0 >= p.prefix) {
    const int q_last = min(q0 + kSQ - 1, p.N - 1);
    kv_end = min(p.N, p.prefix + ((q_last - p.prefix) / p.frame_tokens + 1) * p.frame_tokens);
  }
  // chunk staging: this thread's float4 of K and of V (rows idx / 16, columns (idx % 16) * 4)
  float4 rk[kALoads], rv[kALoads];
  auto load = [&](int k0) {
#pragma unroll
    for (int t = 0; t < kALoads; ++t) {
      const int idx = threadIdx.x + kAThreads * t, kr = idx >> 4, c = (idx & 15) * 4, key = k0 + kr;
      rk[t] = rv[t] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (key < p.N) {
        rk[t] = __ldg(reinterpret_cast<const float4*>(base + (size_t)key * ld + D + c));
        rv[t] = __ldg(reinterpret_cast<const float4*>(base + (size_t)key * ld + 2 * D + c));
      }
    }
  };
  float m_run = -INFINITY, l_run = 0.0f, o[kOpt] = {};
  if (kv_end > 0) load(0);
  for (int k0 = 0; k0 < kv_end; k0 += kSK) {
    __syncthreads();  // the previous chunk's K / V reads are done
#pragma unroll
    for (int t = 0; t < kALoads; ++t) {
      const int idx = threadIdx.x + kAThreads * t, kr = idx >> 4, c = (idx & 15) * 4;
      *reinterpret_cast<float4*>(&Ks[kr][c]) = rk[t];
      *reinterpret_cast<float4*>(&Vs[kr][c]) = rv[t];
    }
    __syncthreads();
    if (k0 + kSK < kv_end) load(k0 + kSK);  // in flight while this chunk is used
    float s[kKpt];
#pragma unroll
    for (int j = 0; j < kKpt; ++j) {
      const int kr = sub + kTpr * j, key = k0 + kr;
      float d0 = 0.0f, d1 = 0.0f;
#pragma unroll
      for (int c = 0; c < kSHD; c += 8) {
        const float4 x = *reinterpret_cast<const float4*>(&Ks[kr][c]);
        const float4 y = *reinterpret_cast<const float4*>(&Ks[kr][c + 4]);
        d0 = fmaf(qv[c], x.x, d0);
        d0 = fmaf(qv[c + 1], x.y, d0);
        d0 = fmaf(qv[c + 2], x.z, d0);
        d0 = fmaf(qv[c + 3], x.w, d0);
        d1 = fmaf(qv[c + 4], y.x, d1);
        d1 = fmaf(qv[c + 5], y.y, d1);
        d1 = fmaf(qv[c + 6], y.z, d1);
        d1 = fmaf(qv[c + 7], y.w, d1);
      }
      s[j] = (key >= lo && key < hi) ? d0 + d1 : -INFINITY;
    }
    float cm = s[0];
#pragma unroll
    for (int j = 1; j < kKpt; ++j) cm = fmaxf(cm, s[j]);
#pragma unroll
    for (int off = kTpr / 2; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
    const float m_new = fmaxf(m_run, cm);
    // nothing visible yet: p = 0 and nothing to rescale
    const float alpha = (m_new == -INFINITY) ? 1.0f : expf(m_run - m_new);
    float ps = 0.0f;
#pragma unroll
    for (int j = 0; j < kKpt; ++j) {
      const float pj = (m_new == -INFINITY) ? 0.0f : expf(s[j] - m_new);
      Ps[r][sub + kTpr * j] = pj;
      ps += pj;
    }
#pragma unroll
    for (int off = kTpr / 2; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l_run = l_run * alpha + ps;
    m_run = m_new;
    __syncwarp();  // the row's probabilities (written by its threads, all in this warp) are visible
#pragma unroll
    for (int e = 0; e < kOpt; ++e) o[e] *= alpha;
#pragma unroll 8
    for (int kr = 0; kr < kSK; ++kr) {
      const float pk = Ps[r][kr];
#pragma unroll
      for (int e = 0; e < kOpt; e += 4) {
        const float4 v = *reinterpret_cast<const float4*>(&Vs[kr][sub * kOpt + e]);
        o[e] = fmaf(pk, v.x, o[e]);
        o[e + 1] = fmaf(pk, v.y, o[e + 1]);
        o[e + 2] = fmaf(pk, v.z, o[e + 2]);
        o[e + 3] = fmaf(pk, v.w, o[e + 3]);
      }
    }
    __syncwarp();  // Ps of this row is read before the next chunk overwrites it
  }
  if (q < p.N) {
    float* dst = reinterpret_cast<float*>(p.out) + ((size_t)b * p.N + q) * D + h * kSHD + sub * kOpt;
    const float inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;
#pragma unroll
    for (int e = 0; e < kOpt; e += 4)
      *reinterpret_cast<float4*>(dst + e) = make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv, o[e + 3] * inv);
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
  return launch_kernel(attn_simt_kernel, grid, dim3(kAThreads), 0, s, qkv, q);
}

}  // namespace jepa
