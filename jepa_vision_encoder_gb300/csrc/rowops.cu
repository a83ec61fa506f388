// rowops.cu -- the memory-bound kernels of the encoder: pixel -> patch rearrangement,
// LayerNorm, the 3-D RoPE cos/sin table, the CLS prefix rows, plus the tensor-map helpers
// and the bounded-wait failure probe.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace jepa {

// ------------------------------------------------------------------ pixel -> patch rows
// ("Architecture", The shared ViT graph: rows [N, C*t*P*P]; element k = ((c t + dt) P + dy) P + dx;
// token i = (tt gh + hh) gw + ww, i.e. T-major then H then W.)
namespace {

__device__ __forceinline__ size_t pix_index(int layout, int T, int C, int H, int W, int b, int f, int c, int y,
                                            int x) {
  return layout == 0 ? ((((size_t)b * T + f) * C + c) * H + y) * (size_t)W + x
                     : ((((size_t)b * C + c) * T + f) * H + y) * (size_t)W + x;
}

// Vectorised path: one CTA per patch row (persistent over rows when there are more rows than the
// grid), one thread per 8 consecutive elements of the row (16 bytes of bf16, read as two float4 of
// one pixel row). A thread's element offset within the row, and so its (channel, frame offset,
// dy, dx) and pixel offset, is the same for every row and is computed once; each row adds the
// patch's own (item, frame, y, x) origin. Needs P % 8 == 0, W % 4 == 0 and K / 8 <= 1024.
__global__ void patchify_bf16_v8_kernel(const float* __restrict__ pix, int B, int T, int C, int H, int W, int t,
                                        int P, int layout, __nv_bfloat16* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int gt = T / t, gh = H / P, gw = W / P;
  const int K = C * t * P * P, np = gt * gh * gw;
  const int k = threadIdx.x * 8;
  if (k >= K) return;
  const int dx = k % P, dy = (k / P) % P, dt = (k / (P * P)) % t, c = k / (P * P * t);
  const long long rows = (long long)B * np;
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const int b = (int)(row / np), i = (int)(row % np);
    const int tt = i / (gh * gw), hw = i % (gh * gw), hh = hw / gw, ww = hw % gw;
    const float4* src = reinterpret_cast<const float4*>(
        pix + pix_index(layout, T, C, H, W, b, tt * t + dt, c, hh * P + dy, ww * P + dx));
    const float4 u = __ldg(src), v = __ldg(src + 1);
    uint4 w;
    w.x = pack_bf16x2(u.x, u.y);
    w.y = pack_bf16x2(u.z, u.w);
    w.z = pack_bf16x2(v.x, v.y);
    w.w = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint4*>(out + row * K + k) = w;
  }
}

// Generic path, one element per thread (any P, fp32 or bf16 output).
template <bool BF16>
__global__ void patchify_scalar_kernel(const float* __restrict__ pix, int B, int T, int C, int H, int W, int t,
                                       int P, int layout, void* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int gt = T / t, gh = H / P, gw = W / P;
  const int K = C * t * P * P;
  const long long total = (long long)B * gt * gh * gw * K;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long row = idx / K;
    const int k = (int)(idx % K);
    const int b = (int)(row / ((long long)gt * gh * gw));
    const int i = (int)(row % ((long long)gt * gh * gw));
    const int tt = i / (gh * gw), hh = (i % (gh * gw)) / gw, ww = i % gw;
    const int dx = k % P, dy = (k / P) % P, dt = (k / (P * P)) % t, c = k / (P * P * t);
    const float v = __ldg(pix + pix_index(layout, T, C, H, W, b, tt * t + dt, c, hh * P + dy, ww * P + dx));
    if (BF16)
      reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    else
      reinterpret_cast<float*>(out)[idx] = v;
  }
}

int grid_for(long long work, int threads) {
  long long blocks = (work + threads - 1) / threads;
  const long long cap = (long long)num_sms() * 16;
  if (blocks > cap) blocks = cap;
  return (int)(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t patchify_launch(const float* pix, int B, int T, int C, int H, int W, int t, int P, int layout,
                            bool out_bf16, void* out, cudaStream_t s) {
  const long long rows = (long long)B * (T / t) * (H / P) * (W / P);
  const int K = C * t * P * P;
  if (rows <= 0) return cudaSuccess;
  if (out_bf16 && P % 8 == 0 && W % 4 == 0 && K / 8 <= 1024 && (reinterpret_cast<uintptr_t>(pix) & 15) == 0) {
    const int threads = ((K / 8 + 31) / 32) * 32;
    const long long cap = (long long)num_sms() * (2048 / threads);
    const int grid = (int)(rows < cap ? rows : cap);
    return launch_kernel(patchify_bf16_v8_kernel, dim3(grid), dim3(threads), 0, s, pix, B, T, C, H, W, t, P, layout,
                         reinterpret_cast<__nv_bfloat16*>(out));
  }
  return launch_kernel(out_bf16 ? patchify_scalar_kernel<true> : patchify_scalar_kernel<false>,
                       dim3(grid_for(rows * K, 256)), dim3(256), 0, s, pix, B, T, C, H, W, t, P, layout, out);
}

// ------------------------------------------------------------------ LayerNorm
// One warp per row, the row held in registers (D <= 2048): mean, then the centred sum of
// squares (two passes over registers, no E[x^2] - mean^2), eps inside the square root.
// Persistent: the grid is what fits on the GPU at once and each warp strides over the rows,
// loading its next row into a second register set before normalising the current one, so that
// every SM keeps a row per warp in flight and no partial last wave idles the memory system.
namespace {

template <int V>
__device__ __forceinline__ void ln_load(const float* __restrict__ x, int row, int D, int lane, float4 (&v)[V]) {
  const float* xr = x + (size_t)row * D;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int c = (lane + 32 * i) * 4;
    v[i] = (c < D) ? __ldg(reinterpret_cast<const float4*>(xr + c)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// g, bta: gamma and beta as staged in the block's shared memory.
template <int V, bool BF16>
__device__ __forceinline__ void ln_row(const float4 (&v)[V], int row, int D, int lane, const float* g,
                                       const float* bta, float eps, void* __restrict__ y) {
  float sum = 0.0f;
#pragma unroll
  for (int i = 0; i < V; ++i) sum += (v[i].x + v[i].y) + (v[i].z + v[i].w);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float mu = sum / (float)D;
  float sq = 0.0f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int c = (lane + 32 * i) * 4;
    if (c < D) {
      const float a = v[i].x - mu, b = v[i].y - mu, cc = v[i].z - mu, d = v[i].w - mu;
      sq += (a * a + b * b) + (cc * cc + d * d);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  const float rstd = rsqrtf(sq / (float)D + eps);
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int c = (lane + 32 * i) * 4;
    if (c >= D) continue;
    const float4 gg = *reinterpret_cast<const float4*>(g + c);
    const float4 bb = *reinterpret_cast<const float4*>(bta + c);
    const float o0 = (v[i].x - mu) * rstd * gg.x + bb.x;
    const float o1 = (v[i].y - mu) * rstd * gg.y + bb.y;
    const float o2 = (v[i].z - mu) * rstd * gg.z + bb.z;
    const float o3 = (v[i].w - mu) * rstd * gg.w + bb.w;
    if (BF16) {
      uint2 w;
      w.x = pack_bf16x2(o0, o1);
      w.y = pack_bf16x2(o2, o3);
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(y) + (size_t)row * D + c) = w;
    } else {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(y) + (size_t)row * D + c) = make_float4(o0, o1, o2, o3);
    }
  }
}

template <int V, bool BF16>
__global__ void __launch_bounds__(256, 2) layernorm_kernel(const float* __restrict__ x, int M, int D,
                                                        const float* __restrict__ g, const float* __restrict__ bta,
                                                        float eps, void* __restrict__ y) {
  // gamma and beta are weights, written by no kernel of the sequence: staged in shared memory
  // before waiting for the previous kernel
  __shared__ __align__(16) float sg[V * 128], sb[V * 128];
  for (int c = threadIdx.x * 4; c < D; c += 256 * 4) {
    *reinterpret_cast<float4*>(sg + c) = __ldg(reinterpret_cast<const float4*>(g + c));
    *reinterpret_cast<float4*>(sb + c) = __ldg(reinterpret_cast<const float4*>(bta + c));
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int stride = gridDim.x * 8;  // warps in the grid
  int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  float4 a[V], b[V];  // the current row and the next one, alternating
  if (row < M) ln_load<V>(x, row, D, lane, a);
  while (row < M) {
    const int r1 = row + stride;
    if (r1 < M) ln_load<V>(x, r1, D, lane, b);
    ln_row<V, BF16>(a, row, D, lane, sg, sb, eps, y);
    if (r1 >= M) break;
    const int r2 = r1 + stride;
    if (r2 < M) ln_load<V>(x, r2, D, lane, a);
    ln_row<V, BF16>(b, r1, D, lane, sg, sb, eps, y);
    row = r2;
  }
}

template <int V, bool BF16>
int ln_resident_blocks() {
  static int cached = 0;
  if (cached == 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, layernorm_kernel<V, BF16>, 256, 0) != cudaSuccess ||
        per_sm <= 0) {
      cudaGetLastError();
      per_sm = 1;
    }
    cached = per_sm * num_sms();
  }
  return cached;
}

template <int V>
cudaError_t ln_v(const float* x, int M, int D, const float* g, const float* b, float eps, bool bf16, void* y,
                 cudaStream_t s) {
  const int rows_blocks = (M + 7) / 8;
  const int fit = bf16 ? ln_resident_blocks<V, true>() : ln_resident_blocks<V, false>();
  const int grid = rows_blocks < fit ? rows_blocks : fit;
  return launch_kernel(bf16 ? layernorm_kernel<V, true> : layernorm_kernel<V, false>, dim3(grid), dim3(256), 0, s, x,
                       M, D, g, b, eps, y);
}

}  // namespace

cudaError_t layernorm_launch(const float* x, int M, int D, const float* g, const float* b, float eps,
                             bool out_bf16, void* y, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (D % 4 != 0 || D > 2048) return cudaErrorInvalidValue;
  const int v = (D + 127) / 128;  // float4 per lane
  if (v <= 2) return ln_v<2>(x, M, D, g, b, eps, out_bf16, y, s);
  if (v <= 4) return ln_v<4>(x, M, D, g, b, eps, out_bf16, y, s);
  if (v <= 8) return ln_v<8>(x, M, D, g, b, eps, out_bf16, y, s);
  if (v <= 12) return ln_v<12>(x, M, D, g, b, eps, out_bf16, y, s);
  return ln_v<16>(x, M, D, g, b, eps, out_bf16, y, s);
}

// ------------------------------------------------------------------ 3-D RoPE table
// ("Architecture", 3-D RoPE): patch i at (t, h, w) = (i / (gh gw), (i % (gh gw)) / gw, i % gw),
// h and w rescaled by (ref - 1) / (g - 1) under interpolate_rope; omega_k = theta^(-2k/d).
// table[i][axis][k] = (cos, sin)(pos_axis * omega_k), computed in double. The encoder itself uses
// the factored form axes[c][k] over the t coordinates, then h, then w (gt + gh + gw rows): the
// same entries, computed by the same function, in 3 KB instead of one row per token.
namespace {
__device__ __forceinline__ float2 rope_entry(int axis, int coord, int g, int d, int k, double theta, int interp,
                                             int ref) {
  double pos = (double)coord;
  if (axis > 0 && interp && g > 1) pos *= (double)(ref - 1) / (double)(g - 1);
  const double omega = 1.0 / pow(theta, 2.0 * k / (double)d);
  double sn, cs;
  sincos(pos * omega, &sn, &cs);
  return make_float2((float)cs, (float)sn);
}

__global__ void rope_table_kernel(int gt, int gh, int gw, int d, double theta, int interp, int ref,
                                  float2* __restrict__ table) {
  const int dh = d / 2;
  const int total = gt * gh * gw * 3 * dh;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += gridDim.x * blockDim.x) {
    const int k = idx % dh, axis = (idx / dh) % 3, i = idx / (3 * dh);
    const int coord = axis == 0 ? i / (gh * gw) : (axis == 1 ? (i % (gh * gw)) / gw : i % gw);
    table[idx] = rope_entry(axis, coord, axis == 0 ? gt : (axis == 1 ? gh : gw), d, k, theta, interp, ref);
  }
}

__global__ void rope_axes_kernel(int gt, int gh, int gw, int d, double theta, int interp, int ref,
                                 float2* __restrict__ axes) {
  const int dh = d / 2;
  const int total = (gt + gh + gw) * dh;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += gridDim.x * blockDim.x) {
    const int k = idx % dh, row = idx / dh;
    const int axis = row < gt ? 0 : (row < gt + gh ? 1 : 2);
    const int coord = axis == 0 ? row : (axis == 1 ? row - gt : row - gt - gh);
    axes[idx] = rope_entry(axis, coord, axis == 0 ? gt : (axis == 1 ? gh : gw), d, k, theta, interp, ref);
  }
}
}  // namespace

cudaError_t rope_axes_launch(int gt, int gh, int gw, int head_dim, float theta, int interpolate, int ref_grid,
                             float2* axes, cudaStream_t s) {
  const int d = 2 * ((head_dim / 3) / 2);
  const int total = (gt + gh + gw) * (d / 2);
  if (total <= 0) return cudaSuccess;
  rope_axes_kernel<<<grid_for(total, 256), 256, 0, s>>>(gt, gh, gw, d, (double)theta, interpolate, ref_grid, axes);
  return cudaGetLastError();
}

cudaError_t rope_table_launch(int gt, int gh, int gw, int head_dim, float theta, int interpolate, int ref_grid,
                              float2* table, cudaStream_t s) {
  const int d = 2 * ((head_dim / 3) / 2);
  const int total = gt * gh * gw * 3 * (d / 2);
  if (total <= 0) return cudaSuccess;
  rope_table_kernel<<<grid_for(total, 256), 256, 0, s>>>(gt, gh, gw, d, (double)theta, interpolate, ref_grid, table);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ CLS prefix rows
namespace {
__global__ void prefix_rows_kernel(float* X, int B, int N, int D, const float* cls, const float* pos,
                                   const float* vec) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float v = cls[c];
    if (pos) v += pos[c];  // row 0 of a learned table belongs to CLS
    if (vec) v += vec[c];
    X[(size_t)b * N * D + c] = v;
  }
}
}  // namespace

cudaError_t prefix_rows_launch(float* X, int B, int N, int D, const float* cls, const float* pos, const float* vec,
                               cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  return launch_kernel(prefix_rows_kernel, dim3(B), dim3(256), 0, s, X, B, N, D, cls, pos, vec);
}

// ------------------------------------------------------------------ bounded-wait probe
namespace {
__global__ void wait_timeout_probe_kernel(int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl wc{&abort_flag, err, limit_ns};
    mbar_wait(smem_u32(&bar), 0, wc);  // nobody arrives: returns false after limit_ns
  }
  __syncthreads();
}
}  // namespace

cudaError_t wait_timeout_probe_launch(int* err, uint64_t limit_ns, cudaStream_t s) {
  wait_timeout_probe_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ host helpers
namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}
}  // namespace

bool make_tmap_2d_bf16(CUtensorMap* tm, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_2d_out(CUtensorMap* tm, const void* ptr, uint64_t rows, uint64_t cols, int elem_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || (elem_bytes != 2 && elem_bytes != 4)) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (cuuint64_t)elem_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)(64 / elem_bytes), 32};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
            const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_3d_bf16(CUtensorMap* tm, const void* ptr, uint64_t B, uint64_t N, uint64_t cols, uint32_t box_rows,
                       uint32_t box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || (box_cols != 64 && box_cols != 32)) return false;
  const cuuint64_t dims[3] = {cols, N, B};
  const cuuint64_t strides[2] = {cols * 2, N * cols * 2};
  const cuuint32_t box[3] = {box_cols, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static std::atomic<int> cached{0};
  int v = cached.load();
  if (v == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
    cached.store(v);
  }
  return v;
}

bool& pdl_launches() {
  thread_local bool on = false;
  return on;
}

uint64_t default_wait_limit_ns() { return 1000000000ull; }  // 1 s: far above any legitimate wait

}  // namespace jepa
