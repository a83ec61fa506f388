// epilogue.cuh -- what a GEMM does with a row fragment of its fp32 accumulator: the fused
// bias / GELU(erf) / residual / 3-D RoPE / patch-embedding row remap of the encoder.
//
// A fragment is E consecutive columns n0 .. n0+E-1 (n0 even, E even) of output row m, held
// by one thread. The fp32 SIMT GEMM (E = 4) and the patch embedding of the tcgen05 GEMMs call
// epi_fragment, which stores from registers; the other tcgen05 epilogues run the same bias /
// GELU / RoPE arithmetic (epi_math_tc) on 32-column chunks and store through shared memory and
// TMA (EpiStage).
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace jepa {

enum EpiKind : int { kEpiBias = 0, kEpiGelu = 1, kEpiResidual = 2, kEpiQkvRope = 3, kEpiPatch = 4 };

struct EpiArgs {
  int kind;
  int M, N;
  const float* bias;      // [N]
  void* out;              // bf16 or fp32, leading dimension N (PATCH: D = N, remapped rows)
  // 3-D RoPE ("Architecture", 3-D RoPE): rows are tokens of items of rows_per_item tokens,
  // the first `prefix` of which are not rotated; q columns [0, D), k columns [D, 2D).
  const float2* rope;     // [Np, 3, dh] (cos, sin) of the item's patch grid
  int rows_per_item, prefix, n_head, head_dim, rope_layout, rope_d;
  // patch embedding: input row m = patch i of item b (i = m % patches_per_item)
  int patches_per_item;
  const float* pos;       // [rows_per_item, N] or null
  const float* vec;       // [N] or null
};

__device__ __forceinline__ float gelu_erf(float x) { return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f)); }

// 3-D RoPE on 32 consecutive columns of one head of width 64 starting at head dim J0 (0 or 32):
// d = 2*((64/3)/2) = 20 rotated dims per axis (t: 0-19, h: 20-39, w: 40-59), 60-63 untouched.
// Every index is a compile-time constant; LAYOUT 0 = tiled (frequency j mod 10), 1 = interleaved
// (frequency j / 2). row = the token's table [3][10] of (cos, sin).
template <int J0, int LAYOUT>
__device__ __forceinline__ void rope_hd64_chunk(float (&v)[32], const float2* __restrict__ row) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    constexpr int kD = 20, kDh = 10;
    const int j = J0 + e;  // even dim inside the head
    if (j < 3 * kD) {
      const int axis = j / kD, jj = j - axis * kD;
      const int k0 = LAYOUT == 0 ? (jj % kDh) : (jj >> 1);
      const int k1 = LAYOUT == 0 ? ((jj + 1) % kDh) : ((jj + 1) >> 1);
      const float2 c0 = __ldg(row + axis * kDh + k0);
      const float2 c1 = __ldg(row + axis * kDh + k1);
      const float x0 = v[e], x1 = v[e + 1];
      // x cos + rot90(x) sin, rot90(y1, y2) = (-y2, y1): each member uses its own angle
      v[e] = fmaf(x0, c0.x, -x1 * c0.y);
      v[e + 1] = fmaf(x1, c1.x, x0 * c1.y);
    }
  }
}

// 3-D RoPE on E consecutive columns n0.. (n0 even) of token row p of an item, any even head width:
// q columns [0, D) and k columns [D, 2D) are rotated, v columns pass.
template <int E>
__device__ __forceinline__ void rope_generic(const EpiArgs& a, int p, int n0, float (&v)[E]) {
  const int D = a.n_head * a.head_dim;
  const int d = a.rope_d, dh = d >> 1;
  const float2* row = a.rope + (size_t)(p - a.prefix) * 3 * dh;
  float r[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int n = n0 + e;
    r[e] = v[e];
    if (n < 2 * D) {
      const int j = (n % D) % a.head_dim;  // dim inside the head
      if (j < 3 * d) {
        const int axis = j / d, jj = j - axis * d;
        const int k = (a.rope_layout == 0) ? (jj % dh) : (jj >> 1);
        const float2 cs = __ldg(row + axis * dh + k);
        // x cos + rot90(x) sin, rot90(y1, y2) = (-y2, y1) on (even, odd) pairs
        const float partner = v[e ^ 1];
        r[e] = (jj & 1) ? fmaf(v[e], cs.x, partner * cs.y) : fmaf(v[e], cs.x, -partner * cs.y);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = r[e];
}

// OUT_BF16 selects bf16 storage of BIAS / GELU / QKV_ROPE (the bf16 path); RESIDUAL and PATCH
// always store fp32 (the residual stream).
template <int E, bool OUT_BF16>
__device__ __forceinline__ void epi_fragment(const EpiArgs& a, int m, int n0, float (&v)[E]) {
  if (m >= a.M) return;
  if ((E % 4) == 0 && n0 + E <= a.N && (n0 & 3) == 0) {
    const float4* b4 = reinterpret_cast<const float4*>(a.bias + n0);
#pragma unroll
    for (int e = 0; e < E; e += 4) {
      const float4 b = __ldg(b4 + e / 4);
      v[e] += b.x;
      v[e + 1] += b.y;
      v[e + 2] += b.z;
      v[e + 3] += b.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] += (n0 + e < a.N) ? __ldg(a.bias + n0 + e) : 0.0f;
  }

  if (a.kind == kEpiGelu) {
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = gelu_erf(v[e]);
  } else if (a.kind == kEpiQkvRope && a.rope != nullptr) {
    const int p = m % a.rows_per_item;
    bool done = p < a.prefix;  // prefix (CLS) rows are not rotated
    if constexpr (E == 32) {
      // tcgen05 GEMM fast path: a 32-column chunk is one half of one head of width 64
      if (!done && a.head_dim == 64 && (n0 & 31) == 0) {
        if (n0 < 2 * a.n_head * 64) {
          const float2* row = a.rope + (size_t)(p - a.prefix) * 30;
          const bool upper = (n0 & 63) != 0;
          if (a.rope_layout == 0) {
            if (upper) rope_hd64_chunk<32, 0>(v, row); else rope_hd64_chunk<0, 0>(v, row);
          } else {
            if (upper) rope_hd64_chunk<32, 1>(v, row); else rope_hd64_chunk<0, 1>(v, row);
          }
        }
        done = true;
      }
    }
    if (!done) rope_generic<E>(a, p, n0, v);  // any even head width, any fragment (the fp32 SIMT GEMM)
  }

  if (a.kind == kEpiResidual) {
    float* out = reinterpret_cast<float*>(a.out) + (size_t)m * a.N + n0;
    if (n0 + E <= a.N && (E % 4) == 0) {
#pragma unroll
      for (int e = 0; e < E; e += 4) {
        float4 x = *reinterpret_cast<float4*>(out + e);
        x.x += v[e];
        x.y += v[e + 1];
        x.z += v[e + 2];
        x.w += v[e + 3];
        *reinterpret_cast<float4*>(out + e) = x;
      }
    } else {
      for (int e = 0; e < E && n0 + e < a.N; ++e) out[e] += v[e];
    }
    return;
  }
  if (a.kind == kEpiPatch) {
    const int b = m / a.patches_per_item, i = m % a.patches_per_item;
    const int row = a.prefix + i;
    float* out = reinterpret_cast<float*>(a.out) + ((size_t)b * a.rows_per_item + row) * a.N + n0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (n0 + e < a.N) {
        float x = v[e];
        if (a.pos) x += __ldg(a.pos + (size_t)row * a.N + n0 + e);
        if (a.vec) x += __ldg(a.vec + n0 + e);
        v[e] = x;
      }
    }
    if (n0 + E <= a.N && (E % 4) == 0) {
#pragma unroll
      for (int e = 0; e < E; e += 4) *reinterpret_cast<float4*>(out + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
    } else {
      for (int e = 0; e < E && n0 + e < a.N; ++e) out[e] = v[e];
    }
    return;
  }
  // BIAS / GELU / QKV_ROPE store
  if (OUT_BF16) {
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) + (size_t)m * a.N + n0;
    if (n0 + E <= a.N && (E % 8) == 0) {
#pragma unroll
      for (int e = 0; e < E; e += 8) {
        uint4 w;
        w.x = pack_bf16x2(v[e], v[e + 1]);
        w.y = pack_bf16x2(v[e + 2], v[e + 3]);
        w.z = pack_bf16x2(v[e + 4], v[e + 5]);
        w.w = pack_bf16x2(v[e + 6], v[e + 7]);
        *reinterpret_cast<uint4*>(out + e) = w;
      }
    } else {
      for (int e = 0; e < E && n0 + e < a.N; ++e) out[e] = __float2bfloat16_rn(v[e]);
    }
  } else {
    float* out = reinterpret_cast<float*>(a.out) + (size_t)m * a.N + n0;
    if (n0 + E <= a.N && (E % 4) == 0) {
#pragma unroll
      for (int e = 0; e < E; e += 4) *reinterpret_cast<float4*>(out + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
    } else {
      for (int e = 0; e < E && n0 + e < a.N; ++e) out[e] = v[e];
    }
  }
}


// ---------------------------------------------------------------- tensor-core GEMM epilogues
// The tcgen05 GEMMs take the epilogue kind as a template argument (EK) so each kernel holds only
// its own arithmetic. epi_math_tc applies the bias and then GELU or 3-D RoPE to 32 consecutive
// columns n0.. of row m; the caller stages the result in shared memory and stores it with TMA.
template <int EK>
__device__ __forceinline__ void epi_math_tc(const EpiArgs& a, int m, int n0, float (&v)[32]) {
  const float4* b4 = reinterpret_cast<const float4*>(a.bias + n0);  // n0 is warp-uniform: broadcast
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    const float4 b = __ldg(b4 + e / 4);
    v[e] += b.x;
    v[e + 1] += b.y;
    v[e + 2] += b.z;
    v[e + 3] += b.w;
  }
  if constexpr (EK == kEpiGelu) {
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = gelu_erf(v[e]);
  } else if constexpr (EK == kEpiQkvRope) {
    const int p = m % a.rows_per_item;
    if (a.rope != nullptr && p >= a.prefix && n0 < 2 * a.n_head * a.head_dim) {
      if (a.head_dim == 64) {
        const float2* row = a.rope + (size_t)(p - a.prefix) * 30;
        const bool upper = (n0 & 63) != 0;
        if (a.rope_layout == 0) {
          if (upper) rope_hd64_chunk<32, 0>(v, row); else rope_hd64_chunk<0, 0>(v, row);
        } else {
          if (upper) rope_hd64_chunk<32, 1>(v, row); else rope_hd64_chunk<0, 1>(v, row);
        }
      } else {
        rope_generic<32>(a, p, n0, v);  // any even head width
      }
    }
  }
}

// A warp's ring of two 2 KB shared-memory buffers, each 32 rows (one per lane) x 64 bytes, laid
// out with the 64-byte TMA swizzle (16-byte unit u of row r at u ^ ((r >> 1) & 3)), so the
// lanes' 16-byte writes hit distinct banks. put() stores the piece through the output tensor
// map (box 64 bytes x 32 rows) at column x, row y, or adds it into global memory (fp32).
struct EpiStage {
  uint8_t* base;  // 1024-byte aligned, 4 KB
  uint32_t n;     // pieces issued by this warp

  __device__ __forceinline__ void put(int lane, const uint32_t (&w)[16], const CUtensorMap* tm, int x, int y,
                                      bool add) {
    uint8_t* buf = base + (n & 1u) * 2048u;
    if (n >= 2) {  // the store issued two pieces ago read this buffer
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
    }
    uint4* row = reinterpret_cast<uint4*>(buf + lane * 64);
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int u = 0; u < 4; ++u) row[u ^ sw] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (add)
        tma_reduce_add_2d(tm, smem_u32(buf), x, y);
      else
        tma_store_2d(tm, smem_u32(buf), x, y);
      bulk_commit();
    }
    ++n;
  }
  // Every store of this warp complete (before the kernel exits).
  __device__ __forceinline__ void finish(int lane) {
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
};

// One 32-column chunk of row m (= first row y0 of the warp's slab + lane) of a tensor-core GEMM:
// math, then staged store (bf16: one piece) or staged fp32 add into the residual stream (two).
template <int EK>
__device__ __forceinline__ void epi_chunk_tc(const EpiArgs& a, const CUtensorMap* tm_out, EpiStage& st, int lane,
                                             int y0, int n0, float (&v)[32]) {
  if constexpr (EK == kEpiPatch) {
    epi_fragment<32, false>(a, y0 + lane, n0, v);
  } else {
    epi_math_tc<EK>(a, y0 + lane, n0, v);
    if constexpr (EK == kEpiResidual) {
      uint32_t w[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(v[e]);
      st.put(lane, w, tm_out, n0, y0, true);
#pragma unroll
      for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(v[16 + e]);
      st.put(lane, w, tm_out, n0 + 16, y0, true);
    } else {
      uint32_t w[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
      st.put(lane, w, tm_out, n0, y0, false);
    }
  }
}

}  // namespace jepa
