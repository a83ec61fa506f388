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
  const float2* rope;     // [Np, 3, dh] (cos, sin) of the item's patch grid, or
  const float2* rope_axes;  // [gt + gh + gw, dh]: the t rows, then h, then w (used when not null)
  int rope_gt, rope_gh, rope_gw;
  int rows_per_item, prefix, n_head, head_dim, rope_layout, rope_d;
  // optional: the patch position id of every output row m (rope_ids[m]), for token sequences that
  // are not the patch grid in order (the masked predictor's context and target tokens)
  const int* rope_ids;
  // patch embedding: input row m = patch i of item b (i = m % patches_per_item)
  int patches_per_item;
  const float* pos;       // [rows_per_item, N] or null
  const float* vec;       // [N] or null
};

__device__ __forceinline__ float gelu_erf(float x) { return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f)); }

// GELU of the bf16 tensor-core epilogue, two values at a time in packed fp32 arithmetic.
// q = Phi(-|x|) = erfc(|x| / sqrt(2)) / 2 is evaluated as exp(-x^2 / 2) * sum_k c_k a^k with
// a = min(|x|, 16), a fit of the scaled complementary error function (gelu_fit.py in this
// directory prints the coefficients and the bound |q - Phi(-|x|)| <= 1.8e-5, so the GELU is
// within 1.8e-5 |x|, far below bf16 rounding); past |x| = 16 the exponential is below the smallest
// normal float and q is 0. Then GELU(x) = x Phi(x) = x / 2 + |x| (1/2 - q).
__device__ __forceinline__ float2 gelu_fast2(float2 x) {
  constexpr float c[7] = {5.0000000000e-01f, -3.9842587502e-01f, 2.4521308688e-01f, -1.1811391615e-01f,
                          4.0482376797e-02f, -8.2998320074e-03f, 7.3464815428e-04f};
  constexpr float kNegHalfLog2e = -0.72134752044448170f;  // -log2(e) / 2
  const float2 ax = make_float2(fabsf(x.x), fabsf(x.y));
  const float2 a = make_float2(fminf(ax.x, 16.0f), fminf(ax.y, 16.0f));
  const float2 t = __fmul2_rn(__fmul2_rn(x, x), make_float2(kNegHalfLog2e, kNegHalfLog2e));
  float2 p = make_float2(c[6], c[6]);
#pragma unroll
  for (int k = 5; k >= 0; --k) p = __ffma2_rn(p, a, make_float2(c[k], c[k]));
  const float2 q = __fmul2_rn(p, make_float2(ex2_approx(t.x), ex2_approx(t.y)));
  const float2 h = __ffma2_rn(q, make_float2(-1.0f, -1.0f), make_float2(0.5f, 0.5f));  // 1/2 - q
  return __ffma2_rn(ax, h, __fmul2_rn(x, make_float2(0.5f, 0.5f)));
}

// The (cos, sin) rows (dh entries each) of the t, h and w axes of output row m, row p of its item.
__device__ __forceinline__ void rope_axis_rows(const EpiArgs& a, int m, int p, int dh, const float2* (&r)[3]) {
  // rows past M (the ragged tail of the last tile, never stored) must not read past rope_ids
  const int pp = a.rope_ids != nullptr ? (m < a.M ? __ldg(a.rope_ids + m) : 0) : p - a.prefix;
  if (a.rope_axes != nullptr) {
    const int hw = a.rope_gh * a.rope_gw;
    const int t = pp / hw, rem = pp - t * hw, h = rem / a.rope_gw, w = rem - h * a.rope_gw;
    r[0] = a.rope_axes + (size_t)t * dh;
    r[1] = a.rope_axes + (size_t)(a.rope_gt + h) * dh;
    r[2] = a.rope_axes + (size_t)(a.rope_gt + a.rope_gh + w) * dh;
  } else {
    const float2* row = a.rope + (size_t)pp * 3 * dh;
    r[0] = row;
    r[1] = row + dh;
    r[2] = row + 2 * dh;
  }
}

// 3-D RoPE on 32 consecutive columns of one head of width 64 starting at head dim J0 (0 or 32):
// d = 2*((64/3)/2) = 20 rotated dims per axis (t: 0-19, h: 20-39, w: 40-59), 60-63 untouched.
// Every index is a compile-time constant; LAYOUT 0 = tiled (frequency j mod 10), 1 = interleaved
// (frequency j / 2). r = the token's (cos, sin) rows of its three axes, 10 entries each.
template <int J0, int LAYOUT>
__device__ __forceinline__ void rope_hd64_chunk(float (&v)[32], const float2* const (&r)[3]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    constexpr int kD = 20, kDh = 10;
    const int j = J0 + e;  // even dim inside the head
    if (j < 3 * kD) {
      const int axis = j / kD, jj = j - axis * kD;
      const int k0 = LAYOUT == 0 ? (jj % kDh) : (jj >> 1);
      const int k1 = LAYOUT == 0 ? ((jj + 1) % kDh) : ((jj + 1) >> 1);
      const float2 c0 = __ldg(r[axis] + k0);
      const float2 c1 = __ldg(r[axis] + k1);
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
__device__ __forceinline__ void rope_generic(const EpiArgs& a, int m, int p, int n0, float (&v)[E]) {
  const int D = a.n_head * a.head_dim;
  const int d = a.rope_d, dh = d >> 1;
  const float2* rows[3];
  rope_axis_rows(a, m, p, dh, rows);
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
        const float2 cs = __ldg(rows[axis] + k);
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
  } else if (a.kind == kEpiQkvRope && (a.rope != nullptr || a.rope_axes != nullptr)) {
    const int p = m % a.rows_per_item;
    bool done = p < a.prefix;  // prefix (CLS) rows are not rotated
    if constexpr (E == 32) {
      // tcgen05 GEMM fast path: a 32-column chunk is one half of one head of width 64
      if (!done && a.head_dim == 64 && (n0 & 31) == 0) {
        if (n0 < 2 * a.n_head * 64) {
          const float2* rows[3];
          rope_axis_rows(a, m, p, 10, rows);
          const bool upper = (n0 & 63) != 0;
          if (a.rope_layout == 0) {
            if (upper) rope_hd64_chunk<32, 0>(v, rows); else rope_hd64_chunk<0, 0>(v, rows);
          } else {
            if (upper) rope_hd64_chunk<32, 1>(v, rows); else rope_hd64_chunk<0, 1>(v, rows);
          }
        }
        done = true;
      }
    }
    if (!done) rope_generic<E>(a, m, p, n0, v);  // any even head width, any fragment (the fp32 SIMT GEMM)
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
// The bias of a warp's 32-column chunk is held one value per lane (lane e: column n0 + e), loaded
// while the tile's main loop still runs (epi_bias_lanes), and handed to every row by shuffles.
template <int EK>
__device__ __forceinline__ void epi_math_tc(const EpiArgs& a, int m, int n0, float (&v)[32], float blane) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const float2 b = make_float2(__shfl_sync(0xffffffffu, blane, e), __shfl_sync(0xffffffffu, blane, e + 1));
    const float2 r = __fadd2_rn(make_float2(v[e], v[e + 1]), b);
    v[e] = r.x;
    v[e + 1] = r.y;
  }
  if constexpr (EK == kEpiGelu) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const float2 g = gelu_fast2(make_float2(v[e], v[e + 1]));
      v[e] = g.x;
      v[e + 1] = g.y;
    }
  } else if constexpr (EK == kEpiQkvRope) {
    const int p = m % a.rows_per_item;
    if ((a.rope != nullptr || a.rope_axes != nullptr) && p >= a.prefix && n0 < 2 * a.n_head * a.head_dim) {
      if (a.head_dim == 64) {
        const float2* rows[3];
        rope_axis_rows(a, m, p, 10, rows);
        const bool upper = (n0 & 63) != 0;
        if (a.rope_layout == 0) {
          if (upper) rope_hd64_chunk<32, 0>(v, rows); else rope_hd64_chunk<0, 0>(v, rows);
        } else {
          if (upper) rope_hd64_chunk<32, 1>(v, rows); else rope_hd64_chunk<0, 1>(v, rows);
        }
      } else {
        rope_generic<32>(a, m, p, n0, v);  // any even head width
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
      if (add)  // the residual stream is read again by the next LayerNorm: keep it in L2
        tma_reduce_add_2d_hint(tm, smem_u32(buf), x, y, l2_policy_evict_last());
      else
        tma_store_2d(tm, smem_u32(buf), x, y);
      bulk_commit();
    }
    ++n;
  }
  // Every store of this warp done reading shared memory (before the CTA exits; the global writes
  // complete with the grid, before any dependent grid passes its wait).
  __device__ __forceinline__ void finish(int lane) {
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
  }
};

// One 32-column chunk of row m (= first row y0 of the warp's slab + lane) of a tensor-core GEMM:
// math, then staged store (bf16: one piece) or staged fp32 add into the residual stream (two).
template <int EK>
__device__ __forceinline__ void epi_chunk_tc(const EpiArgs& a, const CUtensorMap* tm_out, EpiStage& st, int lane,
                                             int y0, int n0, float (&v)[32], float blane) {
  if constexpr (EK == kEpiPatch) {
    if (a.prefix == 0 && a.rows_per_item == a.patches_per_item) {
      // output rows are the patch rows (no CLS): bias (+ position row) (+ modality vector), then
      // the same staged TMA store as the other epilogues, in fp32
      epi_math_tc<EK>(a, y0 + lane, n0, v, blane);
      if (a.pos != nullptr) {  // row i of the item's table (a fixed table: patch rows only)
        const float4* p4 =
            reinterpret_cast<const float4*>(a.pos + (size_t)((y0 + lane) % a.patches_per_item) * a.N + n0);
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 q = __ldg(p4 + e / 4);
          v[e] += q.x;
          v[e + 1] += q.y;
          v[e + 2] += q.z;
          v[e + 3] += q.w;
        }
      }
      if (a.vec != nullptr) {
        const float4* v4 = reinterpret_cast<const float4*>(a.vec + n0);
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 m = __ldg(v4 + e / 4);
          v[e] += m.x;
          v[e + 1] += m.y;
          v[e + 2] += m.z;
          v[e + 3] += m.w;
        }
      }
      uint32_t w[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(v[e]);
      st.put(lane, w, tm_out, n0, y0, false);
#pragma unroll
      for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(v[16 + e]);
      st.put(lane, w, tm_out, n0 + 16, y0, false);
    } else {
      epi_fragment<32, false>(a, y0 + lane, n0, v);  // rows remapped per item: stores from registers
    }
  } else {
    epi_math_tc<EK>(a, y0 + lane, n0, v, blane);
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

// RoPE of one 32-column half (J0 = 0: head dims 0-31, J0 = 32: dims 32-63) of a width-64 head,
// with the row's (cos, sin) values already in registers: cs[axis][k].
template <int J0, int LAYOUT>
__device__ __forceinline__ void rope_hd64_regs(float (&v)[32], const float2 (&cs)[3][10]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    constexpr int kD = 20, kDh = 10;
    const int j = J0 + e;
    if (j < 3 * kD) {
      const int axis = j / kD, jj = j - axis * kD;
      const int k0 = LAYOUT == 0 ? (jj % kDh) : (jj >> 1);
      const int k1 = LAYOUT == 0 ? ((jj + 1) % kDh) : ((jj + 1) >> 1);
      const float x0 = v[e], x1 = v[e + 1];
      v[e] = fmaf(x0, cs[axis][k0].x, -x1 * cs[axis][k0].y);
      v[e + 1] = fmaf(x1, cs[axis][k1].x, x0 * cs[axis][k1].y);
    }
  }
}

// QKV epilogue of a warp whose chunks are all head halves J0 (chunks 2i + J0/32 of the tile): the
// row's (cos, sin) values for the two axes those dims use come from epi_prepare (loaded once per
// tile, before the accumulator is ready), and every chunk rotates from registers.
template <int EK, int NCHUNK>
struct EpiPre;

template <int J0, int NCHUNK>
__device__ __forceinline__ void epi_warp_qkv_hd64(const EpiArgs& a, const CUtensorMap* tm, EpiStage& st, int lane,
                                                  uint32_t trow, int y0, int n_tile0,
                                                  const EpiPre<kEpiQkvRope, NCHUNK>& pre) {
  constexpr int kA0 = J0 == 0 ? 0 : 1;  // axes touched by this half: t, h (J0 = 0) or h, w (J0 = 32)
  float2 cs[3][10];
#pragma unroll
  for (int ax = 0; ax < 3; ++ax)
#pragma unroll
    for (int k = 0; k < 10; ++k)
      cs[ax][k] = (ax == kA0 || ax == kA0 + 1) ? pre.cs[ax == kA0 ? 0 : 1][k] : make_float2(1.0f, 0.0f);
  const float (&bl)[NCHUNK] = pre.bl;
  const int qk_cols = 2 * a.n_head * 64;
  uint32_t r[2][32];
  tmem_ld32(trow + (J0 / 32) * 32, r[0]);
#pragma unroll
  for (int i = 0; i < NCHUNK; ++i) {
    const int c = 2 * i + J0 / 32;
    tmem_ld_wait(r[i & 1]);
    if (i + 1 < NCHUNK) tmem_ld32(trow + (c + 2) * 32, r[(i + 1) & 1]);
    float v[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[i & 1][e]);
    const int n0 = n_tile0 + c * 32;
    if (n0 >= a.N) continue;  // past the last column (a ragged last tile): nothing to store
    epi_math_tc<kEpiBias>(a, y0 + lane, n0, v, bl[i]);
    if (n0 < qk_cols) {  // q and k columns rotate (warp-uniform); v columns pass
      if (a.rope_layout == 0)
        rope_hd64_regs<J0, 0>(v, cs);
      else
        rope_hd64_regs<J0, 1>(v, cs);
    }
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
    st.put(lane, w, tm, n0, y0, false);
  }
}

// 3-D RoPE of one head of width 32 held in v: d = 2*((32/3)/2) = 10 rotated dims per axis (t: 0-9,
// h: 10-19, w: 20-29), 30-31 untouched; 5 frequencies per axis, so in the tiled layout the odd
// member of a pair wraps (frequency (jj + 1) mod 5). cs = the row's (cos, sin) values, cs[axis][k].
template <int LAYOUT>
__device__ __forceinline__ void rope_hd32_regs(float (&v)[32], const float2 (&cs)[3][5]) {
#pragma unroll
  for (int e = 0; e < 30; e += 2) {
    constexpr int kD = 10, kDh = 5;
    const int axis = e / kD, jj = e - axis * kD;
    const int k0 = LAYOUT == 0 ? (jj % kDh) : (jj >> 1);
    const int k1 = LAYOUT == 0 ? ((jj + 1) % kDh) : ((jj + 1) >> 1);
    const float x0 = v[e], x1 = v[e + 1];
    v[e] = fmaf(x0, cs[axis][k0].x, -x1 * cs[axis][k0].y);
    v[e + 1] = fmaf(x1, cs[axis][k1].x, x0 * cs[axis][k1].y);
  }
}

// QKV epilogue of a warp for heads of width 32 (every 32-column chunk is one head): the row's 15
// (cos, sin) values are loaded once per tile and each q / k chunk rotates from registers.
template <int NCHUNK>
__device__ __forceinline__ void epi_warp_qkv_hd32(const EpiArgs& a, const CUtensorMap* tm, EpiStage& st, int lane,
                                                  uint32_t trow, int y0, int n_tile0, int half,
                                                  const float (&bl)[NCHUNK]) {
  const int m = y0 + lane;
  const int p = m % a.rows_per_item;
  const bool rot = (a.rope != nullptr || a.rope_axes != nullptr) && p >= a.prefix;
  float2 cs[3][5];
#pragma unroll
  for (int ax = 0; ax < 3; ++ax)
#pragma unroll
    for (int k = 0; k < 5; ++k) cs[ax][k] = make_float2(1.0f, 0.0f);
  if (rot) {
    const float2* rows[3];
    rope_axis_rows(a, m, p, 5, rows);
#pragma unroll
    for (int ax = 0; ax < 3; ++ax)
#pragma unroll
      for (int k = 0; k < 5; ++k) cs[ax][k] = __ldg(rows[ax] + k);
  }
  const int qk_cols = 2 * a.n_head * 32;
  const int c0 = half * NCHUNK;
  uint32_t r[2][32];
  tmem_ld32(trow + c0 * 32, r[0]);
#pragma unroll
  for (int i = 0; i < NCHUNK; ++i) {
    tmem_ld_wait(r[i & 1]);
    if (i + 1 < NCHUNK) tmem_ld32(trow + (c0 + i + 1) * 32, r[(i + 1) & 1]);
    float v[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[i & 1][e]);
    const int n0 = n_tile0 + (c0 + i) * 32;
    if (n0 >= a.N) continue;  // past the last column (a ragged last tile): nothing to store
    epi_math_tc<kEpiBias>(a, m, n0, v, bl[i]);
    if (n0 < qk_cols) {  // q and k heads rotate (warp-uniform); v heads pass
      if (a.rope_layout == 0)
        rope_hd32_regs<0>(v, cs);
      else
        rope_hd32_regs<1>(v, cs);
    }
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
    st.put(lane, w, tm, n0, y0, false);
  }
}

// Column of chunk i of a warp's share of a tile: QKV with width-64 heads takes every other 32-column
// chunk (the head half `half`), the other kinds the warp's contiguous half of the tile.
template <int EK, int NCHUNK>
__device__ __forceinline__ int epi_chunk_col(const EpiArgs& a, int i, int half) {
  return (EK == kEpiQkvRope && a.head_dim == 64) ? (2 * i + half) * 32 : (half * NCHUNK + i) * 32;
}

// The bias of the warp's chunks of the tile at column n_tile0, one value per lane per chunk,
// requested before the accumulator is ready so that no chunk waits on a load from L2.
template <int EK, int NCHUNK>
__device__ __forceinline__ void epi_bias_lanes(const EpiArgs& a, int lane, int n_tile0, int half, float (&bl)[NCHUNK]) {
#pragma unroll
  for (int i = 0; i < NCHUNK; ++i) {
    const int n = n_tile0 + epi_chunk_col<EK, NCHUNK>(a, i, half) + lane;
    bl[i] = n < a.N ? __ldg(a.bias + n) : 0.0f;  // columns past N: a ragged last tile
  }
}

// What a warp's epilogue of one tile reads besides the accumulator, requested while the tile's
// main loop runs so that no chunk waits on L2: the bias (one value per lane per chunk) and, for QKV
// with width-64 heads, the row's (cos, sin) values of the two axes its head half rotates.
template <int EK, int NCHUNK>
struct EpiPre {
  float bl[NCHUNK];
  float2 cs[2][10];
};

template <int EK, int NCHUNK>
__device__ __forceinline__ void epi_prepare(const EpiArgs& a, int lane, int y0, int n_tile0, int half,
                                            EpiPre<EK, NCHUNK>& pre) {
  epi_bias_lanes<EK, NCHUNK>(a, lane, n_tile0, half, pre.bl);
  if constexpr (EK == kEpiQkvRope) {
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int k = 0; k < 10; ++k) pre.cs[j][k] = make_float2(1.0f, 0.0f);
    const int m = y0 + lane, p = m % a.rows_per_item;
    if (a.head_dim == 64 && (a.rope != nullptr || a.rope_axes != nullptr) && p >= a.prefix) {
      const float2* rows[3];
      rope_axis_rows(a, m, p, 10, rows);
      const float2* r0 = half ? rows[1] : rows[0];  // axes t, h (half 0) or h, w (half 1)
      const float2* r1 = half ? rows[2] : rows[1];
#pragma unroll
      for (int k = 0; k < 10; ++k) {
        pre.cs[0][k] = __ldg(r0 + k);
        pre.cs[1][k] = __ldg(r1 + k);
      }
    }
  }
}

// The epilogue of one warp for one accumulator tile: NCHUNK 32-column chunks of its 32 TMEM lanes
// (rows y0 .. y0+31), the next tcgen05.ld in flight while a chunk is processed. half selects which
// chunks: 0 or 1 of the warp pair sharing the lane quarter; pre = epi_prepare of the tile.
template <int EK, int NCHUNK>
__device__ __forceinline__ void epi_warp_tile(const EpiArgs& a, const CUtensorMap* tm, EpiStage& st, int lane,
                                              uint32_t trow, int y0, int n_tile0, int half,
                                              const EpiPre<EK, NCHUNK>& pre) {
  const float (&bl)[NCHUNK] = pre.bl;
  if constexpr (EK == kEpiQkvRope) {
    if (a.head_dim == 64) {  // heads never straddle a 64-column boundary: chunk parity = head half
      if (half == 0)
        epi_warp_qkv_hd64<0, NCHUNK>(a, tm, st, lane, trow, y0, n_tile0, pre);
      else
        epi_warp_qkv_hd64<32, NCHUNK>(a, tm, st, lane, trow, y0, n_tile0, pre);
      return;
    }
    if (a.head_dim == 32) {
      epi_warp_qkv_hd32<NCHUNK>(a, tm, st, lane, trow, y0, n_tile0, half, bl);
      return;
    }
  }
  const int c0 = half * NCHUNK;
  uint32_t r[2][32];
  tmem_ld32(trow + c0 * 32, r[0]);
#pragma unroll
  for (int i = 0; i < NCHUNK; ++i) {
    tmem_ld_wait(r[i & 1]);
    if (i + 1 < NCHUNK) tmem_ld32(trow + (c0 + i + 1) * 32, r[(i + 1) & 1]);
    float v[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[i & 1][e]);
    if (n_tile0 + (c0 + i) * 32 >= a.N) continue;  // past the last column (a ragged last tile)
    epi_chunk_tc<EK>(a, tm, st, lane, y0, n_tile0 + (c0 + i) * 32, v, bl[i]);
  }
}

}  // namespace jepa
