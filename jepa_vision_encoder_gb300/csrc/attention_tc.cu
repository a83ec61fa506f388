// attention_tc.cu -- tcgen05 flash attention for sm_103a, head_dim 64, bf16 in / bf16 out,
// fp32 softmax and accumulation: o = softmax(q k^T / sqrt(64) + mask) v per (item, head)
// ("Architecture", Attention and precision; Block-causal attention).
//
// One CTA = one tile of 128 queries of one (item, head); two CTAs per SM (256 TMEM columns
// and ~82 KB of shared memory each), so one CTA's softmax overlaps the other's MMAs.
//   warp 0      TMA: the Q tile once, then K and V tiles of 128 keys into a 2-stage ring
//               (3-D tensor map over qkv [B][N][3D]: rows beyond N read as zeros)
//   warp 1      MMA: S = Q K^T (4 x M128 N128 K16, both K-major) into TMEM columns [0,128);
//               after the softmax has written P, O += P V (8 x M128 N64 K16, P read from TMEM
//               columns [128,192), V MN-major in shared memory) into columns [192,256)
//   warps 2..5  softmax, one query row per thread (TMEM lane): pass 1 row max of S, pass 2
//               p = 2^(s*log2e/8 - m) stored to TMEM as bf16; the running max only moves when
//               a tile raises it by more than 2^8, and then O is rescaled in TMEM; at the end
//               o = O / l is written as bf16.
// Block-causal: a query tile only visits keys below the last frame its rows can see, and the
// per-element predicate runs only on tiles that straddle a frame edge, the CLS row/column or N.
#include <cuda_bf16.h>

#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace jepa {

namespace {

constexpr int kQT = 128;  // queries per CTA
constexpr int kKT = 128;  // keys per tile
constexpr int kHD = 64;
constexpr int kTileBytes = kQT * kHD * 2;  // 16 KB: one 128 x 64 bf16 tile
constexpr int kKvStages = 2;
constexpr int kSmemBytes = 1024 + kTileBytes * (1 + 2 * kKvStages) + 256;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColP = 128, kColO = 192;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p stays below 2^8 between rescales

struct AttnDev {
  int N, H, D;
  int attn_mode, prefix, frame_tokens;
  __nv_bfloat16* out;
  float scale_log2;
  int* err;
  uint64_t limit_ns;
};

// Visible keys of query row q are [lo, hi).
__device__ __forceinline__ void row_window(const AttnDev& a, int q, int& lo, int& hi) {
  lo = 0;
  hi = a.N;
  if (a.attn_mode == 1 && q >= a.prefix) {
    const int f = (q - a.prefix) / a.frame_tokens;
    lo = a.prefix;
    hi = min(a.N, a.prefix + (f + 1) * a.frame_tokens);
  }
}

__global__ void __launch_bounds__(192, 2) attn_tc_kernel(const __grid_constant__ CUtensorMap tm, AttnDev a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* sQ = smem;
  uint8_t* sK = smem + kTileBytes;                    // kKvStages tiles
  uint8_t* sV = smem + kTileBytes * (1 + kKvStages);  // kKvStages tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kTileBytes * (1 + 2 * kKvStages));
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = bars + 1 + kKvStages;
  uint64_t* s_full = bars + 1 + 2 * kKvStages;
  uint64_t* p_full = s_full + 1;
  uint64_t* o_done = s_full + 2;
  uint64_t* mma_done = s_full + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * kQT, h = blockIdx.y, b = blockIdx.z;

  // Key range of this query tile: a tile holding a prefix (CLS) row sees every key.
  int kv_end = a.N;
  if (a.attn_mode == 1 && q0 >= a.prefix) {
    const int q_last = min(q0 + kQT - 1, a.N - 1);
    kv_end = min(a.N, a.prefix + ((q_last - a.prefix) / a.frame_tokens + 1) * a.frame_tokens);
  }
  const int num_kt = (kv_end + kKT - 1) / kKT;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    for (int s = 0; s < kKvStages; ++s) {
      mbar_init(smem_u32(kv_full + s), 1);
      mbar_init(smem_u32(kv_empty + s), 1);
    }
    mbar_init(smem_u32(s_full), 1);
    mbar_init(smem_u32(p_full), 128);
    mbar_init(smem_u32(o_done), 1);
    mbar_init(smem_u32(mma_done), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, a.err, a.limit_ns};

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t qb = smem_u32(q_full);
      mbar_arrive_expect_tx(qb, kTileBytes);
      tma_load_3d(smem_u32(sQ), &tm, qb, h * kHD, q0, b);
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_phase = 0;
      for (int j = 0; j < num_kt; ++j) {
        if (!mbar_wait(smem_u32(kv_empty + stage), phase ^ 1u, wc)) break;
        const uint32_t fb = smem_u32(kv_full + stage);
        mbar_arrive_expect_tx(fb, 2 * kTileBytes);
        tma_load_3d(smem_u32(sK + stage * kTileBytes), &tm, fb, a.D + h * kHD, j * kKT, b);
        tma_load_3d(smem_u32(sV + stage * kTileBytes), &tm, fb, 2 * a.D + h * kHD, j * kKT, b);
        armed |= 1u << stage;
        armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == kKvStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      mbar_drain(qb, 0, a.limit_ns, a.err);
      for (int s = 0; s < kKvStages; ++s)
        if (armed & (1u << s)) mbar_drain(smem_u32(kv_full + s), (armed_phase >> s) & 1u, a.limit_ns, a.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kKT, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, kHD, 0, 1);
      bool ok = mbar_wait(smem_u32(q_full), 0, wc);
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t q_addr = smem_u32(sQ);
      for (int j = 0; j < num_kt && ok; ++j) {
        if (!mbar_wait(smem_u32(kv_full + stage), phase, wc)) break;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(sK + stage * kTileBytes), v_addr = smem_u32(sV + stage * kTileBytes);
#pragma unroll
        for (int k = 0; k < kHD / 16; ++k)
          mma_ss(tmem + kColS, smem_desc_sw128(q_addr + k * 32, 1024, 1024),
                 smem_desc_sw128(k_addr + k * 32, 1024, 1024), idesc_s, k != 0 ? 1u : 0u);
        mma_commit(smem_u32(s_full));
        if (!mbar_wait(smem_u32(p_full), (uint32_t)(j & 1), wc)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kKT / 16; ++k)
          mma_ts(tmem + kColO, tmem + kColP + k * 8, smem_desc_sw128(v_addr + k * 2048, 1024, 1024), idesc_o,
                 (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(smem_u32(o_done));
        mma_commit(smem_u32(kv_empty + stage));
        if (++stage == kKvStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      mma_commit(smem_u32(mma_done));
      mbar_drain(smem_u32(mma_done), 0, a.limit_ns, a.err);
    }
  } else {
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row inside the tile = TMEM lane
    const int q = q0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    int lo, hi;
    row_window(a, q, lo, hi);
    const float sc = a.scale_log2;
    float m_run = -INFINITY, l_run = 0.0f;
    bool ok = true;
    for (int j = 0; j < num_kt; ++j) {
      const int k0 = j * kKT;
      // uniform per CTA: does this tile need the element predicate?
      bool masked = (k0 + kKT > a.N);
      if (a.attn_mode == 1) {
        const int q_first = max(q0, a.prefix), q_last = min(q0 + kQT - 1, a.N - 1);
        const int f_min = (q_first - a.prefix) / a.frame_tokens;
        const int k_last = min(k0 + kKT - 1, a.N - 1);
        const int fk_max = (k_last - a.prefix) / a.frame_tokens;
        masked = masked || q0 < a.prefix || k0 < a.prefix || fk_max > f_min || q_last < q_first;
      }
      if (!mbar_wait(smem_u32(s_full), (uint32_t)(j & 1), wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // pass 1: row max of the raw scores
      float mx = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < kKT / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(lane_base + kColS + c * 32, rr);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int key = k0 + c * 32 + e;
          const float s = __uint_as_float(rr[e]);
          if (!masked || (key >= lo && key < hi)) mx = fmaxf(mx, s);
        }
      }
      const float m_tile = mx * sc;
      float m_new = m_run;
      if (j == 0 || m_tile > m_run + kRescaleThreshold) m_new = fmaxf(m_run, m_tile);
      // O and P are free once the previous P V has completed
      if (j > 0) {
        if (!mbar_wait(smem_u32(o_done), (uint32_t)((j - 1) & 1), wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // The rescale is decided per row, but the TMEM ld/st are warp-collective (.sync.aligned):
        // the whole warp rescales when any of its rows needs it, the others with alpha = 1.
        const bool need = m_new > m_run;
        const float alpha = need ? ex2_approx(m_run - m_new) : 1.0f;
        l_run *= alpha;
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
          for (int c = 0; c < kHD / 16; ++c) {
            uint32_t ov[16];
            tmem_ld16(lane_base + kColO + c * 16, ov);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st16(lane_base + kColO + c * 16, ov);
          }
        }
      }
      m_run = m_new;
      const float base = (m_run == -INFINITY) ? 0.0f : m_run;
      // pass 2: p = 2^(s*sc - m) as bf16 pairs into the P columns
      float lsum = 0.0f;
#pragma unroll 1
      for (int c = 0; c < kKT / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(lane_base + kColS + c * 32, rr);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int key = k0 + c * 32 + e;
          float p0 = ex2_approx(fmaf(__uint_as_float(rr[e]), sc, -base));
          float p1 = ex2_approx(fmaf(__uint_as_float(rr[e + 1]), sc, -base));
          if (masked) {
            if (!(key >= lo && key < hi)) p0 = 0.0f;
            if (!(key + 1 >= lo && key + 1 < hi)) p1 = 0.0f;
          }
          lsum += p0 + p1;
          pk[e >> 1] = pack_bf16x2(p0, p1);
        }
        tmem_st16(lane_base + kColP + c * 16, pk);
      }
      l_run += lsum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(p_full));
    }
    bool store = ok && num_kt > 0 && mbar_wait(smem_u32(o_done), (uint32_t)((num_kt - 1) & 1), wc);
    store = __all_sync(0xffffffffu, store);  // the TMEM loads below are warp-collective
    if (store) {
      tc_fence_after();
      const float inv = (l_run > 0.0f) ? 1.0f / l_run : 0.0f;
      __nv_bfloat16* dst = a.out + ((size_t)b * a.N + q) * a.D + h * kHD;
#pragma unroll 1
      for (int c = 0; c < kHD / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(lane_base + kColO + c * 32, ov);
        tmem_ld_wait();
        if (q < a.N) {
          uint4 w[4];
          uint32_t* wp = reinterpret_cast<uint32_t*>(w);
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            wp[e >> 1] = pack_bf16x2(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv);
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int t = 0; t < 4; ++t) d4[t] = w[t];
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t gemm_tc_init_attributes();

cudaError_t tc_kernels_init() {
  static std::once_flag once;
  static cudaError_t result = cudaSuccess;
  std::call_once(once, [] {
    result = gemm_tc_init_attributes();
    if (result == cudaSuccess)
      result = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  return result;
}

cudaError_t attention_tc_launch(const CUtensorMap& tmQKV, const AttnParams& p, int* err, uint64_t limit_ns,
                                cudaStream_t s) {
  if (p.head_dim != kHD) return cudaErrorInvalidValue;
  if (p.B <= 0 || p.N <= 0) return cudaSuccess;
  AttnDev a;
  a.N = p.N;
  a.H = p.H;
  a.D = p.H * kHD;
  a.attn_mode = p.attn_mode;
  a.prefix = p.prefix;
  a.frame_tokens = p.frame_tokens > 0 ? p.frame_tokens : 1;
  a.out = reinterpret_cast<__nv_bfloat16*>(p.out);
  a.scale_log2 = 1.4426950408889634f / 8.0f;  // log2(e) / sqrt(64)
  a.err = err;
  a.limit_ns = limit_ns;
  dim3 grid((p.N + kQT - 1) / kQT, p.H, p.B);
  attn_tc_kernel<<<grid, 192, kSmemBytes, s>>>(tmQKV, a);
  return cudaGetLastError();
}

}  // namespace jepa
