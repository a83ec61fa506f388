// attention_tc.cu -- tcgen05 flash attention for sm_103a, head_dim 64 (or 32: the masked
// predictor's heads, in 64-byte-swizzled tiles), bf16 in / bf16 out, fp32 softmax and
// accumulation: o = softmax(q k^T / sqrt(head_dim) + mask) v per (item, head)
// ("Architecture", Attention and precision; Block-causal attention).
//
// One CTA = two tiles of 128 queries (Q0, Q1) of one (item, head), one CTA per SM:
//   warps 0..3  softmax of Q0, warps 4..7 softmax of Q1: one query row per thread (TMEM lane).
//               The thread reads its 128 scores from TMEM once, takes their max (independent
//               three-input max chains) and writes p = 2^(s*log2e/8 - m) to TMEM as bf16 pairs
//               (packed two-lane FMA for the scaling, four two-lane chains for the row sum). The
//               running max only moves when a tile raises it by more than 2^8, and then the
//               warp rescales its O rows in TMEM. At the end o = O / l is stored as bf16.
//   warp 8      TMA: Q0 and Q1 once, then K and V tiles of 128 keys into a 3-stage ring
//               (3-D tensor map over qkv [B][N][3D]: rows beyond N read as zeros).
//   warps 10-11 MMA, taking the key tiles in turn (each warp runs its loop whole, an elected
//               lane issues); per key tile j:
//               S_g(j+1) = Q_g K(j+1)^T for both tiles as soon as warpgroup g has read S_g(j)
//               into registers (so the next scores are ready when its softmax ends), then
//               O_g += P_g(j) V(j) for both tiles once P_g(j) is in TMEM.
//               S = Q K^T: M128 N128 K16 x (HD/16) (both K-major); O += P V: M128 N(HD) K16 x8
//               with P read from TMEM and V MN-major in shared memory.
//   warp 9      idle: the third warpgroup is whole so that it can hand registers to the softmax
//               warpgroups (setmaxnreg: 200 per softmax thread, 104 in warpgroup 2).
// TMEM (512 columns): S0 [0,128) S1 [128,256) P0 [256,320) P1 [320,384) O0, O1 from 384 (HD each).
// Block-causal: a CTA only visits keys below the last frame its rows can see, and a query tile
// that sees none of a key tile's keys writes P = 0 without computing exponentials. When a frame is
// a whole number of 128-row tiles, the query and key tiles start at the first patch row (after the
// CLS prefix), so every tile lies inside one frame and no tile needs the per-element predicate
// (except the ragged end at N); the CTAs covering one frame's rows (heaviest frames first) see
// key tiles 0 .. the end of that frame. The prefix rows, which see every key, are one extra CTA per
// (item, head) computing them in fp32 on the CUDA cores. Otherwise the tiles start at row 0 and
// tiles that straddle a frame edge, the CLS row/column or N take the per-element predicate.
#include <cuda_bf16.h>

#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace jepa {

namespace {

constexpr int kQT = 128;  // queries per tile (per softmax warpgroup)
constexpr int kKT = 128;  // keys per tile
constexpr int kKvStages = 3;
constexpr int kIssuers = 2, kFirstIssuer = 10;  // MMA issuing warps 10 and 11
// barriers (q_full, kv_full, kv_empty, s_full, o_done, mma_done, p_full, s_free), TMEM slot, abort flag
static_assert((1 + 2 * kKvStages + 5 + 4 * kIssuers) * 8 + 8 <= 256, "barrier area");
// Per head width HD (64, or 32 for the masked predictor): a 128-row tile of q, k or v is
// 128 x HD bf16 with HD x 2 bytes per row, stored in the TMA / UMMA swizzle of that row length.
template <int HD>
struct Width {
  static constexpr int kTileBytes = kQT * HD * 2;  // 16 KB (HD 64) or 8 KB (HD 32)
  static constexpr int kSmemBytes = 1024 + kTileBytes * (2 + 2 * kKvStages) + 256;
  static constexpr uint32_t kRowBytes = HD * 2;    // 128 or 64: the swizzle span
};
// softmax warpgroups 0 and 1; warpgroup 2: TMA warp 8, idle warp 9, MMA warps 10 and 11
constexpr int kThreads = 384;
// Register budgets after the split: 200 per softmax thread, 104 in warpgroup 2; launched with 168
// per thread (384 x 168 = 64512 >= 256 x 200 + 128 x 104 = 64512).
constexpr uint32_t kSoftmaxRegs = 200, kProducerRegs = 104, kLaunchRegs = 168;
static_assert(256 * kSoftmaxRegs + 128 * kProducerRegs <= kThreads * kLaunchRegs, "register split exceeds the launch");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColP = 256, kColO = 384;  // + 128 / 64 / HD per tile
constexpr float kRescaleThreshold = 8.0f;                 // log2 units: p stays below 2^8 between rescales

struct AttnDev {
  int N, H, D;
  int attn_mode, prefix, frame_tokens;
  int out_hd;  // output columns per head: the head width
  __nv_bfloat16* out;
  const __nv_bfloat16* qkv;  // [B*N, 3D]: read by the prefix-row CTAs
  float scale_log2;
  int* err;
  uint64_t limit_ns;
  // frame-aligned block-causal tiling: tiles start at row k_origin (= prefix), the first
  // n_prefix_ctas CTAs of each (head, item) compute the prefix rows, the next n_main CTAs take the
  // 256-row query blocks, last block first
  int aligned, k_origin, n_prefix_ctas, n_main;
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

// Last key (exclusive) any query in [q_begin, q_end) can see.
__device__ __forceinline__ int keys_needed(const AttnDev& a, int q_begin, int q_end) {
  if (a.attn_mode != 1 || q_begin < a.prefix) return a.N;
  const int q_last = min(q_end, a.N) - 1;
  if (q_last < q_begin) return 0;
  return min(a.N, a.prefix + ((q_last - a.prefix) / a.frame_tokens + 1) * a.frame_tokens);
}

// Shared-memory descriptor of a 128 x HD tile: 128-byte swizzle (8-row groups 1024 bytes apart)
// for HD 64, 64-byte swizzle (groups 512 bytes apart) for HD 32; K-major for q and k, MN-major
// for v; the leading offset is unused (one swizzle atom across the row).
template <int HD>
__device__ __forceinline__ uint64_t tile_desc(uint32_t saddr) {
  if constexpr (HD == 64) return smem_desc_sw128(saddr, 1024, 1024);
  else return smem_desc_sw64(saddr, 512, 512);
}

// The prefix (CLS) rows of one (item, head) under the block-causal mask: each sees every key, so
// this is full attention of `prefix` query rows over N keys, in fp32 on the CUDA cores: scores of
// all keys into shared memory (one key row per thread at a time), their max, p = 2^(s - max) and
// the sum, then o = sum_k p_k v_k with each warp taking every twelfth key and each lane HD/32 of
// the columns, the warps' partial rows added in shared memory. sm holds N + (kThreads/32 + 1) * HD + 64
// floats.
template <int HD>
__device__ __forceinline__ void attn_prefix_rows(const AttnDev& a, int h, int b, float* sm) {
  constexpr int kWarps = kThreads / 32, kPer = HD / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t ld = 3 * (size_t)a.D;
  const __nv_bfloat16* rows = a.qkv + (size_t)b * a.N * ld;
  float* sc = sm;                        // [N] scores, then p
  float* part = sm + ((a.N + 3) & ~3);   // [kWarps][HD] partial outputs
  float* qv = part + kWarps * HD;        // [HD] the query row
  float* red = qv + HD;                  // [2 * kWarps] reductions
  for (int r = 0; r < a.prefix; ++r) {
    if (tid < HD) qv[tid] = __bfloat162float(rows[(size_t)r * ld + h * HD + tid]);
    __syncthreads();
    float mx = -INFINITY;
    for (int k = tid; k < a.N; k += kThreads) {
      const uint4* kr = reinterpret_cast<const uint4*>(rows + (size_t)k * ld + a.D + h * HD);
      float dot = 0.0f;
#pragma unroll
      for (int u = 0; u < HD / 8; ++u) {
        const uint4 w = __ldg(kr + u);
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[t]));
          dot = fmaf(qv[u * 8 + 2 * t], f.x, dot);
          dot = fmaf(qv[u * 8 + 2 * t + 1], f.y, dot);
        }
      }
      const float sv = dot * a.scale_log2;
      sc[k] = sv;
      mx = fmaxf(mx, sv);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = red[0];
    for (int w = 1; w < kWarps; ++w) mx = fmaxf(mx, red[w]);
    float sum = 0.0f;
    for (int k = tid; k < a.N; k += kThreads) {
      const float pv = ex2_approx(sc[k] - mx);
      sc[k] = pv;
      sum += pv;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) red[kWarps + warp] = sum;
    __syncthreads();  // every p is in sc and every partial sum in red
    float acc[kPer];
#pragma unroll
    for (int t = 0; t < kPer; ++t) acc[t] = 0.0f;
    for (int k = warp; k < a.N; k += kWarps) {
      const float pv = sc[k];
      const __nv_bfloat16* vr = rows + (size_t)k * ld + 2 * a.D + h * HD + lane * kPer;
      if constexpr (kPer == 2) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(vr));
        acc[0] = fmaf(pv, f.x, acc[0]);
        acc[1] = fmaf(pv, f.y, acc[1]);
      } else {
        acc[0] = fmaf(pv, __bfloat162float(*vr), acc[0]);
      }
    }
#pragma unroll
    for (int t = 0; t < kPer; ++t) part[warp * HD + lane * kPer + t] = acc[t];
    __syncthreads();
    if (tid < HD) {
      float l = 0.0f, o = 0.0f;
      for (int w = 0; w < kWarps; ++w) {
        l += red[kWarps + w];
        o += part[w * HD + tid];
      }
      a.out[((size_t)b * a.N + r) * (a.H * a.out_hd) + h * a.out_hd + tid] = __float2bfloat16_rn(o / l);
    }
    __syncthreads();  // sc, part, qv and red are reused by the next prefix row
  }
}

// BC: the block-causal form (per-row key windows, tiles without visible keys skipped, the
// frame-aligned tiling and the prefix-row CTAs); the full-attention form compiles without them.
template <int HD, bool BC>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ CUtensorMap tm, AttnDev a) {
  constexpr int kHD = HD;
  constexpr int kTileBytes = Width<HD>::kTileBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* sQ = smem;                                 // 2 tiles
  uint8_t* sK = smem + 2 * kTileBytes;                // kKvStages tiles
  uint8_t* sV = smem + (2 + kKvStages) * kTileBytes;  // kKvStages tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (2 + 2 * kKvStages) * kTileBytes);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = bars + 1 + kKvStages;
  uint64_t* s_full = bars + 1 + 2 * kKvStages;  // [2]
  uint64_t* o_done = s_full + 2;                // [2]
  uint64_t* mma_done = s_full + 4;
  // Per issuer (key tile j on [g][j % kIssuers]), so that each barrier's phases are waited in
  // order by one warp: a parity wait cannot tell a phase two ahead from the one before.
  uint64_t* p_full = s_full + 5;                // [2][kIssuers]: P_g(j) is in TMEM
  uint64_t* s_free = p_full + 2 * kIssuers;     // [2][kIssuers]: the warpgroup has read S_g(j)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_free + 2 * kIssuers);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the aligned form's grid is (head, item, job) so that jobs run heaviest first over all (item,
  // head) pairs: job 0 the prefix rows, then the query blocks from the last frame back
  const bool aligned = BC && a.aligned;
  const int k_origin = BC ? a.k_origin : 0;
  const int h = aligned ? blockIdx.x : blockIdx.y, b = aligned ? blockIdx.y : blockIdx.z;
  const int job = aligned ? (int)blockIdx.z : (int)blockIdx.x;
  if (aligned && job < a.n_prefix_ctas) {
    pdl_trigger();
    pdl_wait();  // qkv comes from the previous kernel
    attn_prefix_rows<HD>(a, h, b, reinterpret_cast<float*>(smem));
    return;
  }
  // first query row of the CTA: 256-row blocks from k_origin, in the aligned form last block first
  const int q0 = aligned ? k_origin + (a.n_main - 1 - (job - a.n_prefix_ctas)) * 2 * kQT : job * 2 * kQT;
  const int num_kt = BC ? (keys_needed(a, q0, q0 + 2 * kQT) - k_origin + kKT - 1) / kKT : (a.N + kKT - 1) / kKT;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    for (int s = 0; s < kKvStages; ++s) {
      mbar_init(smem_u32(kv_full + s), 1);
      mbar_init(smem_u32(kv_empty + s), 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(smem_u32(s_full + g), 1);
      mbar_init(smem_u32(o_done + g), 1);
      for (int w = 0; w < kIssuers; ++w) {
        mbar_init(smem_u32(p_full + g * kIssuers + w), 128);
        mbar_init(smem_u32(s_free + g * kIssuers + w), 4);
      }
    }
    mbar_init(smem_u32(mma_done), kIssuers);  // each issuer's last commit
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm);
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, a.err, a.limit_ns};
  pdl_trigger();
  pdl_wait();  // qkv comes from the previous kernel; the output may still be read by older ones
  if (warp >= 8) {
  // warpgroup 2 gives registers back to the softmax warpgroups (each branch is entered by a
  // whole warpgroup, which executes its register budget change together)
  warpgroup_regs_dec<kProducerRegs>();
  if (warp == 8) {
    if (lane == 0) {
      const uint32_t qb = smem_u32(q_full);
      mbar_arrive_expect_tx(qb, 2 * kTileBytes);
      tma_load_3d(smem_u32(sQ), &tm, qb, h * kHD, q0, b);
      tma_load_3d(smem_u32(sQ + kTileBytes), &tm, qb, h * kHD, q0 + kQT, b);
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_phase = 0;
      for (int j = 0; j < num_kt; ++j) {
        if (!mbar_wait(smem_u32(kv_empty + stage), phase ^ 1u, wc)) break;
        const uint32_t fb = smem_u32(kv_full + stage);
        mbar_arrive_expect_tx(fb, 2 * kTileBytes);
        tma_load_3d(smem_u32(sK + stage * kTileBytes), &tm, fb, a.D + h * kHD, k_origin + j * kKT, b);
        tma_load_3d(smem_u32(sV + stage * kTileBytes), &tm, fb, 2 * a.D + h * kHD, k_origin + j * kKT, b);
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
  } else if (warp >= kFirstIssuer && warp < kFirstIssuer + kIssuers) {
    // Warps 10 and 11 take the key tiles in turn (tile j by warp 10 + j % 2, tile 0's scores by
    // warp 10): issuing MMAs slows the other warps of the issuer's sub-partition, and a tile's
    // softmax ends with its slowest lane quarter, so the cost is shared by two sub-partitions.
    // The issuers need no ordering among themselves: S_g(j+1) follows s_free_g(j), and P_g(j) V(j)
    // follows p_full_g(j), which the softmax arrives on only after o_done_g(j-1).
    // Each warp runs its loop whole (waits and descriptor arithmetic warp-uniform); one elected
    // lane issues each MMA and commit.
    const int me = warp - kFirstIssuer;
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, kKT, 0, 0);
    constexpr uint32_t idesc_o = idesc_bf16_f32(128, kHD, 0, 1);
    // descriptors built once; a K step or a stage only moves the start address
    const uint64_t q_desc = tile_desc<HD>(smem_u32(sQ));
    const uint64_t k_desc = tile_desc<HD>(smem_u32(sK));
    const uint64_t v_desc = tile_desc<HD>(smem_u32(sV));
    auto wait = [&](const uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), parity, wc));
    };
    auto issue_s = [&](int g, int st) {
      const uint64_t qd = desc_advance(q_desc, g * kTileBytes), kd = desc_advance(k_desc, st * kTileBytes);
      const uint32_t d = tmem + kColS + g * 128;
#pragma unroll
      for (int k = 0; k < kHD / 16; ++k) mma_ss_warp(d, desc_advance(qd, k * 32), desc_advance(kd, k * 32), idesc_s, k != 0);
      mma_commit_warp(smem_u32(s_full + g));
    };
    auto issue_pv = [&](int g, int st, int j) {
      const uint64_t vd = desc_advance(v_desc, st * kTileBytes);
      const uint32_t d = tmem + kColO + g * kHD, p = tmem + kColP + g * 64;
#pragma unroll
      for (int k = 0; k < kKT / 16; ++k)  // 16 keys = 16 rows of V per K step
        mma_ts_warp(d, p + k * 8, desc_advance(vd, k * 16 * Width<HD>::kRowBytes), idesc_o, (j > 0 || k > 0) ? 1u : 0u);
      mma_commit_warp(smem_u32(o_done + g));
    };
    bool ok = num_kt > 0;
    if (me == 0 && ok) {
      ok = wait(q_full, 0) && wait(kv_full, 0);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        issue_s(1, 0);
      }
    }
    for (int j = me; j < num_kt && ok; j += kIssuers) {
      const int stage = j % kKvStages, nst = (j + 1) % kKvStages;
      const uint32_t nph = (uint32_t)(((j + 1) / kKvStages) & 1);
      const bool more = j + 1 < num_kt;
      // S_g(j+1) as soon as warpgroup g holds S_g(j) in registers (while it computes P), for
      // both tiles, then P_g(j) V(j) once P is in TMEM: neither tile's next scores wait
      // behind the other tile's softmax
      if (more) {
#pragma unroll
        for (int g = 0; g < 2 && ok; ++g) {
          if (!(ok = wait(s_free + g * kIssuers + me, (uint32_t)((j / kIssuers) & 1)))) break;
          // K(j+1) after s_free_0(j): that implies S(j) has run, so tile j-2 (the stage's previous
          // load, whose wait another issuer may have done) is complete and the parity cannot alias
          if (g == 0 && !(ok = wait(kv_full + nst, nph))) break;
          tc_fence_after();
          issue_s(g, nst);
        }
      }
#pragma unroll
      for (int g = 0; g < 2 && ok; ++g) {
        if (!(ok = wait(p_full + g * kIssuers + me, (uint32_t)((j / kIssuers) & 1)))) break;
        tc_fence_after();
        issue_pv(g, stage, j);
      }
      if (!ok) break;
      mma_commit_warp(smem_u32(kv_empty + stage));  // K(j), V(j) no longer read once these complete
    }
    mma_commit_warp(smem_u32(mma_done));
    mbar_drain(smem_u32(mma_done), 0, a.limit_ns, a.err);
  }
  } else {
    warpgroup_regs_inc<kSoftmaxRegs>();
    const int g = warp >> 2;                 // which query tile
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;       // query row inside the tile = TMEM lane
    const int qt0 = q0 + g * kQT;            // first query of this tile
    const int q = qt0 + r;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + kColS + g * 128;
    const uint32_t tP = tmem + lane_off + kColP + g * 64;
    const uint32_t tO = tmem + lane_off + kColO + g * kHD;
    int lo, hi;
    row_window(a, q, lo, hi);
    const float sc = a.scale_log2;
    // uniform per warpgroup: the tile's query span for the mask classification
    const int q_first = max(qt0, a.prefix), q_last = min(qt0 + kQT - 1, a.N - 1);
    const int f_min = (BC && q_last >= q_first) ? (q_first - a.prefix) / a.frame_tokens : 0;
    // key tiles this tile's rows can see at all; past them the group writes P = 0 (no exponentials)
    const int kt_vis = BC ? (keys_needed(a, qt0, qt0 + kQT) - k_origin + kKT - 1) / kKT : num_kt;
    float m_run = -INFINITY, l_run = 0.0f;
    bool ok = true;
    for (int j = 0; j < num_kt; ++j) {
      const int k0 = k_origin + j * kKT;
      const bool none = BC && j >= kt_vis;  // uniform over the warpgroup
      bool masked = (k0 + kKT > a.N);
      if (BC && !aligned) {
        const int k_last = min(k0 + kKT - 1, a.N - 1);
        const int fk_max = (k_last - a.prefix) / a.frame_tokens;
        masked = masked || qt0 < a.prefix || k0 < a.prefix || fk_max > f_min || q_last < q_first;
      }
      if (!mbar_wait(smem_u32(s_full + g), (uint32_t)(j & 1), wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the thread's 128 raw scores, read from TMEM in one load
      uint32_t sr[kKT];
      tmem_ld128(tS, sr);
      tmem_ld_wait(sr);
      uint32_t (&s)[kKT / 32][32] = *reinterpret_cast<uint32_t (*)[kKT / 32][32]>(&sr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(s_free + g * kIssuers + j % kIssuers));  // S may be overwritten now
      if (none) {  // no key of this tile is visible to these rows: P = 0, m and l unchanged
        if (j > 0) {
          if (!mbar_wait(smem_u32(o_done + g), (uint32_t)((j - 1) & 1), wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        uint32_t zero[kKT / 2];
#pragma unroll
        for (int e = 0; e < kKT / 2; ++e) zero[e] = 0u;
        tmem_st64(tP, zero);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(p_full + g * kIssuers + j % kIssuers));
        continue;
      }
      if (masked) {  // invisible keys score -inf: they lose the max and give p = 0
#pragma unroll
        for (int c = 0; c < kKT / 32; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int key = k0 + c * 32 + e;
            if (!(key >= lo && key < hi)) s[c][e] = __float_as_uint(-INFINITY);
          }
      }
      // row max: four independent chains of three-input max
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < kKT / 32; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 8)
#pragma unroll
          for (int t = 0; t < 4; ++t)
            mx4[t] = fmax3(mx4[t], __uint_as_float(s[c][e + 2 * t]), __uint_as_float(s[c][e + 2 * t + 1]));
      const float m_tile = fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3])) * sc;
      float m_new = m_run;
      if (j == 0 || m_tile > m_run + kRescaleThreshold) m_new = fmaxf(m_run, m_tile);
      const bool need = j > 0 && m_new > m_run;  // O (and l) of this row move to the new max
      const float alpha = need ? ex2_approx(m_run - m_new) : 1.0f;
      m_run = m_new;
      const float base = (m_run == -INFINITY) ? 0.0f : m_run;
      // p = 2^(s*sc - m) two keys at a time, as bf16 pairs into the P columns
      const float2 sc2 = make_float2(sc, sc), nb2 = make_float2(-base, -base);
      float2 ls2[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                       make_float2(0.0f, 0.0f)};  // four short chains for the row sum
      uint32_t pk[kKT / 2];
#pragma unroll
      for (int c = 0; c < kKT / 32; ++c) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 x =
              __ffma2_rn(make_float2(__uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1])), sc2, nb2);
          const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          ls2[(e >> 1) & 3] = __fadd2_rn(ls2[(e >> 1) & 3], p);
          pk[c * 16 + (e >> 1)] = pack_bf16x2(p.x, p.y);
        }
      }
      if (j > 0) {
        // P and O of this tile are free once its previous P V has completed: the exponentials
        // above did not need to wait for it, only the P store and the rescale of O do
        if (!mbar_wait(smem_u32(o_done + g), (uint32_t)((j - 1) & 1), wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // The rescale is decided per row, but the TMEM ld/st are warp-collective (.sync.aligned):
        // the whole warp rescales when any of its rows needs it, the others with alpha = 1.
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
          for (int c = 0; c < kHD / 16; ++c) {
            uint32_t ov[16];
            tmem_ld16(tO + c * 16, ov);
            tmem_ld_wait(ov);
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st16(tO + c * 16, ov);
          }
        }
      }
      l_run *= alpha;
      tmem_st64(tP, pk);
      const float2 l01 = __fadd2_rn(ls2[0], ls2[1]), l23 = __fadd2_rn(ls2[2], ls2[3]);
      l_run += (l01.x + l23.x) + (l01.y + l23.y);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(p_full + g * kIssuers + j % kIssuers));
    }
    bool store = ok && num_kt > 0 && mbar_wait(smem_u32(o_done + g), (uint32_t)((num_kt - 1) & 1), wc);
    store = __all_sync(0xffffffffu, store);  // the TMEM loads below are warp-collective
    if (store) {
      tc_fence_after();
      const float inv = (l_run > 0.0f) ? 1.0f / l_run : 0.0f;
      __nv_bfloat16* dst = a.out + ((size_t)b * a.N + q) * (a.H * a.out_hd) + h * a.out_hd;
#pragma unroll 1
      for (int c = 0; c < a.out_hd / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tO + c * 32, ov);
        tmem_ld_wait(ov);
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
  if (warp == 9) {
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
    auto set = [&](const void* f, int bytes) {
      if (result == cudaSuccess) result = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    };
    set((const void*)attn_tc_kernel<64, false>, Width<64>::kSmemBytes);
    set((const void*)attn_tc_kernel<64, true>, Width<64>::kSmemBytes);
    set((const void*)attn_tc_kernel<32, false>, Width<32>::kSmemBytes);
    set((const void*)attn_tc_kernel<32, true>, Width<32>::kSmemBytes);
  });
  return result;
}

cudaError_t attention_tc_launch(const CUtensorMap& tmQKV, const AttnParams& p, int* err, uint64_t limit_ns,
                                cudaStream_t s) {
  if (p.head_dim != 64 && p.head_dim != 32) return cudaErrorInvalidValue;
  if (p.B <= 0 || p.N <= 0) return cudaSuccess;
  AttnDev a;
  a.N = p.N;
  a.H = p.H;
  a.D = p.H * p.head_dim;
  a.attn_mode = p.attn_mode;
  a.prefix = p.prefix;
  a.frame_tokens = p.frame_tokens > 0 ? p.frame_tokens : 1;
  a.out = reinterpret_cast<__nv_bfloat16*>(p.out);
  a.qkv = reinterpret_cast<const __nv_bfloat16*>(p.qkv);
  a.out_hd = p.head_dim;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)p.head_dim);  // log2(e) / sqrt(head width)
  a.err = err;
  a.limit_ns = limit_ns;
  // Frame-aligned block-causal tiling when frames are whole tiles: the patch rows N - prefix are
  // frames of frame_tokens rows; the prefix rows' scores must fit the shared memory.
  const int smem_bytes = p.head_dim == 32 ? Width<32>::kSmemBytes : Width<64>::kSmemBytes;
  const long long prefix_smem = 4LL * (((long long)p.N + 3) & ~3LL) + 4LL * (kThreads / 32 + 1) * p.head_dim + 4LL * 64;
  a.aligned = p.attn_mode == 1 && p.frame_tokens % kKT == 0 && (p.N - p.prefix) % p.frame_tokens == 0 &&
              p.prefix <= 8 && (p.prefix == 0 || (p.qkv != nullptr && prefix_smem <= smem_bytes - 1024));
  a.k_origin = a.aligned ? p.prefix : 0;
  a.n_prefix_ctas = (a.aligned && p.prefix > 0) ? 1 : 0;
  a.n_main = a.aligned ? (p.N - p.prefix + 2 * kQT - 1) / (2 * kQT) : (p.N + 2 * kQT - 1) / (2 * kQT);
  const dim3 grid = a.aligned ? dim3(p.H, p.B, a.n_prefix_ctas + a.n_main) : dim3(a.n_main, p.H, p.B);
  const bool bc = p.attn_mode == 1;
  if (p.head_dim == 32)
    return launch_kernel(bc ? attn_tc_kernel<32, true> : attn_tc_kernel<32, false>, grid, dim3(kThreads),
                         Width<32>::kSmemBytes, s, tmQKV, a);
  return launch_kernel(bc ? attn_tc_kernel<64, true> : attn_tc_kernel<64, false>, grid, dim3(kThreads),
                       Width<64>::kSmemBytes, s, tmQKV, a);
}

}  // namespace jepa
