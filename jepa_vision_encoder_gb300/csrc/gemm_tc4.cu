// gemm_tc4.cu -- the pair GEMM (gemm_tc2.cu) run by clusters of four CTAs: two 2-SM pairs that
// compute the two 256 x 256 tiles of one 256-row block side by side (columns n and n + 256) and
// share its rows of A through TMA multicast.
//
// Each pair reads the same 256 rows of A for its K blocks. Here every CTA loads one 64-row
// quarter of a stage's A and multicasts it to the CTA at the same place in the other pair (ranks
// r and r ^ 2), so each CTA fetches 8 KB of A per 64-deep K block instead of 16 (24 KB of
// operands instead of 32 with its 16 KB half of B). B is loaded as in the pair kernel.
//
// Hand-offs (ranks 0, 1 = pair 0 with leader 0; ranks 2, 3 = pair 1 with leader 2):
//   full[s]   on each leader: every copy landing in its pair (its own and the other pair's
//             multicast quarters of A, both halves of B) completes there; the leader arms it with
//             the 64 KB of the pair's stage.
//   empty[s]  on every CTA: two arrivals, one multicast commit from each leader, since the slot
//             of a stage in any CTA is written by copies of both pairs.
//   tfull / tempty / mma_done: per pair, as in the pair kernel.
// Both pairs walk the same sequence of row blocks and K blocks, so their stage rings stay in step.
// Every wait is bounded; each leader drains the phases it armed and its MMAs, and the four CTAs
// meet at a cluster barrier before TMEM is freed.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace jepa {

namespace {

constexpr int kTileM = 256, kTileN = 256, kBK = 64;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kABytes = 128 * kBK * 2;      // 16 KB of A per CTA and stage
constexpr int kAQuarter = 64 * kBK * 2;     // 8 KB: the 64 rows one CTA loads and multicasts
constexpr int kBBytes = 128 * kBK * 2;      // 16 KB: this CTA's 128 columns of B
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kStages = 6;
constexpr int kEpiBytes = kEpiWarps * 4096;
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kEpiBytes + 512;
constexpr uint32_t kTmemCols = 2 * kTileN;

// Copy of one 64-row box of A into the same offset of the CTAs in `mask`; each copy completes on
// the barrier at `bar`'s offset in the leader of the receiving CTA's pair (`bar` names a leader).
__device__ __forceinline__ void tma_load_2d_pair_mc(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int32_t x,
                                                    int32_t y, uint16_t mask, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster.L2::cache_hint"
      " [%0], [%1, {%4, %5}], [%2], %3, %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "h"(mask), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

template <int EK>
__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_tc4_kernel(const __grid_constant__ CUtensorMap tmA64, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmO, EpiArgs epi, int M, int N, int K, int* err,
                    uint64_t limit_ns) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* sA = smem;                           // kStages x 16 KB
  uint8_t* sB = smem + kStages * kABytes;       // kStages x 16 KB
  uint8_t* sEpi = smem + kStages * kStageBytes; // kEpiWarps x 4 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + kEpiBytes);
  uint64_t* full = bars;                        // [kStages], used on the leaders
  uint64_t* empty = bars + kStages;             // [kStages]
  uint64_t* tfull = bars + 2 * kStages;         // [2]
  uint64_t* tempty = bars + 2 * kStages + 2;    // [2], used on the leaders
  uint64_t* mma_done = bars + 2 * kStages + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();      // 0..3
  const uint32_t r2 = rank & 1u;                // which half of the pair's 256 rows
  const uint32_t pr = rank >> 1;                // which pair: columns n0 + 256 * pr
  const uint32_t leader = rank & ~1u;
  const uint16_t pair_mask = (uint16_t)(3u << leader);
  const int cluster = blockIdx.x >> 2, num_clusters = gridDim.x >> 2;
  const int num_n2 = N / (2 * kTileN), num_k = K / kBK;
  const int num_units = ((M + kTileM - 1) / kTileM) * num_n2;  // 256 x 512 blocks

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 2);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(tfull + a), 1);
      mbar_init(smem_u32(tempty + a), 2 * kEpiWarps);
    }
    mbar_init(smem_u32(mma_done), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA64);
    prefetch_tmap(&tmB);
    if (EK != kEpiPatch) prefetch_tmap(&tmO);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers exist before any remote arrive, copy or commit
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{abort_flag, err, limit_ns};
  pdl_trigger();
  pdl_wait();  // A and the residual stream come from earlier kernels

  if (warp == 0) {
    if (lane == 0) {
      // A of the residual GEMMs (attention output, FFN hidden) is read once: let it go first
      const uint64_t a_policy = (EK == kEpiResidual) ? l2_policy_evict_first() : l2_policy_evict_normal();
      const uint64_t b_policy = l2_policy_evict_last();
      // this CTA's quarter of A goes to itself and to the CTA holding the same rows in the other pair
      const uint16_t a_mask = (uint16_t)((1u << rank) | (1u << (rank ^ 2u)));
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_phase = 0;
      bool ok = true;
      for (int u = cluster; u < num_units && ok; u += num_clusters) {
        const int mb = u / num_n2, nb = u % num_n2;
        const int a_row = mb * kTileM + (int)r2 * 128 + (int)pr * 64;  // the quarter this CTA loads
        const int b_row = (2 * nb + (int)pr) * kTileN + (int)r2 * 128;
        for (int kb = 0; kb < num_k; ++kb) {
          if (!mbar_wait(smem_u32(empty + stage), phase ^ 1u, wc)) {
            ok = false;
            break;
          }
          const uint32_t fb_lead = mapa_shared(smem_u32(full + stage), leader);
          if (r2 == 0) mbar_arrive_expect_tx(smem_u32(full + stage), 2 * kStageBytes);
          tma_load_2d_pair_mc(smem_u32(sA + stage * kABytes + (int)pr * kAQuarter), &tmA64, fb_lead, kb * kBK, a_row,
                              a_mask, a_policy);
          tma_load_2d_pair_hint(smem_u32(sB + stage * kBBytes), &tmB, fb_lead, kb * kBK, b_row, b_policy);
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // each leader drains every phase it armed (copies from all four CTAs land on it)
      if (r2 == 0)
        for (int s = 0; s < kStages; ++s)
          if (armed & (1u << s)) mbar_drain(smem_u32(full + s), (armed_phase >> s) & 1u, limit_ns, err);
    }
  } else if (warp == 1) {
    if (r2 == 0) {
      // leader: the MMA issuer of its pair (whole warp runs the loop, an elected lane issues)
      constexpr uint32_t idesc = idesc_bf16_f32(kTileM, kTileN, 0, 0);
      const uint64_t a_desc = smem_desc_sw128(smem_u32(sA), 1024, 1024);
      const uint64_t b_desc = smem_desc_sw128(smem_u32(sB), 1024, 1024);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int u = cluster; u < num_units && ok; u += num_clusters) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(tempty + acc), acc_phase ^ 1u, wc))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kTileN);
        for (int kb = 0; kb < num_k; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(full + stage), phase, wc))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = desc_advance(a_desc, stage * kABytes), bd = desc_advance(b_desc, stage * kBBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_ss_pair_warp(d_tmem, desc_advance(ad, k * 32), desc_advance(bd, k * 32), idesc, (kb | k) != 0 ? 1u : 0u);
          mma_commit_pair_mc_warp(smem_u32(empty + stage), 0xF);  // the slot is free in all four CTAs
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair_mc_warp(smem_u32(tfull + acc), pair_mask);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      mma_commit_pair_mc_warp(smem_u32(mma_done), (uint16_t)(1u << rank));
      mbar_drain(smem_u32(mma_done), 0, limit_ns, err);
    }
  } else {
    const int q = warp & 3;
    constexpr int kChunks = kTileN / 32 / 2;
    const int half = (warp - 2) >> 2;
    const uint32_t tempty_lead = mapa_shared(smem_u32(tempty), leader);
    EpiStage stage{sEpi + (warp - 2) * 4096, 0};
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = cluster; u < num_units; u += num_clusters) {
      const int mb = u / num_n2, nb = u % num_n2;
      const int m0 = mb * kTileM + (int)r2 * 128, n0 = (2 * nb + (int)pr) * kTileN;
      if (!mbar_wait(smem_u32(tfull + acc), acc_phase, wc)) break;
      tc_fence_after();
      const int y0 = m0 + q * 32;
      const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kTileN);
      epi_warp_tile<EK, kChunks>(epi, &tmO, stage, lane, trow, y0, n0, half);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(tempty_lead + (uint32_t)(acc * sizeof(uint64_t)));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    stage.finish(lane);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both pairs' MMAs are drained (no copy or commit into a peer remains)
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <int EK>
cudaError_t launch_quad(const CUtensorMap& tmA64, const CUtensorMap& tmB, const CUtensorMap& tmO, const EpiArgs& epi,
                        int M, int N, int K, int* err, uint64_t limit_ns, cudaStream_t s) {
  const int units = ((M + kTileM - 1) / kTileM) * (N / (2 * kTileN));
  const int max_clusters = gemm_tc4_max_clusters();
  const int clusters = units < max_clusters ? units : max_clusters;
  return launch_kernel(gemm_tc4_kernel<EK>, dim3(4 * clusters), dim3(kThreads), kSmemBytes, s, tmA64, tmB, tmO, epi, M,
                       N, K, err, limit_ns);
}

}  // namespace

cudaError_t gemm_tc4_init_attributes() {
  cudaError_t e = cudaSuccess;
  auto set = [&](const void* f) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  };
  set((const void*)gemm_tc4_kernel<kEpiBias>);
  set((const void*)gemm_tc4_kernel<kEpiGelu>);
  set((const void*)gemm_tc4_kernel<kEpiResidual>);
  set((const void*)gemm_tc4_kernel<kEpiQkvRope>);
  set((const void*)gemm_tc4_kernel<kEpiPatch>);
  return e;
}

// Clusters of four that can be resident at once (0 if none).
int gemm_tc4_max_clusters() {
  static int cached = -1;
  if (cached < 0) {
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(4 * (num_sms() / 4), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc4_kernel<kEpiBias>, &cfg) != cudaSuccess || n < 0) {
      cudaGetLastError();
      n = 0;
    }
    cached = n;
  }
  return cached;
}

cudaError_t gemm_tc4_launch(const CUtensorMap& tmA64, const CUtensorMap& tmB, const CUtensorMap& tmO,
                            const EpiArgs& epi, int M, int N, int K, int* err, uint64_t limit_ns, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (N % 512 || K % kBK || gemm_tc4_max_clusters() <= 0) return cudaErrorInvalidValue;
  switch (epi.kind) {
    case kEpiBias: return launch_quad<kEpiBias>(tmA64, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    case kEpiGelu: return launch_quad<kEpiGelu>(tmA64, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    case kEpiResidual: return launch_quad<kEpiResidual>(tmA64, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    case kEpiQkvRope: return launch_quad<kEpiQkvRope>(tmA64, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    case kEpiPatch: return launch_quad<kEpiPatch>(tmA64, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace jepa
