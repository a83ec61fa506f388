// gemm_tc2.cu -- the 2-SM form of the tcgen05 GEMM: out = epilogue(A[M,K] B[N,K]^T) with
// 256 x 256 tiles computed by a cluster of two CTAs on two SMs (tcgen05 cta_group::2).
//
// Each CTA of the pair loads, per 64-wide K block, its own 128 rows of A and its own 128 of the
// tile's 256 columns of B (32 KB per stage instead of the 48 KB a 1-SM 128 x 256 tile needs per
// SM), so the operand traffic into each SM's shared memory drops by a third at the same tensor
// work. Only the even CTA issues the MMAs (M = 256: rows 0-127 land in its TMEM, 128-255 in the
// peer's). (A 256 x 128 pair tile, measured, was slower than both this and the 1-SM tiles at
// every encoder shape.) Tiles are numbered N-fastest: the pairs working at the same time share rows of A (read from
// HBM once) and sweep the weights B, which stay in L2.
//
// Per CTA (320 threads, one CTA per SM, grid = 2 x pairs, tiles strided over pairs):
//   warp 0      TMA producer of this CTA's halves; every copy of the pair completes on the even
//               CTA's stage barrier, which the even CTA arms with the bytes of both halves
//   warp 1      even CTA: MMA issuer (odd CTA: idle)
//   warps 2..9  epilogue of this CTA's 128 rows (two warps per TMEM lane quarter, half the
//               columns each, stored through swizzled shared memory with TMA as in the 1-SM
//               kernel), releasing the accumulator with an arrive on the even CTA.
// Stage and accumulator hand-offs from the even CTA use multicast commits to both CTAs.
// Every wait is bounded; the even CTA drains every stage phase it armed (both CTAs' copies)
// and its MMAs, then both CTAs meet at a cluster barrier before TMEM is freed.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace jepa {

namespace {

constexpr int kTileM = 256;   // rows per pair tile (128 per CTA)
constexpr int kBK = 64;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kEpiBytes = kEpiWarps * 4096;          // two 2 KB staging buffers per epilogue warp

template <int TN>
struct PairCfg {
  static constexpr int kBRows = TN / 2;              // B rows each CTA loads
  static constexpr int kABytes = 128 * kBK * 2;      // 16 KB: 128 rows x 64 bf16
  static constexpr int kBBytes = kBRows * kBK * 2;   // 16 KB (TN 256) or 8 KB (TN 128)
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (6 * 32768) / kStageBytes;  // 6 or 8: 192 KB of operand stages
  static constexpr uint32_t kTmemCols = 2 * TN;      // two accumulators
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kEpiBytes + 512;
};

template <int TN, int EK>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmO, EpiArgs epi, int M, int N, int K, int* err,
                    uint64_t limit_ns) {
  using C = PairCfg<TN>;
  constexpr int kStages = C::kStages, kTileN = TN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* sA = smem;                              // kStages x 16 KB
  uint8_t* sB = smem + kStages * C::kABytes;       // kStages x kBBytes
  uint8_t* sEpi = smem + kStages * C::kStageBytes; // kEpiWarps x 4 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + kEpiBytes);
  uint64_t* full = bars;                           // own copies landed
  uint64_t* empty = bars + kStages;                // stage free (multicast from the even CTA)
  // bars + 2 * kStages .. + 3 * kStages: unused (keeps the layout of the barrier block)
  uint64_t* tfull = bars + 3 * kStages;            // accumulator ready (multicast)
  uint64_t* tempty = bars + 3 * kStages + 2;       // even CTA: accumulator drained by both CTAs
  uint64_t* mma_done = bars + 3 * kStages + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * kStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;
  // N need not be a multiple of the tile: the last column tile's rows of B past N load as zeros
  // (TMA fill) and its columns past N are not stored
  const int num_m = (M + kTileM - 1) / kTileM, num_n = (N + kTileN - 1) / kTileN, num_k = K / kBK;
  const int num_tiles = num_m * num_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(tfull + a), 1);
      mbar_init(smem_u32(tempty + a), 2 * kEpiWarps);
    }
    mbar_init(smem_u32(mma_done), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (EK != kEpiPatch) prefetch_tmap(&tmO);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrive or multicast
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{abort_flag, err, limit_ns};
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // Both CTAs load their halves; every copy completes on the even CTA's stage barrier,
      // which the even CTA arms with the bytes of both halves (tx-count may run ahead of the
      // arm within a phase: the phase cannot complete before the even CTA's arrive).
      const uint64_t a_policy = l2_policy_evict_first(), b_policy = l2_policy_evict_last();
      // The weights are written by no kernel of the sequence: the first tile's first stages of
      // B are requested (and, on the even CTA, armed) before waiting for the previous kernel,
      // whose tail this CTA may overlap; A and the residual stream come from earlier kernels.
      // The loop's first kStages waits for a free stage pass at once (fresh barriers), so every
      // stage armed here also gets its A copies.
      const int pre = pair < num_tiles ? (num_k < kStages ? num_k : kStages) : 0;
      uint32_t phase = 0, armed = 0, armed_phase = 0;
      for (int kb = 0; kb < pre; ++kb) {
        const uint32_t fb_even = mapa_shared(smem_u32(full + kb), 0);
        if (rank == 0) mbar_arrive_expect_tx(smem_u32(full + kb), 2 * C::kStageBytes);
        tma_load_2d_pair_hint(smem_u32(sB + kb * C::kBBytes), &tmB, fb_even, kb * kBK,
                              (pair % num_n) * kTileN + (int)rank * C::kBRows, b_policy);
        armed |= 1u << kb;
      }
      pdl_wait();
      int stage = 0, it = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += num_pairs) {
        const int m0 = (tile / num_n) * kTileM + (int)rank * 128, n0 = (tile % num_n) * kTileN + (int)rank * C::kBRows;
        for (int kb = 0; kb < num_k; ++kb, ++it) {
          if (!mbar_wait(smem_u32(empty + stage), phase ^ 1u, wc)) {
            ok = false;
            break;
          }
          const uint32_t fb_even = mapa_shared(smem_u32(full + stage), 0);
          if (rank == 0 && it >= pre) mbar_arrive_expect_tx(smem_u32(full + stage), 2 * C::kStageBytes);
          if (EK == kEpiResidual)  // A (attention output, FFN hidden) is read once: let it go first
            tma_load_2d_pair_hint(smem_u32(sA + stage * C::kABytes), &tmA, fb_even, kb * kBK, m0, a_policy);
          else
            tma_load_2d_pair(smem_u32(sA + stage * C::kABytes), &tmA, fb_even, kb * kBK, m0);
          if (it >= pre)  // weights: every M tile reads them, keep them in L2
            tma_load_2d_pair_hint(smem_u32(sB + stage * C::kBBytes), &tmB, fb_even, kb * kBK, n0, b_policy);
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // the even CTA drains every phase it armed (its own and the odd CTA's copies)
      if (rank == 0)
        for (int s = 0; s < kStages; ++s)
          if (armed & (1u << s)) mbar_drain(smem_u32(full + s), (armed_phase >> s) & 1u, limit_ns, err);
    }
  } else if (warp == 1) {
    pdl_wait();
    if (rank == 0) {
      // even CTA: the MMA issuer of the pair. The whole warp runs the issue loop (waits and
      // descriptor arithmetic warp-uniform); one elected lane issues each MMA and commit.
      constexpr uint32_t idesc = idesc_bf16_f32(kTileM, kTileN, 0, 0);
      const uint64_t a_desc = smem_desc_sw128(smem_u32(sA), 1024, 1024);  // stage 0; stages and K
      const uint64_t b_desc = smem_desc_sw128(smem_u32(sB), 1024, 1024);  // steps move the address
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += num_pairs) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(tempty + acc), acc_phase ^ 1u, wc))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kTileN);
        for (int kb = 0; kb < num_k; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(full + stage), phase, wc))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = desc_advance(a_desc, stage * C::kABytes), bd = desc_advance(b_desc, stage * C::kBBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_ss_pair_warp(d_tmem, desc_advance(ad, k * 32), desc_advance(bd, k * 32), idesc, (kb | k) != 0 ? 1u : 0u);
          mma_commit_pair_mc_warp(smem_u32(empty + stage), 0x3);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair_mc_warp(smem_u32(tfull + acc), 0x3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      mma_commit_pair_mc_warp(smem_u32(mma_done), 0x1);
      mbar_drain(smem_u32(mma_done), 0, limit_ns, err);
    }
  } else {
    pdl_wait();  // the epilogue writes (or adds into) buffers that earlier kernels use
    const int q = warp & 3;                    // TMEM lane quarter this warp may access
    constexpr int kChunks = kTileN / 32 / 2;   // 32-column chunks per warp (half the columns)
    const int half = (warp - 2) >> 2;  // which of the two warps on this lane quarter
    const uint32_t tempty_even = mapa_shared(smem_u32(tempty), 0);
    EpiStage stage{sEpi + (warp - 2) * 4096, 0};
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = pair; tile < num_tiles; tile += num_pairs) {
      const int m0 = (tile / num_n) * kTileM + (int)rank * 128, n0 = (tile % num_n) * kTileN;
      EpiPre<EK, kChunks> pre;  // requested while the main loop runs
      epi_prepare<EK, kChunks>(epi, lane, m0 + q * 32, n0, half, pre);
      if (!mbar_wait(smem_u32(tfull + acc), acc_phase, wc)) break;
      tc_fence_after();
      const int y0 = m0 + q * 32;
      const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kTileN);
      epi_warp_tile<EK, kChunks>(epi, &tmO, stage, lane, trow, y0, n0, half, pre);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(tempty_even + (uint32_t)(acc * sizeof(uint64_t)));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    stage.finish(lane);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the pair's MMAs are drained and both epilogues are done with TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

template <int TN>
cudaError_t set_pair_attrs() {
  cudaError_t e = cudaSuccess;
  auto set = [&](const void* f) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg<TN>::kSmemBytes);
  };
  set((const void*)gemm_tc2_kernel<TN, kEpiBias>);
  set((const void*)gemm_tc2_kernel<TN, kEpiGelu>);
  set((const void*)gemm_tc2_kernel<TN, kEpiResidual>);
  set((const void*)gemm_tc2_kernel<TN, kEpiQkvRope>);
  set((const void*)gemm_tc2_kernel<TN, kEpiPatch>);
  return e;
}

template <int TN, int EK>
cudaError_t launch_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmO, const EpiArgs& epi,
                        int M, int N, int K, int* err, uint64_t limit_ns, cudaStream_t s) {
  const int tiles = ((M + kTileM - 1) / kTileM) * ((N + TN - 1) / TN);
  const int max_pairs = gemm_tc2_max_pairs();
  const int pairs = tiles < max_pairs ? tiles : max_pairs;
  return launch_kernel(gemm_tc2_kernel<TN, EK>, dim3(2 * pairs), dim3(kThreads), PairCfg<TN>::kSmemBytes, s, tmA, tmB,
                       tmO, epi, M, N, K, err, limit_ns);
}

template <int TN>
cudaError_t launch_pair_kind(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmO,
                             const EpiArgs& epi, int M, int N, int K, int* err, uint64_t limit_ns, cudaStream_t s) {
  switch (epi.kind) {
    case kEpiBias: return launch_pair<TN, kEpiBias>(tmA, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    case kEpiGelu: return launch_pair<TN, kEpiGelu>(tmA, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    case kEpiResidual: return launch_pair<TN, kEpiResidual>(tmA, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    case kEpiQkvRope: return launch_pair<TN, kEpiQkvRope>(tmA, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    case kEpiPatch: return launch_pair<TN, kEpiPatch>(tmA, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t gemm_tc2_init_attributes() { return set_pair_attrs<256>(); }

// Cluster pairs that can be resident at once (the GPCs may not pair up every SM).
int gemm_tc2_max_pairs() {
  static int cached = 0;
  if (cached == 0) {
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = PairCfg<256>::kSmemBytes;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc2_kernel<256, kEpiBias>, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = num_sms() / 2;
    }
    cached = n < num_sms() / 2 ? n : num_sms() / 2;
  }
  return cached;
}

cudaError_t gemm_tc2_launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmO,
                            const EpiArgs& epi, int M, int N, int K, int* err, uint64_t limit_ns, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (N % 64 || K % kBK) return cudaErrorInvalidValue;
  return launch_pair_kind<256>(tmA, tmB, tmO, epi, M, N, K, err, limit_ns, s);
}

}  // namespace jepa
