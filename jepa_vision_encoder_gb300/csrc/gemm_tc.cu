// gemm_tc.cu -- persistent tcgen05 GEMM for sm_103a: out = epilogue(A[M,K] B[N,K]^T), bf16
// operands, fp32 accumulation in tensor memory. Every linear layer of the encoder runs here
// ("Architecture", The shared ViT graph: patch embed, fused qkv, out-projection, FFN).
//
// Warp roles (320 threads, one CTA per SM, grid = min(tiles, SMs), tiles strided over CTAs and
// numbered N-fastest, so the CTAs working at the same time share rows of A and sweep the weights):
//   warp 0      TMA producer: A tile 128x64 and B tile BNx64 per stage (128-byte swizzle); the
//               first tile's weight stages go out before the wait on the previous kernel
//   warp 1      MMA issuer: 4 x tcgen05.mma (M=128, N=BN, K=16) per stage into one of two
//               TMEM accumulators (2 x BN columns), so the epilogue of tile i overlaps the
//               main loop of tile i+1
//   warps 2..9  epilogue: two warps per TMEM lane quarter, each taking half of the tile's columns
//               (for QKV, alternate 32-column chunks, so a warp meets one half of every head and
//               keeps that half's RoPE (cos, sin) row in registers; bias and RoPE values are
//               requested before the accumulator is ready), 32 columns at a time (the
//               next tcgen05.ld in flight while one chunk is processed), then
//               the fused bias / GELU / RoPE of epilogue.cuh; each 32-row x 64-byte piece goes
//               through a per-warp pair of swizzled shared-memory buffers to a TMA store (bf16
//               outputs) or a TMA fp32 add into the residual stream. The patch embedding (rows
//               remapped per item) stores from registers.
// Every mbarrier wait is bounded (ptx.cuh); on the way out the producer drains its loads and the
// MMA thread waits for its MMAs before TMEM is freed.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace jepa {

constexpr int kBM = 128;
constexpr int kBK = 64;  // one 128-byte swizzle atom of bf16 along K
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;

template <int BN>
struct GemmCfg {
  static constexpr int kStages = (BN == 256) ? 4 : (BN == 128 ? 6 : 8);
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr int kEpiBytes = kEpiWarps * 4096;  // two 2 KB staging buffers per epilogue warp
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kEpiBytes + kBarBytes;
};

template <int BN, int EK>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmO, EpiArgs epi, int M, int N, int K, int* err,
                   uint64_t limit_ns) {
  using C = GemmCfg<BN>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * C::kABytes;
  uint8_t* sEpi = smem + S * C::kStageBytes;  // kEpiWarps x 4 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + C::kEpiBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = bars + 2 * S + 2;
  uint64_t* mma_done = bars + 2 * S + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_m = (M + kBM - 1) / kBM, num_n = N / BN, num_k = K / kBK;
  const int num_tiles = num_m * num_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(tfull + a), 1);
      mbar_init(smem_u32(tempty + a), kEpiWarps);
    }
    mbar_init(smem_u32(mma_done), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (EK != kEpiPatch) prefetch_tmap(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{abort_flag, err, limit_ns};
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t a_policy = l2_policy_evict_first(), b_policy = l2_policy_evict_last();
      // The weights are written by no kernel of the sequence: the first tile's first S stages of
      // B are requested (and their stages armed) before waiting for the previous kernel, whose
      // tail this CTA may overlap; A and the residual stream come from earlier kernels.
      // The loop's first S waits for a free stage pass at once (fresh barriers), so every stage
      // armed here also gets its A copy.
      const int pre = blockIdx.x < num_tiles ? (num_k < S ? num_k : S) : 0;
      uint32_t phase = 0, armed = 0, armed_phase = 0;
      for (int kb = 0; kb < pre; ++kb) {
        const uint32_t fb = smem_u32(full + kb);
        mbar_arrive_expect_tx(fb, C::kStageBytes);
        tma_load_2d_hint(smem_u32(sB + kb * C::kBBytes), &tmB, fb, kb * kBK, (blockIdx.x % num_n) * BN, b_policy);
        armed |= 1u << kb;
      }
      pdl_wait();
      int stage = 0, it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int m0 = (tile / num_n) * kBM, n0 = (tile % num_n) * BN;
        for (int kb = 0; kb < num_k; ++kb, ++it) {
          if (!mbar_wait(smem_u32(empty + stage), phase ^ 1u, wc)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(full + stage);
          if (it >= pre) mbar_arrive_expect_tx(fb, C::kStageBytes);
          if (EK == kEpiResidual)  // A (attention output, FFN hidden) is read once: let it go first
            tma_load_2d_hint(smem_u32(sA + stage * C::kABytes), &tmA, fb, kb * kBK, m0, a_policy);
          else
            tma_load_2d(smem_u32(sA + stage * C::kABytes), &tmA, fb, kb * kBK, m0);
          if (it >= pre)  // weights: every M tile reads them, keep them in L2
            tma_load_2d_hint(smem_u32(sB + stage * C::kBBytes), &tmB, fb, kb * kBK, n0, b_policy);
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < S; ++s)
        if (armed & (1u << s)) mbar_drain(smem_u32(full + s), (armed_phase >> s) & 1u, limit_ns, err);
    }
  } else if (warp == 1) {
    pdl_wait();
    // the whole warp runs the issue loop (waits and descriptor arithmetic warp-uniform); one
    // elected lane issues each MMA and commit
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN, 0, 0);
    const uint64_t a_desc = smem_desc_sw128(smem_u32(sA), 1024, 1024);  // stage 0; stages and K
    const uint64_t b_desc = smem_desc_sw128(smem_u32(sB), 1024, 1024);  // steps move the address
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(tempty + acc), acc_phase ^ 1u, wc))) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      for (int kb = 0; kb < num_k; ++kb) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(full + stage), phase, wc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = desc_advance(a_desc, stage * C::kABytes), bd = desc_advance(b_desc, stage * C::kBBytes);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_ss_warp(d_tmem, desc_advance(ad, k * 32), desc_advance(bd, k * 32), idesc, (kb | k) != 0 ? 1u : 0u);
        mma_commit_warp(smem_u32(empty + stage));
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      mma_commit_warp(smem_u32(tfull + acc));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    mma_commit_warp(smem_u32(mma_done));
    mbar_drain(smem_u32(mma_done), 0, limit_ns, err);
  } else {
    pdl_wait();  // the epilogue writes (or adds into) buffers that earlier kernels use
    const int q = warp & 3;                        // TMEM lane quarter this warp may access
    constexpr int kChunks = BN / 32 / 2;           // 32-column chunks per warp (half the tile)
    const int half = (warp - 2) >> 2;              // which of the two warps on this lane quarter
    EpiStage stage{sEpi + (warp - 2) * 4096, 0};
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const int m0 = (tile / num_n) * kBM, n0 = (tile % num_n) * BN;
      EpiPre<EK, kChunks> pre;  // requested while the main loop runs
      epi_prepare<EK, kChunks>(epi, lane, m0 + q * 32, n0, half, pre);
      if (!mbar_wait(smem_u32(tfull + acc), acc_phase, wc)) break;
      tc_fence_after();
      const int y0 = m0 + q * 32;
      const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      epi_warp_tile<EK, kChunks>(epi, &tmO, stage, lane, trow, y0, n0, half, pre);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(tempty + acc));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    stage.finish(lane);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// Tile choice by a small cost model: waves of tiles times the per-SM work of one tile divided
// by the fraction of the tensor peak that tile shape sustains (measured: 1-SM 128x256 0.62,
// 128x128 0.48, 128x64 0.29 of peak with TMA-fed operands; the 2-SM 256x256 pair form 0.75).
// Returns 64, 128, 256, or kPairTile for the 2-SM kernel.
int gemm_tc_pick_bn(int M, int N) {
  const int sms = num_sms();
  const int num_m = (M + kBM - 1) / kBM, num_m2 = (M + 2 * kBM - 1) / (2 * kBM);
  int best = 0;
  double best_cost = 1e30;
  const struct { int bn; double eff; } one[] = {{256, 0.62}, {128, 0.48}, {64, 0.29}};
  for (const auto& c : one) {
    if (N % c.bn) continue;
    const long long tiles = (long long)num_m * (N / c.bn);
    const double cost = (double)((tiles + sms - 1) / sms) * c.bn / c.eff;
    if (cost < best_cost) best_cost = cost, best = c.bn;
  }
  // a last column tile that reaches past N computes zeros there (not stored): taken only while that
  // waste stays under a tenth of the columns computed
  const int n_pad = ((N + 255) / 256) * 256;
  if (N % 64 == 0 && 10 * (n_pad - N) < n_pad && sms >= 2) {
    const long long pair_tiles = (long long)num_m2 * (n_pad / 256);
    const int pairs = gemm_tc2_max_pairs();
    const double cost = (double)((pair_tiles + pairs - 1) / pairs) * 256 / 0.75;
    if (cost < best_cost) best_cost = cost, best = kPairTile;
  }
  return best ? best : 64;
}

int gemm_tc_b_box(int bn) { return bn == kPairTile ? 128 : bn; }

template <int BN, int EK>
static cudaError_t launch_bn(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmO,
                             const EpiArgs& epi, int M, int N, int K, int* err, uint64_t limit_ns, cudaStream_t s) {
  using C = GemmCfg<BN>;
  const int tiles = ((M + kBM - 1) / kBM) * (N / BN);
  const int grid = tiles < num_sms() ? tiles : num_sms();
  return launch_kernel(gemm_tc_kernel<BN, EK>, dim3(grid), dim3(kThreads), C::kSmemBytes, s, tmA, tmB, tmO, epi, M, N,
                       K, err, limit_ns);
}

template <int BN>
static cudaError_t launch_kind(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmO,
                               const EpiArgs& epi, int M, int N, int K, int* err, uint64_t limit_ns, cudaStream_t s) {
  switch (epi.kind) {
    case kEpiBias: return launch_bn<BN, kEpiBias>(tmA, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    case kEpiGelu: return launch_bn<BN, kEpiGelu>(tmA, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    case kEpiResidual: return launch_bn<BN, kEpiResidual>(tmA, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    case kEpiQkvRope: return launch_bn<BN, kEpiQkvRope>(tmA, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    case kEpiPatch: return launch_bn<BN, kEpiPatch>(tmA, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int BN>
static cudaError_t set_smem_attr() {
  cudaError_t e = cudaSuccess;
  auto set = [&](const void* f) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, GemmCfg<BN>::kSmemBytes);
  };
  set((const void*)gemm_tc_kernel<BN, kEpiBias>);
  set((const void*)gemm_tc_kernel<BN, kEpiGelu>);
  set((const void*)gemm_tc_kernel<BN, kEpiResidual>);
  set((const void*)gemm_tc_kernel<BN, kEpiQkvRope>);
  set((const void*)gemm_tc_kernel<BN, kEpiPatch>);
  return e;
}

cudaError_t gemm_tc2_init_attributes();

cudaError_t gemm_tc_init_attributes() {
  cudaError_t e = gemm_tc2_init_attributes();
  if (e == cudaSuccess) e = set_smem_attr<256>();
  if (e == cudaSuccess) e = set_smem_attr<128>();
  if (e == cudaSuccess) e = set_smem_attr<64>();
  return e;
}

cudaError_t gemm_tc_launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmO, int BN,
                           const EpiArgs& epi, int M, int N, int K, int* err, uint64_t limit_ns, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (BN == kPairTile) return gemm_tc2_launch(tmA, tmB, tmO, epi, M, N, K, err, limit_ns, s);
  switch (BN) {
    case 256: return launch_kind<256>(tmA, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    case 128: return launch_kind<128>(tmA, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    case 64: return launch_kind<64>(tmA, tmB, tmO, epi, M, N, K, err, limit_ns, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace jepa
