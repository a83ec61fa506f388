// kernels.h -- host-side launchers of the CUDA kernels (internal to libjepa_gb300.so).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "epilogue.cuh"

#include <utility>

namespace jepa {

// Launch mode of the calling thread: while set (the encoder's launch sequence), kernels go out as
// programmatic dependent launches, so each one's set-up overlaps the end of the previous kernel.
bool& pdl_launches();

// Launches `kernel` on `s`, programmatic when pdl_launches() is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pdl_launches()) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Encodes a 2-D bf16 tensor map (row-major [rows, cols], 128-byte swizzle, box = box_rows x 64).
// Returns false if the driver refuses the map.
bool make_tmap_2d_bf16(CUtensorMap* tm, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);
// GEMM output map: row-major [rows, cols] of bf16 (elem_bytes 2) or fp32 (4), box 32 rows x 64
// bytes with the 64-byte swizzle (the epilogue's staging layout).
bool make_tmap_2d_out(CUtensorMap* tm, const void* ptr, uint64_t rows, uint64_t cols, int elem_bytes);
// 3-D map of a [B][N][cols] bf16 array with box box_cols x box_rows x 1 (attention Q/K/V tiles of
// one head): box_cols 64 with the 128-byte swizzle, or 32 with the 64-byte swizzle.
bool make_tmap_3d_bf16(CUtensorMap* tm, const void* ptr, uint64_t B, uint64_t N, uint64_t cols, uint32_t box_rows,
                       uint32_t box_cols = 64);

int num_sms();
// Sets the dynamic shared-memory limits of the tcgen05 kernels (once per process; call before
// any stream capture).
cudaError_t tc_kernels_init();
uint64_t default_wait_limit_ns();

// tcgen05 GEMM: out = epilogue(A[M,K] * B[N,K]^T), bf16 operands. tmA box 128x64, tmB box
// gemm_tc_b_box(BN) x 64 where BN = gemm_tc_pick_bn(M, N); BN == kPairTile selects the 2-SM
// (cluster pair) kernel with 256 x 256 tiles. tmO = make_tmap_2d_out over epi.out (bf16 for
// BIAS / GELU / QKV_ROPE, fp32 for RESIDUAL; unused for PATCH, which stores from registers).
// B holds weights: in a programmatic launch sequence its first stages are requested before the
// wait on the previous kernel, so no kernel of the sequence may write it.
constexpr int kPairTile = 512;
int gemm_tc_pick_bn(int M, int N);
int gemm_tc_b_box(int bn);
int gemm_tc2_max_pairs();
cudaError_t gemm_tc2_launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmO,
                            const EpiArgs& epi, int M, int N, int K, int* err, uint64_t limit_ns, cudaStream_t s);
cudaError_t gemm_tc_launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmO, int BN,
                           const EpiArgs& epi, int M, int N, int K, int* err, uint64_t limit_ns, cudaStream_t s);

// fp32 SIMT GEMM with the same epilogues. In a programmatic launch sequence its first B (weight)
// step is read before the wait on the previous kernel, like the tcgen05 GEMMs' first weight stages.
cudaError_t gemm_simt_launch(const float* A, const float* Bw, const EpiArgs& epi, int M, int N, int K,
                             cudaStream_t s);

// tcgen05 flash attention over qkv [B][N][3*H*64] bf16 (3-D tensor map, box 64 x 128).
struct AttnParams {
  int B, N, H, head_dim;
  int attn_mode, prefix, frame_tokens;
  void* out;                  // [B*N, H*head_dim]
  const void* qkv = nullptr;  // [B*N, 3*H*head_dim]: read directly by the block-causal prefix rows
};
cudaError_t attention_tc_launch(const CUtensorMap& tmQKV, const AttnParams& p, int* err, uint64_t limit_ns,
                                cudaStream_t s);
// fp32 attention (SIMT, online softmax).
cudaError_t attention_simt_launch(const float* qkv, const AttnParams& p, cudaStream_t s);

// Element-wise / row kernels.
cudaError_t patchify_launch(const float* pix, int B, int T, int C, int H, int W, int t, int P, int layout,
                            bool out_bf16, void* out, cudaStream_t s);
cudaError_t layernorm_launch(const float* x, int M, int D, const float* g, const float* b, float eps,
                             bool out_bf16, void* y, cudaStream_t s);
cudaError_t rope_table_launch(int gt, int gh, int gw, int head_dim, float theta, int interpolate, int ref_grid,
                              float2* table, cudaStream_t s);
// The same entries factored per axis: [gt + gh + gw][d/2] (t rows, then h, then w).
cudaError_t rope_axes_launch(int gt, int gh, int gw, int head_dim, float theta, int interpolate, int ref_grid,
                             float2* axes, cudaStream_t s);
// X rows b*N + r for r < prefix: cls (+ pos[r]) (+ vec).
cudaError_t prefix_rows_launch(float* X, int B, int N, int D, const float* cls, const float* pos,
                               const float* vec, cudaStream_t s);
// Fixed sin-cos position table [gt*gh*gw, D] (kind 0: 2-D with gt == 1, kind 1: 3-D) and its
// resizing (mode 0 trilinear, mode 1 bicubic per frame) to another grid.
bool sincos_widths(int kind, int D, int uniform_power, int* d0, int* d1, int* d2);
cudaError_t sincos_table_launch(int kind, int gt, int gh, int gw, int D, int w_first, int uniform_power, float* out,
                                cudaStream_t s);
cudaError_t pos_resize_launch(const float* src, int st, int sh, int sw, int D, int mode, float* dst, int dt, int dh,
                              int dw, cudaStream_t s);
// A kernel whose wait can never complete (failure-path check of the bounded waits).
cudaError_t wait_timeout_probe_launch(int* err, uint64_t limit_ns, cudaStream_t s);

}  // namespace jepa
