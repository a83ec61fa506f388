// internal.h -- helpers the C-ABI translation units share (not part of the public header):
// the thread-local error text, the CUDA-call check, sizes and the weight synthesiser.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <string>

#include "jepa.h"

namespace jepa {

// Record a reason in the thread-local error text (jepa_error_text) and return `s`.
jepa_status fail(jepa_status s, const char* fmt, ...);

constexpr size_t kDefaultBudget = 8ull << 30;  // 8 GiB, the default arena ceiling of the pages

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Rotated dims per axis of the 3-D RoPE: d = 2 * ((head_dim / 3) / 2).
inline int rope_d(int head_dim) { return 2 * ((head_dim / 3) / 2); }

// Fill `n` values of the synthetic tensor `name` (synth/jepa_synth.h recipe) on all host cores.
void synth_parallel(uint64_t seed, const std::string& name, int bf16_matrices, size_t n, float* dst);

// Bits of a device error word: the low bits count bounded waits that gave up; kErrBadIds marks
// an index argument outside its range (the kernel used a safe substitute instead).
constexpr int kErrBadIds = 1 << 24;

}  // namespace jepa

#define CUDA_TRY(expr)                                                                               \
  do {                                                                                               \
    cudaError_t e_ = (expr);                                                                         \
    if (e_ != cudaSuccess)                                                                           \
      return ::jepa::fail(e_ == cudaErrorMemoryAllocation ? JEPA_E_OOM : JEPA_E_CUDA, "%s: %s (%s:%d)", \
                          #expr, cudaGetErrorString(e_), __FILE__, __LINE__);                         \
  } while (0)
