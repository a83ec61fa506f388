// internal.h -- helpers the C-ABI translation units share (not part of the public header):
// the thread-local error text, the CUDA-call check, sizes and the weight synthesiser.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <string>
#include <utility>
#include <vector>

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

// ---- GGUF files (gguf.cpp)
struct GgufValue {
  uint32_t type = 0;                   // GGUF value type
  uint64_t u = 0;                      // integer and bool values
  int64_t i = 0;
  double f = 0.0;                      // float values (and integers, converted)
  std::string s;                       // string values
  uint32_t array_type = 0;             // arrays: element type, length, integer elements
  uint64_t array_len = 0;
  std::vector<int64_t> ints;
};
struct GgufTensor {
  std::string name;
  std::vector<uint64_t> dims;          // ggml order: dims[0] is the innermost (PyTorch's last)
  uint32_t type = 0;                   // ggml type (0 f32, 1 f16, 30 bf16, quantized types)
  uint64_t offset = 0;                 // absolute file offset of the data
  uint64_t n = 0, bytes = 0;           // elements, bytes
};
struct GgufFile {
  std::string path;
  uint64_t file_size = 0, data_start = 0;
  uint32_t version = 0, alignment = 32;
  std::vector<std::pair<std::string, GgufValue>> kvs;
  std::vector<GgufTensor> tensors;
  const GgufValue* get(const std::string& key) const;
  const GgufTensor* find(const std::string& name) const;
};
// Parse the header, keys and tensor infos, and check every tensor's bytes lie inside the file.
jepa_status gguf_open(const char* path, GgufFile* g);
// Read tensor t (f32, f16 or bf16) as floats into dst[t.n]; other types -> JEPA_E_UNSUPPORTED.
jepa_status gguf_read_f32(const GgufFile& g, const GgufTensor& t, float* dst);
const char* gguf_type_name(uint32_t type);

}  // namespace jepa

#define CUDA_TRY(expr)                                                                               \
  do {                                                                                               \
    cudaError_t e_ = (expr);                                                                         \
    if (e_ != cudaSuccess)                                                                           \
      return ::jepa::fail(e_ == cudaErrorMemoryAllocation ? JEPA_E_OOM : JEPA_E_CUDA, "%s: %s (%s:%d)", \
                          #expr, cudaGetErrorString(e_), __FILE__, __LINE__);                         \
  } while (0)
