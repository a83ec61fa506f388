/* Exported wrappers around jepa_synth.h for the Python tests and the bench
 * (ctypes). Build: gcc -O2 -ffp-contract=off -shared -fPIC. */
#include "jepa_synth.h"

uint64_t jsynth_api_splitmix_at(uint64_t s, uint64_t i) { return jsynth_splitmix_at(s, i); }
uint64_t jsynth_api_fnv1a64(const char* name) { return jsynth_fnv1a64(name); }
double jsynth_api_ln(double x) { return jsynth_ln(x); }
double jsynth_api_cos2pi(double v) { return jsynth_cos2pi(v); }
double jsynth_api_normal(uint64_t seed, const char* name, uint64_t i) {
  return jsynth_normal(jsynth_stream(seed, name), i);
}
void jsynth_api_fill(uint64_t seed, const char* name, int kind, double a, double b, int round_bf16,
                     uint64_t first, uint64_t n, float* dst) {
  jsynth_fill(seed, name, kind, a, b, round_bf16, first, (size_t)n, dst);
}
void jsynth_api_param(uint64_t seed, const char* name, int bf16_matrices, uint64_t n, float* dst) {
  jsynth_param(seed, name, bf16_matrices, (size_t)n, dst);
}
void jsynth_api_pixels(uint64_t seed, uint64_t first, uint64_t n, float* dst) {
  jsynth_pixels(seed, first, (size_t)n, dst);
}
float jsynth_api_round_bf16(float f) { return jsynth_round_bf16(f); }
