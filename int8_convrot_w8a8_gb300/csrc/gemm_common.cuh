// Output descriptors shared by the GEMM kernels: one entry per linear that
// consumes the same packed activation (up to 8, e.g. q/k/v or gate/up).
#pragma once

#include <cstdint>

namespace convrot {

constexpr int kMaxLinears = 8;

struct GemmOut {
  const int8_t* qw;      // int8 [n, K]
  const uint16_t* qw16;  // fp16 [n, K] (tensor-core path) or nullptr
  const float* sw;       // fp32 [n]
  const float* bias;     // fp32 [n] or nullptr
  void* y;               // bf16 (or int32 for raw accumulators) [M, ldy]
  long long ldy;
  int n;
  int tile_begin;        // first N tile of this linear in the concatenated tile space
};

struct GemmOutputs {
  int count;
  GemmOut o[kMaxLinears];
};

}  // namespace convrot
