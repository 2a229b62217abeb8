// Shared device helpers for the libmars kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/mars.h"

#define MARS_DEV __device__ __forceinline__

namespace mars {

constexpr int kPageSize = 16;     // tokens per KV page (the only page size built)
constexpr int kNumSMs = 152;      // GB300: 2 dies x 76 SMs; used to size grids

MARS_DEV float bf16_to_f32(uint16_t x) { return __uint_as_float(uint32_t(x) << 16); }

MARS_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

MARS_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Unpack 8 bf16 held in a 16-byte vector into floats.
MARS_DEV void unpack8(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

}  // namespace mars
