// Producer step of the indexer inputs: per-group absmax quantisation to e4m3.
//
// The indexer runs in FP8 ("DeepSeek V3.2: How Far Can Open Models Go If You
// Actually Try?", §3.1; FP8 e4m3 with one fp32 scale per query token and per
// key row).  For each group of G consecutive values (a token's 64 x 128
// indexer query, or a key row of 128):
//   scale = amax / 448   (1 when amax = 0),   code = e4m3(x / scale)
// with the division in IEEE fp32 and the conversion rounding to nearest even
// and saturating at +-448 (cvt.rn.satfinite).  The codes and scales can be
// written straight into a cache at a row offset (append).
//
// Groups of at most 1024 values take one warp each (8 per 256-thread CTA) and
// stay in registers between the max and the conversion; larger groups (up to
// 16384) take one warp each in two streaming passes.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace dsa {
namespace quant {

constexpr int kThreads = 256;
constexpr int kWarpGroupMax = 32 * 32;     // largest group handled by one warp
constexpr int kMaxGroup = 16384;

// Four consecutive inputs as fp32 (bf16 widens exactly).
__device__ __forceinline__ float4 load4(const void* x, int64_t i, bool bf16) {
  if (bf16) {
    const uint2 r = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(x) + i));
    return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xFFFF0000u),
                       __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xFFFF0000u));
  }
  return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(x) + i));
}

// e4m3 codes of (a, b): low byte a, high byte b.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float a, float b) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(b), "f"(a));
  return d;
}

__device__ __forceinline__ uint32_t encode4(float4 v, float scale) {
  const uint32_t lo = cvt_e4m3x2(__fdiv_rn(v.x, scale), __fdiv_rn(v.y, scale));
  const uint32_t hi = cvt_e4m3x2(__fdiv_rn(v.z, scale), __fdiv_rn(v.w, scale));
  return lo | (hi << 16);
}

__device__ __forceinline__ float absmax4(float4 v) {
  return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

// One warp per group (group_elems <= 1024, multiple of 4).
__global__ void __launch_bounds__(kThreads) quantize_warp_kernel(const void* __restrict__ x, bool bf16,
                                                                  int64_t groups, int group_elems,
                                                                  uint8_t* __restrict__ codes,
                                                                  float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
  if (g >= groups) return;
  const int nvec = group_elems / 4;   // float4 vectors in the group
  const int64_t base = g * group_elems;
  float4 v[kWarpGroupMax / 128];
  float amax = 0.f;
#pragma unroll
  for (int r = 0; r < kWarpGroupMax / 128; ++r) {
    const int q = lane + 32 * r;
    v[r] = q < nvec ? load4(x, base + 4 * q, bf16) : make_float4(0.f, 0.f, 0.f, 0.f);
    amax = fmaxf(amax, absmax4(v[r]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
#pragma unroll
  for (int r = 0; r < kWarpGroupMax / 128; ++r) {
    const int q = lane + 32 * r;
    if (q < nvec) reinterpret_cast<uint32_t*>(codes + base)[q] = encode4(v[r], scale);
  }
  if (lane == 0) scales[g] = scale;
}

// Groups larger than a warp's register share (up to 16384 values): one warp
// per group in two streaming passes, the absmax pass from HBM and the
// encoding pass re-reading the group (16 KB at most, still in L2), with eight
// loads in flight per lane in each pass.
__global__ void __launch_bounds__(kThreads) quantize_stream_kernel(const void* __restrict__ x, bool bf16,
                                                                    int64_t groups, int group_elems,
                                                                    uint8_t* __restrict__ codes,
                                                                    float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
  if (g >= groups) return;
  const int nvec = group_elems / 4;
  const int64_t base = g * group_elems;
  float amax = 0.f;
  for (int q0 = 0; q0 < nvec; q0 += 32 * 8) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = q0 + lane + 32 * u;
      v[u] = q < nvec ? load4(x, base + 4 * q, bf16) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) amax = fmaxf(amax, absmax4(v[u]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  for (int q0 = 0; q0 < nvec; q0 += 32 * 8) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = q0 + lane + 32 * u;
      v[u] = q < nvec ? load4(x, base + 4 * q, bf16) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = q0 + lane + 32 * u;
      if (q < nvec) reinterpret_cast<uint32_t*>(codes + base)[q] = encode4(v[u], scale);
    }
  }
  if (lane == 0) scales[g] = scale;
}

}  // namespace quant
}  // namespace dsa
