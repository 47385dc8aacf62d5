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
// 16384, e.g. a token's 8192-value query) take one CTA each: every
// thread issues all of its loads at once, the group's maximum is a block
// reduction, and the values are encoded from registers (one read of x).
#pragma once

#include <cstdint>
#include <cstring>
#include <type_traits>
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

// Groups larger than a warp's register share (up to 16384 values): one CTA
// per group, 256 threads for bf16 input and 512 for fp32, so that every
// thread holds at most 16 bf16 or 8 fp32 vectors of 4 values (32 registers
// of raw input words).  Thread t holds the vectors t, t + threads, ... so all
// of its loads are in flight together and x is read once; the maximum is
// reduced over the warps through shared memory, then every thread encodes
// its vectors from registers.
template <bool kBf16>
struct CtaShape {
  static constexpr int kThreads = kBf16 ? 256 : 512;
  static constexpr int kVec = kMaxGroup / 4 / kThreads;
  using Raw = typename std::conditional<kBf16, uint2, uint4>::type;
};

template <bool kBf16>
__global__ void __launch_bounds__(CtaShape<kBf16>::kThreads, kBf16 ? 4 : 2) quantize_cta_kernel(
    const void* __restrict__ x, int group_elems, uint8_t* __restrict__ codes, float* __restrict__ scales) {
  using Sh = CtaShape<kBf16>;
  using Raw = typename Sh::Raw;
  __shared__ float warp_max[Sh::kThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t g = blockIdx.x;
  const int nvec = group_elems / 4;
  const int64_t base = g * group_elems;
  const Raw* __restrict__ src = kBf16
      ? reinterpret_cast<const Raw*>(static_cast<const __nv_bfloat16*>(x) + base)
      : reinterpret_cast<const Raw*>(static_cast<const float*>(x) + base);
  Raw raw[Sh::kVec];
#pragma unroll
  for (int r = 0; r < Sh::kVec; ++r) {
    const int q = tid + Sh::kThreads * r;
    if (q < nvec) raw[r] = __ldg(src + q);
    else memset(&raw[r], 0, sizeof(Raw));
  }
  auto widen = [](const Raw& u) -> float4 {
    if constexpr (kBf16)
      return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                         __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
    else
      return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
  };
  float amax = 0.f;
#pragma unroll
  for (int r = 0; r < Sh::kVec; ++r) amax = fmaxf(amax, absmax4(widen(raw[r])));   // padding is 0
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) warp_max[warp] = amax;
  __syncthreads();
  amax = warp_max[0];
#pragma unroll
  for (int w = 1; w < Sh::kThreads / 32; ++w) amax = fmaxf(amax, warp_max[w]);
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
#pragma unroll
  for (int r = 0; r < Sh::kVec; ++r) {
    const int q = tid + Sh::kThreads * r;
    if (q < nvec) reinterpret_cast<uint32_t*>(codes + base)[q] = encode4(widen(raw[r]), scale);
  }
  if (tid == 0) scales[g] = scale;
}

}  // namespace quant
}  // namespace dsa
