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
// Within a group every value is divided by the same scale, so the correctly
// rounded quotient comes from one reciprocal and a correction step per value
// (CommonDivisor) instead of a full division.
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

// Correctly rounded x / s for many x and one s, by Markstein's correction
// step (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with y = RN(1/s)
// and q = RN(x y) within an ulp of x/s, the remainder r = x - q s is exact
// in one FMA and RN(q + r y) = RN(x / s).  r = 0 means q is already the
// exact quotient (this also keeps the sign of a zero x).  Valid away from
// overflow and from subnormal quotients; every quotient here is at most 448
// in magnitude, and quotients small enough to be subnormal encode as (signed)
// zero in e4m3 either way.
struct CommonDivisor {
  float s, y;
  __device__ __forceinline__ explicit CommonDivisor(float s_) : s(s_) {
    asm("rcp.rn.f32 %0, %1;" : "=f"(y) : "f"(s_));
  }
  __device__ __forceinline__ float div(float x) const {
    const float q = __fmul_rn(x, y);
    const float r = __fmaf_rn(-q, s, x);
    return r == 0.f ? q : __fmaf_rn(r, y, q);
  }
};

__device__ __forceinline__ uint32_t encode4(float4 v, const CommonDivisor& d) {
  const uint32_t lo = cvt_e4m3x2(d.div(v.x), d.div(v.y));
  const uint32_t hi = cvt_e4m3x2(d.div(v.z), d.div(v.w));
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
// of 256 threads per group.  Every thread loads its vectors t, t + 256, ...
// at once, so x is read once with all loads in flight; the maximum is
// reduced over the warps through shared memory, then every thread encodes
// from registers.  Vector kinds: fp32 in 16 bytes (4 values), bf16 in 16
// bytes (8 values, group_elems % 8 == 0) or bf16 in 8 bytes (4 values).
enum VecKind { kF32x4 = 0, kBf16x8 = 1, kBf16x4 = 2 };

template <int kKind>
struct CtaShape {
  static constexpr int kThreads = 256;
  static constexpr int kPerVec = kKind == kBf16x8 ? 8 : 4;          // values per vector
  static constexpr int kVec = kMaxGroup / kPerVec / kThreads;        // vectors per thread (at most)
  using Raw = typename std::conditional<kKind == kBf16x4, uint2, uint4>::type;
};

template <int kKind>
__global__ void __launch_bounds__(256, kKind == kF32x4 ? 2 : 3) quantize_cta_kernel(
    const void* __restrict__ x, int group_elems, uint8_t* __restrict__ codes, float* __restrict__ scales) {
  using Sh = CtaShape<kKind>;
  using Raw = typename Sh::Raw;
  __shared__ float warp_max[Sh::kThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t g = blockIdx.x;
  const int nvec = group_elems / Sh::kPerVec;
  const int64_t base = g * group_elems;
  const Raw* __restrict__ src = kKind == kF32x4
      ? reinterpret_cast<const Raw*>(static_cast<const float*>(x) + base)
      : reinterpret_cast<const Raw*>(static_cast<const __nv_bfloat16*>(x) + base);
  Raw raw[Sh::kVec];
#pragma unroll
  for (int r = 0; r < Sh::kVec; ++r) {
    const int q = tid + Sh::kThreads * r;
    if (q < nvec) raw[r] = __ldg(src + q);
    else memset(&raw[r], 0, sizeof(Raw));
  }
  // the first (and for 8-value vectors the second) four values as fp32;
  // bf16 widens exactly
  auto lo4 = [](const Raw& u) -> float4 {
    if constexpr (kKind == kF32x4)
      return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
    else
      return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                         __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
  };
  auto hi4 = [](const Raw& u) -> float4 {
    if constexpr (kKind == kBf16x8)
      return make_float4(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xFFFF0000u),
                         __uint_as_float(u.w << 16), __uint_as_float(u.w & 0xFFFF0000u));
    else
      return make_float4(0.f, 0.f, 0.f, 0.f);
  };
  float amax = 0.f;
#pragma unroll
  for (int r = 0; r < Sh::kVec; ++r) {   // padding is 0
    amax = fmaxf(amax, absmax4(lo4(raw[r])));
    if constexpr (kKind == kBf16x8) amax = fmaxf(amax, absmax4(hi4(raw[r])));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) warp_max[warp] = amax;
  __syncthreads();
  amax = warp_max[0];
#pragma unroll
  for (int w = 1; w < Sh::kThreads / 32; ++w) amax = fmaxf(amax, warp_max[w]);
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  const CommonDivisor dv(scale);
#pragma unroll
  for (int r = 0; r < Sh::kVec; ++r) {
    const int q = tid + Sh::kThreads * r;
    if (q < nvec) {
      if constexpr (kKind == kBf16x8)
        reinterpret_cast<uint2*>(codes + base)[q] = make_uint2(encode4(lo4(raw[r]), dv), encode4(hi4(raw[r]), dv));
      else
        reinterpret_cast<uint32_t*>(codes + base)[q] = encode4(lo4(raw[r]), dv);
    }
  }
  if (tid == 0) scales[g] = scale;
}

}  // namespace quant
}  // namespace dsa
