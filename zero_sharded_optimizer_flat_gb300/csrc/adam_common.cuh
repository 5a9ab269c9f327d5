// Element-wise building blocks shared by the AdamW step and its rescale: the tile geometry
// (2048-element tiles, 4-element vector accesses, 256 threads), 128-bit loads and stores, the
// fp64 power by square-and-multiply and the bf16 round-out.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace zopt {
namespace adam {

constexpr int kThreads = 256;
constexpr int kGroup = 4;                        // elements per vector access
constexpr int kTile = kThreads * kGroup * 2;     // 2048 elements per tile
constexpr int kBlocksPerSm = 4;

__device__ __forceinline__ double pow_sq_mul(double base, long long e) {
  double r = 1.0;
  while (e > 0) {
    if (e & 1) r = __dmul_rn(r, base);
    base = __dmul_rn(base, base);
    e >>= 1;
  }
  return r;
}

struct Vec4 { float x[4]; };

__device__ __forceinline__ Vec4 ld4(const float* p) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  return Vec4{{a.x, a.y, a.z, a.w}};
}
__device__ __forceinline__ void st4(float* p, const Vec4& v) {
  *reinterpret_cast<float4*>(p) = make_float4(v.x[0], v.x[1], v.x[2], v.x[3]);
}
__device__ __forceinline__ Vec4 ldg4(const float* p) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  return Vec4{{a.x, a.y, a.z, a.w}};
}
__device__ __forceinline__ Vec4 ldg4(const __nv_bfloat16* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  return Vec4{{__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
               __uint_as_float(u.y & 0xFFFF0000u)}};
}
__device__ __forceinline__ float ldg1(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ldg1(const __nv_bfloat16* p) {
  return __uint_as_float(static_cast<unsigned int>(__ldg(reinterpret_cast<const unsigned short*>(p))) << 16);
}

__device__ __forceinline__ unsigned short bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

}  // namespace adam
}  // namespace zopt
