// Device-side pieces of the norm / clip reduction, shared by the kernels that produce a
// sum of squares (the norm pass and the gradient-accumulation pass).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

#include "zopt.h"

namespace zopt {

constexpr int kNormThreads = 256;
constexpr int kNormBlocksPerSm = 8;
constexpr int64_t kNormMaxBlocks = 4096;

// Workspace header: the arrival counter, padded to 256 bytes, then one fp64 partial per block.
struct NormWorkspace {
  unsigned int arrive;
  unsigned int reserved[63];
  double partials[1];  // [grid] in practice
};
static_assert(offsetof(NormWorkspace, partials) == 256, "workspace header is 256 bytes");

size_t norm_grid_blocks(int64_t n);
// Blocks one launch over n elements uses on the current device (<= norm_grid_blocks(n)).
int norm_launch_blocks(int64_t n, zopt_dtype dtype);
zopt_status check_norm_args(const char* fn, const void* grad, zopt_dtype dtype, int64_t n, float max_norm,
                            const zopt_clip_stats* stats);

// Stats from a sum of squares, exactly as the pages state the contract (see norm.cu).
__device__ __forceinline__ void write_clip_stats(zopt_clip_stats* out, double ss, float max_norm) {
  const double norm64 = (ss >= 0.0) ? __dsqrt_rn(ss) : __longlong_as_double(0x7FF8000000000000LL);
  const float norm = __double2float_rn(norm64);
  const bool found_inf = !isfinite(norm);
  float coef = 0.0f;
  if (!found_inf) {
    coef = __fdiv_rn(max_norm, __fadd_rn(norm, 1e-6f));
    if (!(coef < 1.0f)) coef = 1.0f;
  }
  out->sumsq = ss;
  out->norm = norm;
  out->clip_coef = coef;
  out->clipped = (!found_inf && coef < 1.0f) ? 1 : 0;
  out->found_inf = found_inf ? 1 : 0;
}

// Sum of squares of 8 values: fp32 pairwise, exact fp64 outside the safe fp32 range.
__device__ __forceinline__ double sumsq8(const float (&x)[8]) {
  const float s01 = __fadd_rn(__fmul_rn(x[0], x[0]), __fmul_rn(x[1], x[1]));
  const float s23 = __fadd_rn(__fmul_rn(x[2], x[2]), __fmul_rn(x[3], x[3]));
  const float s45 = __fadd_rn(__fmul_rn(x[4], x[4]), __fmul_rn(x[5], x[5]));
  const float s67 = __fadd_rn(__fmul_rn(x[6], x[6]), __fmul_rn(x[7], x[7]));
  const float s = __fadd_rn(__fadd_rn(s01, s23), __fadd_rn(s45, s67));
  if (s >= 0x1p-96f && s <= FLT_MAX) return static_cast<double>(s);
  unsigned int any = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) any |= __float_as_uint(x[k]) & 0x7FFFFFFFu;
  if (any == 0) return 0.0;
  double d = 0.0;
#pragma unroll
  for (int k = 0; k < 8; ++k) d = __dadd_rn(d, __dmul_rn(static_cast<double>(x[k]), static_cast<double>(x[k])));
  return d;
}

// fp32 pairwise sum of squares of 8 values (no range check).
__device__ __forceinline__ float sumsq8f(const float (&x)[8]) {
  const float s01 = __fadd_rn(__fmul_rn(x[0], x[0]), __fmul_rn(x[1], x[1]));
  const float s23 = __fadd_rn(__fmul_rn(x[2], x[2]), __fmul_rn(x[3], x[3]));
  const float s45 = __fadd_rn(__fmul_rn(x[4], x[4]), __fmul_rn(x[5], x[5]));
  const float s67 = __fadd_rn(__fmul_rn(x[6], x[6]), __fmul_rn(x[7], x[7]));
  return __fadd_rn(__fadd_rn(s01, s23), __fadd_rn(s45, s67));
}

// Sum of squares of 32 values: fp32 pairwise while every 8-sum lies in [2^-96, 2^124] (no
// overflow in the 32-sum, no loss to fp32 underflow worth a bf16 result); otherwise each 8 as
// sumsq8 does (exact fp64 outside the safe range, NaN and Inf carried). One fp64 add per 32
// elements keeps the fp64 pipe, slow on this part, off the critical path.
__device__ __forceinline__ double sumsq32(const float (&a)[8], const float (&b)[8], const float (&c)[8],
                                          const float (&d)[8]) {
  const float s0 = sumsq8f(a), s1 = sumsq8f(b), s2 = sumsq8f(c), s3 = sumsq8f(d);
  const float lo = fminf(fminf(s0, s1), fminf(s2, s3)), hi = fmaxf(fmaxf(s0, s1), fmaxf(s2, s3));
  if (lo >= 0x1p-96f && hi <= 0x1p124f) return static_cast<double>(__fadd_rn(__fadd_rn(s0, s1), __fadd_rn(s2, s3)));
  return __dadd_rn(__dadd_rn(sumsq8(a), sumsq8(b)), __dadd_rn(sumsq8(c), sumsq8(d)));
}

// The raw bits of 8 elements (one 16-byte load of bf16, two of fp32) and their values.
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  uint4 a;
};
template <>
struct Raw8<float> {
  uint4 a, b;
};
__device__ __forceinline__ void ld_raw8(const __nv_bfloat16* p, Raw8<__nv_bfloat16>& r) {
  r.a = __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void ld_raw8(const float* p, Raw8<float>& r) {
  r.a = __ldg(reinterpret_cast<const uint4*>(p));
  r.b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
}
__device__ __forceinline__ void unpack8(const Raw8<__nv_bfloat16>& r, float (&x)[8]) {
  const unsigned int w[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = __uint_as_float(w[k] << 16);
    x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void unpack8(const Raw8<float>& r, float (&x)[8]) {
  x[0] = __uint_as_float(r.a.x); x[1] = __uint_as_float(r.a.y); x[2] = __uint_as_float(r.a.z);
  x[3] = __uint_as_float(r.a.w); x[4] = __uint_as_float(r.b.x); x[5] = __uint_as_float(r.b.y);
  x[6] = __uint_as_float(r.b.z); x[7] = __uint_as_float(r.b.w);
}
// 8-element vectors per round: 128 bytes of loads in flight per thread.
template <typename T>
constexpr int kRound = 16 / static_cast<int>(sizeof(T));

__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const unsigned int w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = __uint_as_float(w[k] << 16);
    x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float load1(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load1(const __nv_bfloat16* p) {
  return __uint_as_float(static_cast<unsigned int>(__ldg(reinterpret_cast<const unsigned short*>(p))) << 16);
}

// 4-element units: a warp's 32 consecutive units are 512 contiguous bytes of fp32 (256 of
// bf16), so every load instruction is fully coalesced.
__device__ __forceinline__ float4 load4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                     __uint_as_float(u.y & 0xFFFF0000u));
}
// sum of squares of two 4-element units (as one run of 8)
__device__ __forceinline__ double sumsq44(const float4& a, const float4& b) {
  const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  return sumsq8(x);
}

// Butterfly sum of an fp64 value over the block (fixed order); result valid in thread 0.
__device__ __forceinline__ double block_sum(double v, double* smem32) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __dadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) smem32[warp] = v;
  __syncthreads();
  double r = 0.0;
  if (warp == 0) {
    r = (lane < static_cast<int>(blockDim.x >> 5)) ? smem32[lane] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r = __dadd_rn(r, __shfl_xor_sync(0xFFFFFFFFu, r, o));
  }
  __syncthreads();
  return r;
}

// Publishes this block's partial; the last block to arrive reduces all partials in a fixed
// order, writes the stats and re-zeroes the arrival counter.
__device__ __forceinline__ void finish_sumsq(double acc, NormWorkspace* ws, zopt_clip_stats* stats,
                                             float max_norm) {
  __shared__ double red[32];
  __shared__ bool is_last;
  const double block = block_sum(acc, red);
  if (threadIdx.x == 0) {
    ws->partials[blockIdx.x] = block;
    __threadfence();
    const unsigned int ticket = atomicAdd(&ws->arrive, 1u);
    is_last = (ticket == gridDim.x - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  double a = 0.0;
  const volatile double* parts = ws->partials;
  for (unsigned int i = threadIdx.x; i < gridDim.x; i += blockDim.x) a = __dadd_rn(a, parts[i]);
  const double total = block_sum(a, red);
  if (threadIdx.x == 0) {
    write_clip_stats(stats, total, max_norm);
    ws->arrive = 0u;
    __threadfence();
  }
}

// Σ g² over n elements in one pass. Threads stride over 8-element vectors (16-byte aligned
// grad), kRound of them per round so that 128 bytes per thread are in flight; squares are
// summed in fp32 over runs of 32 (sumsq32: exact fp64 outside the safe range) and the runs in
// fp64 — the fp64 pipe, slow on this part, handles one add per 32 elements. The n % 8 tail
// goes to thread 0 of block 0 in fp64.
template <typename T>
__global__ void __launch_bounds__(kNormThreads) norm_kernel(const T* __restrict__ g, int64_t n, float max_norm,
                                                             NormWorkspace* ws, zopt_clip_stats* stats) {
  constexpr int R = kRound<T>;
  const int64_t n8 = n / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  double acc = 0.0;
  for (; j + (R - 1) * stride < n8; j += R * stride) {
    Raw8<T> r[R];
#pragma unroll
    for (int k = 0; k < R; ++k) ld_raw8(g + 8 * (j + k * stride), r[k]);
#pragma unroll
    for (int k = 0; k < R; k += 4) {
      float x0[8], x1[8], x2[8], x3[8];
      unpack8(r[k], x0);
      unpack8(r[k + 1], x1);
      unpack8(r[k + 2], x2);
      unpack8(r[k + 3], x3);
      acc = __dadd_rn(acc, sumsq32(x0, x1, x2, x3));
    }
  }
  for (; j < n8; j += stride) {
    float x[8];
    load8(g + 8 * j, x);
    acc = __dadd_rn(acc, sumsq8(x));
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    for (int64_t k = n8 * 8; k < n; ++k) {
      const double d = static_cast<double>(load1(g + k));
      acc = __dadd_rn(acc, __dmul_rn(d, d));
    }
  }
  finish_sumsq(acc, ws, stats, max_norm);
}

}  // namespace zopt
