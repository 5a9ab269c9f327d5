// Micro-step gradient accumulation into the fp32 shard gradient, with the clip statistics
// fused into the last micro-step's pass.
//
// deg/zero.py, ZeroMaster: a step's bf16 gradients from several parts are summed in fp32
// (``collect`` keeps an fp32 sum; ``reduce_scatter`` sums into the owner's fp32 shard
// gradient), and ``grad_sq_norm`` then reads that fp32 shard. Here the sum lives in HBM and
// the last micro-step's pass produces the sum of squares of the finished sum, so the norm
// costs no extra read of the shard (4 B per element saved).
//
// acc = g_1 (first micro-step: acc is not read), then acc = acc + g_k in fp32, each addition
// rounded, in micro-step order. Bytes per element: 6 (first, bf16), 10 (later micro-steps).
// The arrays are walked in 4-element units, a warp's 32 units contiguous (512 B of fp32, 256 B of
// bf16 per load instruction); each thread issues the loads of four units before it adds and
// stores any of them, so that enough bytes are in flight to keep HBM busy.
//
// A micro-step gradient may also sit in page-locked host memory: the pass then reads it through
// the device mapping of that memory, over the CPU-GPU link, with no staging copy in HBM (the
// host-to-device transfer and the addition are one pass).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "launch.cuh"
#include "norm_impl.cuh"

namespace zopt {
namespace {

__device__ __forceinline__ float4 add4(const float4& a, const float4& b) {
  return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}

template <typename T, bool kFirst, bool kLast, bool kTwo>
__global__ void __launch_bounds__(kNormThreads) accum_kernel(float* __restrict__ acc, const T* __restrict__ g,
                                                              const T* __restrict__ g2, int64_t n, float max_norm,
                                                              NormWorkspace* ws, zopt_clip_stats* stats) {
  const int64_t n4 = n / 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  float4* acc4 = reinterpret_cast<float4*>(acc);
  double ss = 0.0;
  for (; j + 3 * stride < n4; j += 4 * stride) {
    float4 x[4], a[4], y[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {  // every load of the four units first
      x[u] = load4(g + 4 * (j + u * stride));
      if (kTwo) y[u] = load4(g2 + 4 * (j + u * stride));
      if (!kFirst) a[u] = acc4[j + u * stride];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (!kFirst) x[u] = add4(a[u], x[u]);
      if (kTwo) x[u] = add4(x[u], y[u]);
      acc4[j + u * stride] = x[u];
    }
    if (kLast) ss = __dadd_rn(ss, __dadd_rn(sumsq44(x[0], x[1]), sumsq44(x[2], x[3])));
  }
  for (; j < n4; j += stride) {
    float4 x = load4(g + 4 * j);
    if (!kFirst) x = add4(acc4[j], x);
    if (kTwo) x = add4(x, load4(g2 + 4 * j));
    acc4[j] = x;
    if (kLast) ss = __dadd_rn(ss, sumsq44(x, make_float4(0.f, 0.f, 0.f, 0.f)));
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    for (int64_t k = n4 * 4; k < n; ++k) {
      float v = kFirst ? load1(g + k) : __fadd_rn(acc[k], load1(g + k));
      if (kTwo) v = __fadd_rn(v, load1(g2 + k));
      acc[k] = v;
      if (kLast) ss = __dadd_rn(ss, __dmul_rn(static_cast<double>(v), static_cast<double>(v)));
    }
  }
  if (kLast) finish_sumsq(ss, ws, stats, max_norm);
}

template <typename K>
int resident_blocks(K kernel) {
  int o = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kernel, kNormThreads, 0) != cudaSuccess || o < 1) o = 1;
  return o < kNormBlocksPerSm ? o : kNormBlocksPerSm;
}

template <typename T, bool kFirst, bool kLast, bool kTwo>
zopt_status launch(float* acc, const void* g, const void* g2, int64_t n, float max_norm, NormWorkspace* ws,
                   zopt_clip_stats* stats, cudaStream_t s) {
  // The grid decides how the sum of squares is split over threads and blocks, so every pass that
  // produces the stats (kLast) runs on one grid: a wave of whichever of the single-part and
  // two-part last kernels holds fewer blocks per SM. A two-part last pass is then bit for bit
  // the single-part calls it replaces, and neither kernel runs its grid in more than one wave.
  // A pass without stats runs on a wave of its own kernel.
  const int occ = once([] {
    if (!kLast) return resident_blocks(accum_kernel<T, kFirst, kLast, kTwo>);
    const int one = resident_blocks(accum_kernel<T, false, true, false>);
    const int two = resident_blocks(accum_kernel<T, false, true, true>);
    return one < two ? one : two;
  });
  const int sms = sm_count();
  if (sms <= 0) return fail(ZOPT_ECUDA, "zopt_grad_accumulate: no CUDA device");
  int64_t blocks = static_cast<int64_t>(norm_grid_blocks(n));
  const int64_t wave = static_cast<int64_t>(sms) * occ;
  if (blocks > wave) blocks = wave;
  accum_kernel<T, kFirst, kLast, kTwo><<<static_cast<unsigned>(blocks), kNormThreads, 0, s>>>(
      acc, static_cast<const T*>(g), static_cast<const T*>(g2), n, max_norm, ws, stats);
  ZOPT_CUDA_TRY(cudaGetLastError());
  return ok();
}

template <typename T, bool kTwo>
zopt_status dispatch(bool first, bool last, float* acc, const void* g, const void* g2, int64_t n, float max_norm,
                     NormWorkspace* ws, zopt_clip_stats* stats, cudaStream_t s) {
  if (first && last) return launch<T, true, true, kTwo>(acc, g, g2, n, max_norm, ws, stats, s);
  if (first) return launch<T, true, false, kTwo>(acc, g, g2, n, max_norm, ws, stats, s);
  if (last) return launch<T, false, true, kTwo>(acc, g, g2, n, max_norm, ws, stats, s);
  return launch<T, false, false, kTwo>(acc, g, g2, n, max_norm, ws, stats, s);
}

// The address the kernel reads micro_grad through: device (or managed) memory as it is;
// page-locked host memory through its device mapping, so the pass itself pulls the micro-step
// over the host link and no staging copy in HBM is needed. Pageable host memory is refused.
zopt_status device_view(const void* p, const void** out) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(ZOPT_EINVAL, "zopt_grad_accumulate: micro_grad is not a CUDA-visible address");
  }
  int dev = -1;
  ZOPT_CUDA_TRY(cudaGetDevice(&dev));
  switch (a.type) {
    case cudaMemoryTypeDevice:
      if (a.device != dev) return fail(ZOPT_EINVAL, "zopt_grad_accumulate: micro_grad is on another device");
      *out = p;
      return ok();
    case cudaMemoryTypeManaged:
      *out = p;
      return ok();
    case cudaMemoryTypeHost:
      if (a.devicePointer == nullptr)
        return fail(ZOPT_EINVAL, "zopt_grad_accumulate: micro_grad's page-locked host memory has no device mapping");
      *out = a.devicePointer;
      return ok();
    default:
      return fail(ZOPT_EINVAL, "zopt_grad_accumulate: micro_grad is pageable host memory (pin or register it)");
  }
}

}  // namespace
}  // namespace zopt

namespace zopt {
namespace {

// The checks and the launch shared by both entry points (g2 == nullptr: one part).
zopt_status accumulate(const char* fn, float* acc, const void* micro_grad, const void* micro_grad2, zopt_dtype dtype,
                       int64_t n, int32_t flags, float max_norm, void* d_ws, size_t ws_bytes, zopt_clip_stats* d_stats,
                       zopt_stream stream) {
  const std::string f(fn);
  const bool first = (flags & ZOPT_ACC_FIRST) != 0, last = (flags & ZOPT_ACC_LAST) != 0;
  if ((flags & ~(ZOPT_ACC_FIRST | ZOPT_ACC_LAST)) != 0) return fail(ZOPT_EINVAL, f + ": unknown flags");
  if (n < 1) return fail(ZOPT_EINVAL, f + ": n < 1");
  if (acc == nullptr || micro_grad == nullptr) return fail(ZOPT_EINVAL, f + ": NULL pointer");
  if (!aligned16(acc) || !aligned16(micro_grad) || (micro_grad2 != nullptr && !aligned16(micro_grad2)))
    return fail(ZOPT_EINVAL, f + ": acc or a micro_grad is not 16-byte aligned");
  if (dtype != ZOPT_F32 && dtype != ZOPT_BF16) return fail(ZOPT_EUNSUPPORTED, f + ": grad dtype");
  if (last) {
    if (d_stats == nullptr || (reinterpret_cast<uintptr_t>(d_stats) & 7u) != 0)
      return fail(ZOPT_EINVAL, f + ": the last micro-step needs an 8-byte aligned stats struct");
    if (!(max_norm >= 0.0f)) return fail(ZOPT_EINVAL, f + ": max_norm is negative or NaN");
    if (d_ws == nullptr || !aligned16(d_ws) || ws_bytes < zopt_grad_norm_workspace(n))
      return fail(ZOPT_EINVAL, f + ": the last micro-step needs a zopt_grad_norm_workspace(n) workspace");
  }
  const void* g = nullptr;
  const void* g2 = nullptr;
  zopt_status st = device_view(micro_grad, &g);
  if (st == ZOPT_OK && micro_grad2 != nullptr) st = device_view(micro_grad2, &g2);
  if (st != ZOPT_OK) return st;
  if (!aligned16(g) || (g2 != nullptr && !aligned16(g2)))
    return fail(ZOPT_EINVAL, f + ": a micro_grad's device address is not 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  NormWorkspace* ws = static_cast<NormWorkspace*>(d_ws);
  if (g2 == nullptr)
    return dtype == ZOPT_F32 ? dispatch<float, false>(first, last, acc, g, g2, n, max_norm, ws, d_stats, s)
                             : dispatch<__nv_bfloat16, false>(first, last, acc, g, g2, n, max_norm, ws, d_stats, s);
  return dtype == ZOPT_F32 ? dispatch<float, true>(first, last, acc, g, g2, n, max_norm, ws, d_stats, s)
                           : dispatch<__nv_bfloat16, true>(first, last, acc, g, g2, n, max_norm, ws, d_stats, s);
}

}  // namespace
}  // namespace zopt

extern "C" zopt_status zopt_grad_accumulate(float* acc, const void* micro_grad, zopt_dtype dtype, int64_t n,
                                            int32_t flags, float max_norm, void* d_ws, size_t ws_bytes,
                                            zopt_clip_stats* d_stats, zopt_stream stream) {
  return zopt::accumulate("zopt_grad_accumulate", acc, micro_grad, nullptr, dtype, n, flags, max_norm, d_ws,
                          ws_bytes, d_stats, stream);
}

extern "C" zopt_status zopt_grad_accumulate2(float* acc, const void* micro_grad_a, const void* micro_grad_b,
                                             zopt_dtype dtype, int64_t n, int32_t flags, float max_norm, void* d_ws,
                                             size_t ws_bytes, zopt_clip_stats* d_stats, zopt_stream stream) {
  if (micro_grad_b == nullptr) return zopt::fail(ZOPT_EINVAL, "zopt_grad_accumulate2: NULL pointer");
  return zopt::accumulate("zopt_grad_accumulate2", acc, micro_grad_a, micro_grad_b, dtype, n, flags, max_norm, d_ws,
                          ws_bytes, d_stats, stream);
}
