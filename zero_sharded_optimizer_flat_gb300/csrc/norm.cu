// Gradient sum of squares, global norm, clip coefficient and found_inf, kept on the device.
//
// deg/zero.py, grad_sq_norm (the shard gradient's squared L2 norm; no all-reduce for a
// simulated rank); bluscript_zero_ckpt.cpp, global clip block (coef = min(1, max_norm /
// (norm + 1e-6)), a NaN norm never reaches min); dmuon PR #16, sync-free clip stats (0-dim
// device values; an inf norm gives coef 0, found_inf true, clipped false).
//
// One launch: every block reduces a grid-stride share of the gradient to an fp64 partial;
// the last block to arrive (arrival counter in the workspace) sums the partials in a fixed
// order and writes the stats. For a given n and GPU the grid is fixed, so the result is
// bitwise reproducible.
//
// Per element the squares are summed in fp32 over runs of 8 (pairwise), and the run sums
// are accumulated in fp64; GB300's fp64 rate is far too low for one fp64 FMA per element at
// HBM speed. A run sum outside [2^-96, FLT_MAX] (a zero run, values small enough to lose
// bits to underflow, an fp32 overflow, or inf/NaN inputs) is recomputed exactly in fp64,
// so a finite gradient never overflows and non-finite inputs always reach the sum.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>

#include "internal.h"
#include "launch.cuh"
#include "norm_impl.cuh"

namespace zopt {

size_t norm_grid_blocks(int64_t n) {
  const int64_t nvec = n / 8;
  int64_t want = (nvec + kNormThreads * 2 - 1) / (kNormThreads * 2);
  if (want < 1) want = 1;
  return static_cast<size_t>(want < kNormMaxBlocks ? want : kNormMaxBlocks);
}

int norm_launch_blocks(int64_t n, zopt_dtype dtype) {
  // resident blocks per SM of each instantiation
  auto occ_of = [](const void* kernel) {
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kernel, kNormThreads, 0) != cudaSuccess || o < 1) o = 1;
    return o < kNormBlocksPerSm ? o : kNormBlocksPerSm;
  };
  const int occ = dtype == ZOPT_F32 ? once([&] { return occ_of(reinterpret_cast<const void*>(norm_kernel<float>)); })
                                    : once([&] { return occ_of(reinterpret_cast<const void*>(norm_kernel<__nv_bfloat16>)); });
  const int sms = sm_count();
  if (sms <= 0) return 0;
  // one wave of resident blocks; never more blocks than the workspace was sized for
  int64_t blocks = static_cast<int64_t>(norm_grid_blocks(n));
  const int64_t wave = static_cast<int64_t>(sms) * occ;
  return static_cast<int>(blocks < wave ? blocks : wave);
}

zopt_status launch_norm(const void* grad, zopt_dtype dtype, int64_t n, float max_norm, NormWorkspace* ws,
                        zopt_clip_stats* stats, cudaStream_t stream) {
  const int blocks = norm_launch_blocks(n, dtype);
  if (blocks <= 0) return fail(ZOPT_ECUDA, "zopt_grad_norm_clip: no CUDA device");
  if (dtype == ZOPT_F32)
    norm_kernel<float><<<static_cast<unsigned>(blocks), kNormThreads, 0, stream>>>(
        static_cast<const float*>(grad), n, max_norm, ws, stats);
  else
    norm_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), kNormThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(grad), n, max_norm, ws, stats);
  ZOPT_CUDA_TRY(cudaGetLastError());
  return ok();
}

zopt_status check_norm_args(const char* fn, const void* grad, zopt_dtype dtype, int64_t n, float max_norm,
                            const zopt_clip_stats* stats) {
  if (n < 1) return fail(ZOPT_EINVAL, std::string(fn) + ": n < 1");
  if (grad == nullptr || stats == nullptr) return fail(ZOPT_EINVAL, std::string(fn) + ": NULL pointer");
  if (!aligned16(grad)) return fail(ZOPT_EINVAL, std::string(fn) + ": grad is not 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(stats) & 7u) != 0)
    return fail(ZOPT_EINVAL, std::string(fn) + ": stats is not 8-byte aligned");
  if (dtype != ZOPT_F32 && dtype != ZOPT_BF16) return fail(ZOPT_EUNSUPPORTED, std::string(fn) + ": grad dtype");
  if (!(max_norm >= 0.0f)) return fail(ZOPT_EINVAL, std::string(fn) + ": max_norm is negative or NaN");
  return ok();
}

}  // namespace zopt

extern "C" size_t zopt_grad_norm_workspace(int64_t n) {
  if (n < 1) return 0;
  return sizeof(zopt::NormWorkspace) + sizeof(double) * zopt::norm_grid_blocks(n);
}

extern "C" zopt_status zopt_grad_norm_clip(const void* grad, zopt_dtype dtype, int64_t n, float max_norm,
                                           void* d_ws, size_t ws_bytes, zopt_clip_stats* d_stats,
                                           zopt_stream stream) {
  zopt_status st = zopt::check_norm_args("zopt_grad_norm_clip", grad, dtype, n, max_norm, d_stats);
  if (st != ZOPT_OK) return st;
  if (d_ws == nullptr || !zopt::aligned16(d_ws))
    return zopt::fail(ZOPT_EINVAL, "zopt_grad_norm_clip: workspace is NULL or not 16-byte aligned");
  if (ws_bytes < zopt_grad_norm_workspace(n))
    return zopt::fail(ZOPT_EINVAL, "zopt_grad_norm_clip: workspace smaller than zopt_grad_norm_workspace(n)");
  return zopt::launch_norm(grad, dtype, n, max_norm, static_cast<zopt::NormWorkspace*>(d_ws), d_stats,
                           reinterpret_cast<cudaStream_t>(stream));
}

namespace {
__global__ void clip_finalize_kernel(zopt_clip_stats* stats, float max_norm) {
  if (threadIdx.x == 0 && blockIdx.x == 0) zopt::write_clip_stats(stats, stats->sumsq, max_norm);
}
}  // namespace

extern "C" zopt_status zopt_clip_finalize(zopt_clip_stats* d_stats, float max_norm, zopt_stream stream) {
  if (d_stats == nullptr) return zopt::fail(ZOPT_EINVAL, "zopt_clip_finalize: stats is NULL");
  if (!(max_norm >= 0.0f)) return zopt::fail(ZOPT_EINVAL, "zopt_clip_finalize: max_norm is negative or NaN");
  clip_finalize_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(d_stats, max_norm);
  ZOPT_CUDA_TRY(cudaGetLastError());
  return zopt::ok();
}
