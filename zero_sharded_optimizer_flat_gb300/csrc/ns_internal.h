// Internal interfaces of the Newton-Schulz code: between its orchestration (ns.cu) and its fp32
// product kernel (ns_simt.cu), and the many-call options the Muon step (muon.cu) uses. Not part
// of the ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "zopt.h"

namespace zopt {
namespace ns {

// D = alpha * P Q + beta * R, fp32 accumulation. P is [M][K] row-major (leading dim ldp); Q
// is [K][N] (q_kn = 1) or [N][K] (q_kn = 0). symmetric: M == N, D symmetric, only tiles
// with tile column >= tile row are computed and the strictly upper part is mirrored.
// D is fp32 (d_f32) or bf16; d_trans writes D[i, j] at D[j * ldd + i].
// group: matrices in this launch (blockIdx.y), the *_stride fields their distance in elements.
struct GemmF32Args {
  int M, N, K;
  int group;
  const float* P;
  long long ldp, p_stride;
  const float* Q;
  long long ldq, q_stride;
  int q_kn;
  int symmetric;
  float alpha, beta;
  const float* R;
  long long ldr, r_stride;
  void* D;
  long long ldd, d_stride;
  int d_f32;
  int d_trans;
};

zopt_status launch_gemm_f32(const GemmF32Args& a, cudaStream_t stream);

// Where a caller wants the statistics of a job's output: the sum of squares and the largest
// magnitude of each (tile, epilogue warp) part of matrix b's output go to slots of sum + b *
// stride and max + b * stride, at most cap of them per matrix.
struct StatsSink {
  double* sum;
  unsigned* max;
  long long stride, cap;
};

// zopt_ns_orthogonalize_many with per-job options for callers inside the library (null: the
// entry point's behaviour): out_io[j], the dtype job j's X is written in (its G keeps io_dtype);
// norm_ready[j], job j's matrices' norm partials are already in the workspace (see
// many_norm_partials), so the sum-of-squares launch skips them; sinks[j], where the epilogue of
// job j's last product writes its output's statistics when that epilogue is a TMA one (a
// CTA-pair or fused launch), slots_out[j] then the number of slots per matrix it fills (0: the
// job's last product runs elsewhere and writes none).
zopt_status orthogonalize_many(const char* fn, const zopt_ns_job* jobs, int32_t n_jobs, int32_t steps,
                               const float* abc, float eps, void* d_ws, size_t ws_bytes, cudaStream_t s,
                               const zopt_dtype* out_io, const bool* norm_ready, const StatsSink* sinks = nullptr,
                               int* slots_out = nullptr);
// Statistics slots per matrix that any path of a rows x cols job may fill (a bound for sinks).
long long stats_slots_bound(long long rows, long long cols);

// Where job j of a many-call keeps its matrices' norm partials in the workspace d_ws: matrix b's
// blocks' fp64 sums of squares at base[j] + b * stride_doubles, norm_blocks(rows * cols) of them
// (the normalising kernels add them in index order).
void many_norm_partials(const zopt_ns_job* jobs, int32_t n_jobs, void* d_ws, double** base, long long* stride_doubles);
// Norm partial sums a matrix of n elements takes: ceil(n / 32768), at least 1, at most
// kNormPartialsMax (a function of n only, so a matrix's norm is the same in any call).
constexpr int kNormPartialsMax = 512;
int norm_blocks(long long n);

}  // namespace ns
}  // namespace zopt
