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
// job's last product runs elsewhere and writes none); x0_raw[j], job j's matrices are already
// in X0, unnormalised (see many_x0).
zopt_status orthogonalize_many(const char* fn, const zopt_ns_job* jobs, int32_t n_jobs, int32_t steps,
                               const float* abc, float eps, void* d_ws, size_t ws_bytes, cudaStream_t s,
                               const zopt_dtype* out_io, const bool* norm_ready, const StatsSink* sinks = nullptr,
                               int* slots_out = nullptr, const bool* x0_raw = nullptr);
// Whether a job can take its matrices unnormalised in X0 (x0_raw of orthogonalize_many): bf16,
// rows <= cols, cols a multiple of 8. Such a job's matrices are written by the caller, as bf16
// with rows cols elements apart, to base[j] + b * stride[j] (elements); its norm partials go
// where many_norm_partials says (norm_ready), and the first step's products normalise. ok[j]
// tells whether job j can.
bool x0_raw_ok(long long rows, long long cols, zopt_dtype io);
void many_x0(const zopt_ns_job* jobs, int32_t n_jobs, void* d_ws, uint16_t** base, long long* stride, bool* ok);
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

// The error word that kernels with bounded waits set when a wait gives up (mapped host memory):
// returns ZOPT_ETIMEOUT (and clears the word) if a kernel of an earlier call set it, and gives
// the device address for this call's kernels in *dev.
zopt_status take_error_word(const char* fn, int** dev);

}  // namespace ns
}  // namespace zopt
