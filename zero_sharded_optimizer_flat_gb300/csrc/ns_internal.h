// Internal interface between the Newton-Schulz orchestration (ns.cu) and its fp32 product
// kernel (ns_simt.cu). Not part of the ABI.
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

}  // namespace ns
}  // namespace zopt
