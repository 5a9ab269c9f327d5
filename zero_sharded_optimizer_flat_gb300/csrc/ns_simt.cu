// fp32 Newton-Schulz products on the CUDA cores (the precision mode of zopt_ns_orthogonalize).
//
// bf16 tensor-core products keep about 8 significant bits per product; a caller that needs the
// iteration to agree with fp64 to 1e-4 uses compute_dtype ZOPT_F32, which runs the same three
// products (A = X X', B = c A A' + b A, X = B X + a X) in fp32 FMA. TF32 tensor cores (10
// explicit mantissa bits) cannot reach that tolerance, so this is a plain SIMT kernel:
// 128 x 128 output tiles, 256 threads each holding an 8 x 8 sub-tile, 16-deep k-slices staged
// through double-buffered shared memory (k-major, padded rows, float4 reads).
#include <cuda_runtime.h>

#include "internal.h"
#include "ns_internal.h"

namespace zopt {
namespace ns {
namespace {

constexpr int TM = 128, TN = 128, TK = 16, TT = 256;
constexpr int kPad = 4;

__device__ __forceinline__ void tile_of(const GemmF32Args& a, int tiles_n, int t, int& ti, int& tj) {
  if (!a.symmetric) {
    ti = t / tiles_n;
    tj = t % tiles_n;
    return;
  }
  // square tiles: row r holds tiles tj = r .. tiles_n-1
  int r = 0;
  for (;;) {
    const int cnt = tiles_n - r;
    if (t < cnt) {
      ti = r;
      tj = r + t;
      return;
    }
    t -= cnt;
    ++r;
  }
}

__device__ __forceinline__ void put(const GemmF32Args& a, long long off, float v) {
  if (a.d_f32)
    static_cast<float*>(a.D)[off] = v;
  else
    static_cast<__nv_bfloat16*>(a.D)[off] = __float2bfloat16_rn(v);
}

__global__ void __launch_bounds__(TT) gemm_f32_kernel(GemmF32Args a, int tiles_n) {
  {  // this block's matrix of the group
    const long long mb = blockIdx.y;
    a.P += mb * a.p_stride;
    a.Q += mb * a.q_stride;
    if (a.R != nullptr) a.R += mb * a.r_stride;
    a.D = static_cast<uint8_t*>(a.D) + mb * a.d_stride * (a.d_f32 ? 4 : 2);
  }
  __shared__ __align__(16) float As[2][TK][TM + kPad];
  __shared__ __align__(16) float Bs[2][TK][TN + kPad];
  int ti, tj;
  tile_of(a, tiles_n, blockIdx.x, ti, tj);
  const int m0 = ti * TM, n0 = tj * TN;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
  float ra[8], rb[8];

  auto load = [&](int k0) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = tid + TT * q;
      const int r = m0 + (e >> 4), c = k0 + (e & 15);
      ra[q] = (r < a.M && c < a.K) ? a.P[static_cast<long long>(r) * a.ldp + c] : 0.0f;
      if (a.q_kn) {
        const int kr = k0 + (e >> 7), n = n0 + (e & 127);
        rb[q] = (kr < a.K && n < a.N) ? a.Q[static_cast<long long>(kr) * a.ldq + n] : 0.0f;
      } else {
        const int n = n0 + (e >> 4), kc = k0 + (e & 15);
        rb[q] = (n < a.N && kc < a.K) ? a.Q[static_cast<long long>(n) * a.ldq + kc] : 0.0f;
      }
    }
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = tid + TT * q;
      As[buf][e & 15][e >> 4] = ra[q];
      if (a.q_kn)
        Bs[buf][e >> 7][e & 127] = rb[q];
      else
        Bs[buf][e & 15][e >> 4] = rb[q];
    }
  };

  const int nk = (a.K + TK - 1) / TK;
  load(0);
  store(0);
  __syncthreads();
  for (int kt = 0; kt < nk; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < nk) load((kt + 1) * TK);
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (kt + 1 < nk) store(buf ^ 1);
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (r >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
      if (c >= a.N) continue;
      float o = a.alpha * acc[i][j];
      if (a.beta != 0.0f) o = fmaf(a.beta, a.R[static_cast<long long>(r) * a.ldr + c], o);
      if (a.symmetric) {
        if (c >= r) put(a, static_cast<long long>(r) * a.ldd + c, o);
        if (c > r) put(a, static_cast<long long>(c) * a.ldd + r, o);
      } else if (a.d_trans) {
        put(a, static_cast<long long>(c) * a.ldd + r, o);
      } else {
        put(a, static_cast<long long>(r) * a.ldd + c, o);
      }
    }
  }
}

}  // namespace

zopt_status launch_gemm_f32(const GemmF32Args& a, cudaStream_t stream) {
  const int tiles_m = (a.M + TM - 1) / TM, tiles_n = (a.N + TN - 1) / TN;
  long long tiles = 0;
  if (a.symmetric) {
    for (int r = 0; r < tiles_m; ++r) tiles += tiles_n - r;
  } else {
    tiles = static_cast<long long>(tiles_m) * tiles_n;
  }
  if (tiles < 1 || tiles > 0x7FFFFFFF) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: fp32 product too large");
  if (a.group < 1 || a.group > 65535) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: group out of range");
  gemm_f32_kernel<<<dim3(static_cast<unsigned>(tiles), static_cast<unsigned>(a.group)), TT, 0, stream>>>(a, tiles_n);
  ZOPT_CUDA_TRY(cudaGetLastError());
  return ok();
}

}  // namespace ns
}  // namespace zopt
