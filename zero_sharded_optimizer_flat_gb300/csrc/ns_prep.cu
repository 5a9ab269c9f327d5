// Newton-Schulz preparation: the Frobenius norm of every matrix of a group and X0 = G / (||G||
// + eps) in the compute dtype, transposed for a tall matrix.
#include "ns_tile.cuh"

namespace zopt {
namespace ns {

// Sum of squares of each matrix of the group (blockIdx.y = matrix): G_b is rows x cols with
// leading dimension ld, matrices batch_stride elements apart. `flat` = rows are contiguous
// (ld == cols) and 16-byte aligned, so the matrix is one vector.
template <typename T>
__global__ void __launch_bounds__(kNormThreads)
    group_sumsq_kernel(const T* __restrict__ g0, long long rows, long long cols, long long ld,
                       long long batch_stride, int flat, int vec_rows, uint8_t* ws_base,
                       zopt_clip_stats* stats) {
  tc::pdl_launch_dependents();
  tc::pdl_wait();
  const int mb = blockIdx.y;
  const T* g = g0 + mb * batch_stride;
  double acc = 0.0;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (flat) {
    const long long n = rows * cols, nvec = n / 8;
    long long i = tid;
    for (; i + stride < nvec; i += 2 * stride) {
      float x[8], y[8];
      load8(g + 8 * i, x);
      load8(g + 8 * (i + stride), y);
      acc = __dadd_rn(acc, __dadd_rn(sumsq8(x), sumsq8(y)));
    }
    for (; i < nvec; i += stride) {
      float x[8];
      load8(g + 8 * i, x);
      acc = __dadd_rn(acc, sumsq8(x));
    }
    for (long long k = nvec * 8 + tid; k < n; k += stride) {
      const double d = static_cast<double>(load1(g + k));
      acc = __dadd_rn(acc, __dmul_rn(d, d));
    }
  } else {
    const long long c8 = vec_rows ? cols / 8 : 0;
    for (long long e = tid; e < rows * c8; e += stride) {
      const long long r = e / c8, c = e - r * c8;
      float x[8];
      load8(g + r * ld + 8 * c, x);
      acc = __dadd_rn(acc, sumsq8(x));
    }
    const long long tail = cols - 8 * c8;
    for (long long e = tid; e < rows * tail; e += stride) {
      const long long r = e / tail, c = 8 * c8 + (e - r * tail);
      const double d = static_cast<double>(load1(g + r * ld + c));
      acc = __dadd_rn(acc, __dmul_rn(d, d));
    }
  }
  finish_sumsq(acc, prep_ws(ws_base, mb), stats + mb, 0.0f);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void to_out(float v, __nv_bfloat16* p) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void to_out(float v, float* p) { *p = v; }

__device__ __forceinline__ float2 load2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 load2(const __nv_bfloat16* p) {
  const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}
__device__ __forceinline__ void store2(float* p, float a, float b) { *reinterpret_cast<float2*>(p) = make_float2(a, b); }
__device__ __forceinline__ void store2(__nv_bfloat16* p, float a, float b) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
}
__device__ __forceinline__ void store8(float* p, const float (&x)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&x)[8]) {
  __nv_bfloat162 h[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
  *reinterpret_cast<uint4*>(p) = *reinterpret_cast<const uint4*>(h);
}

__device__ __forceinline__ float inv_norm(const zopt_clip_stats* st, double eps) {
  return __double2float_rn(__ddiv_rn(1.0, __dadd_rn(__dsqrt_rn(st->sumsq), eps)));
}

// X0_b = G_b / (||G_b||_F + eps) in the compute dtype U, same orientation (rows <= cols),
// blockIdx.y = matrix. vec: rows of G are 16-byte aligned with cols % 8 == 0, so each thread
// moves 8 elements per access; otherwise one element at a time.
template <typename T, typename U>
__global__ void __launch_bounds__(256) group_scale_kernel(const T* __restrict__ g0, long long rows, long long cols,
                                                          long long ld, long long batch_stride, int vec,
                                                          const zopt_clip_stats* stats, double eps,
                                                          U* __restrict__ x0, long long ldx, long long x_stride) {
  __shared__ float s_inv;
  tc::pdl_launch_dependents();
  tc::pdl_wait();
  const int mb = blockIdx.y;
  const T* g = g0 + mb * batch_stride;
  U* x = x0 + mb * x_stride;
  if (threadIdx.x == 0) s_inv = inv_norm(stats + mb, eps);
  __syncthreads();
  const float inv = s_inv;
  if (vec) {
    const long long c8 = cols / 8;
    for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
      for (long long c = threadIdx.x; c < c8; c += blockDim.x) {
        float v[8];
        load8(g + r * ld + 8 * c, v);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] *= inv;
        store8(x + r * ldx + 8 * c, v);
      }
    }
  } else {
    for (long long r = blockIdx.x; r < rows; r += gridDim.x)
      for (long long c = threadIdx.x; c < cols; c += blockDim.x) to_out(to_f32(g[r * ld + c]) * inv, x + r * ldx + c);
  }
}

// X0_b = (G_b / (||G_b||_F + eps))' for a tall G (rows > cols): 64 x 64 tiles through shared
// memory, 32 x 8 threads; pair: G's rows allow 2-element accesses (each warp then reads and
// writes 128 contiguous bytes of bf16).
template <typename T, typename U>
__global__ void __launch_bounds__(256) group_transpose_kernel(const T* __restrict__ g0, long long rows, long long cols,
                                                              long long ld, long long batch_stride, int pair,
                                                              const zopt_clip_stats* stats, double eps,
                                                              U* __restrict__ x0, long long ldx, long long x_stride) {
  __shared__ float s_inv;
  __shared__ float tile[64][65];
  tc::pdl_launch_dependents();
  tc::pdl_wait();
  const int mb = blockIdx.y;
  const T* g = g0 + mb * batch_stride;
  U* x = x0 + mb * x_stride;
  if (threadIdx.x == 0 && threadIdx.y == 0) s_inv = inv_norm(stats + mb, eps);
  __syncthreads();
  const float inv = s_inv;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const long long tiles_c = (cols + 63) / 64, tiles_r = (rows + 63) / 64;
  for (long long tt = blockIdx.x; tt < tiles_r * tiles_c; tt += gridDim.x) {
    const long long r0 = (tt / tiles_c) * 64, c0 = (tt % tiles_c) * 64;
    const bool full = r0 + 64 <= rows && c0 + 64 <= cols;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int rr = ty + 8 * k;
      const long long r = r0 + rr, c = c0 + 2 * tx;
      if (full && pair) {
        const float2 v = load2(g + r * ld + c);
        tile[rr][2 * tx] = v.x * inv;
        tile[rr][2 * tx + 1] = v.y * inv;
      } else {
        tile[rr][2 * tx] = (r < rows && c < cols) ? to_f32(g[r * ld + c]) * inv : 0.0f;
        tile[rr][2 * tx + 1] = (r < rows && c + 1 < cols) ? to_f32(g[r * ld + c + 1]) * inv : 0.0f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int cc = ty + 8 * k;                    // X0 row = G column c0 + cc
      const long long xr = c0 + cc, xc = r0 + 2 * tx;  // X0[c][r] = G[r][c]
      if (full) {
        store2(x + xr * ldx + xc, tile[2 * tx][cc], tile[2 * tx + 1][cc]);
      } else {
        if (xr < cols && xc < rows) to_out(tile[2 * tx][cc], x + xr * ldx + xc);
        if (xr < cols && xc + 1 < rows) to_out(tile[2 * tx + 1][cc], x + xr * ldx + xc + 1);
      }
    }
    __syncthreads();
  }
}

// X0 = G / (||G||_F + eps), oriented, for every matrix of the group (its prep scratch, and so
// its counters, zeroed first).
zopt_status group_prep(const Group& G, float eps, int sms, cudaStream_t s) {
  zopt_status st = ZOPT_OK;
  const long long rows = G.rows, cols = G.cols, ld_g = G.ld_g, bs_g = G.bs_g;
  const size_t esz = G.esz;
  const int gs = G.gs;
  ZOPT_CUDA_TRY(cudaMemsetAsync(G.ws, 0, static_cast<size_t>(gs) * kPrepWsBytes, s));
  const bool aligned = (reinterpret_cast<uintptr_t>(G.g) & 15u) == 0 && (bs_g * esz) % 16 == 0;
  const int flat = (aligned && ld_g == cols) ? 1 : 0;
  const int vec_rows = (aligned && (ld_g * esz) % 16 == 0) ? 1 : 0;
  // blocks per matrix depend on the matrix size only, so a matrix's sum (and so its result)
  // is bitwise the same whatever group it runs in
  long long bpm = (rows * cols + 8191) / 8192;  // short per-thread chains for small matrices
  bpm = bpm < 1 ? 1 : (bpm > kPrepBlocks ? kPrepBlocks : bpm);
  const dim3 sg(static_cast<unsigned>(bpm), static_cast<unsigned>(gs));
  st = G.io == ZOPT_F32
           ? launch_pdl(group_sumsq_kernel<float>, sg, dim3(kNormThreads), 0, s, reinterpret_cast<const float*>(G.g),
                        rows, cols, ld_g, bs_g, flat, vec_rows, G.ws, G.stats)
           : launch_pdl(group_sumsq_kernel<__nv_bfloat16>, sg, dim3(kNormThreads), 0, s,
                        reinterpret_cast<const __nv_bfloat16*>(G.g), rows, cols, ld_g, bs_g, flat, vec_rows, G.ws,
                        G.stats);
  if (st != ZOPT_OK) return st;
  int sblk = (sms * 8 + gs - 1) / gs;
  sblk = sblk < 1 ? 1 : sblk;
  const dim3 sgrid(static_cast<unsigned>(sblk), static_cast<unsigned>(gs));
  const zopt_clip_stats* stats = G.stats;
  if (!G.transpose) {
    const int vec = (aligned && (ld_g * esz) % 16 == 0 && cols % 8 == 0) ? 1 : 0;
#define ZOPT_SCALE(TI, TO)                                                                                 \
  st = launch_pdl(group_scale_kernel<TI, TO>, sgrid, dim3(256), 0, s, reinterpret_cast<const TI*>(G.g), rows, \
                  cols, ld_g, bs_g, vec, stats, static_cast<double>(eps), reinterpret_cast<TO*>(G.xb[0]),       \
                  G.p.ldx, G.mat_elems)
    if (G.io == ZOPT_F32 && G.f32c) ZOPT_SCALE(float, float);
    else if (G.io == ZOPT_F32) ZOPT_SCALE(float, __nv_bfloat16);
    else if (G.f32c) ZOPT_SCALE(__nv_bfloat16, float);
    else ZOPT_SCALE(__nv_bfloat16, __nv_bfloat16);
#undef ZOPT_SCALE
  } else {
    const int pair = ((reinterpret_cast<uintptr_t>(G.g) % (2 * esz)) == 0 && ld_g % 2 == 0 && bs_g % 2 == 0) ? 1 : 0;
    const dim3 tb(32, 8);
#define ZOPT_TRANSPOSE(TI, TO)                                                                            \
  st = launch_pdl(group_transpose_kernel<TI, TO>, sgrid, tb, 0, s, reinterpret_cast<const TI*>(G.g), rows,   \
                  cols, ld_g, bs_g, pair, stats, static_cast<double>(eps), reinterpret_cast<TO*>(G.xb[0]),     \
                  G.p.ldx, G.mat_elems)
    if (G.io == ZOPT_F32 && G.f32c) ZOPT_TRANSPOSE(float, float);
    else if (G.io == ZOPT_F32) ZOPT_TRANSPOSE(float, __nv_bfloat16);
    else if (G.f32c) ZOPT_TRANSPOSE(__nv_bfloat16, float);
    else ZOPT_TRANSPOSE(__nv_bfloat16, __nv_bfloat16);
#undef ZOPT_TRANSPOSE
  }
  if (st != ZOPT_OK) return st;
  ZOPT_CUDA_TRY(cudaGetLastError());
  return ok();
}

}  // namespace ns
}  // namespace zopt
