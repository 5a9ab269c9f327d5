// Newton-Schulz preparation: the Frobenius norm of every matrix and X0 = G / (||G|| + eps) in
// the compute dtype, transposed for a tall matrix — a few launches for every matrix of every
// job of a call: the sum of squares (unless the caller supplies the partial sums); then X0 by
// scaling (an input the first step cannot read in place: fp32, or rows the TMA cannot address)
// or by transposition (a tall input); or, where the first step reads the input in place (a
// bf16 G no taller than wide, or X0 that the caller wrote unnormalised), only the scale that
// the first step's products apply, from a small launch. Every thread keeps 128 bytes of loads
// in flight, and the normalising kernels issue their first loads before they reduce the norm.
#include <algorithm>
#include <cstring>
#include <type_traits>

#include "ns_tile.cuh"

namespace zopt {
namespace ns {

// Every matrix of a list of groups (one launch for all of them): blockIdx.y is the matrix's
// index across the list, the item it belongs to found by its `first` index.
constexpr int kMaxPrepItems = 16;
constexpr int kScaleVecs = 4096;          // 8-element vectors per scaling block (16 per thread)

struct PrepItem {
  const void* g;  // the group's first input matrix; matrix b at + b * bs elements
  long long rows, cols, ld, bs;
  int flat, vec_rows;  // sum of squares: one contiguous vector; rows of 8-element accesses
  int vec;             // scaling: rows of 8-element accesses (cols % 8 == 0)
  int flat_io;         // scaling: G and X0 both contiguous (ld == ldx == cols)
  int pair;            // fp32-output transpose: 2-element accesses
  int tvec;            // bf16-output transpose: 16-byte row accesses
  int bpm;             // sum-of-squares blocks per matrix (depends on the matrix size only)
  long long chunks;    // scaling / transpose blocks per matrix
  int first;           // index of the group's first matrix in the list (blockIdx.y)
  uint8_t* ws;         // prep scratch of matrix 0 (kPrepWsBytes per matrix): partials, counters
  zopt_clip_stats* stats;
  void* x0;            // X0 of matrix 0 in the compute dtype; matrix b at + b * x_stride
  long long ldx, x_stride;
};

struct PrepList {
  PrepItem it[kMaxPrepItems];
  int n;
  double eps;
};

__device__ __forceinline__ const PrepItem& prep_item(const PrepList& L, int y) {
  int k = 0;
  while (k + 1 < L.n && y >= L.it[k + 1].first) ++k;
  return L.it[k];
}

// The sum of 256 threads' values (linear thread id tid, 8 warps) in a fixed order: butterfly
// within each warp, then over the 8 warp sums; valid in thread 0.
__device__ __forceinline__ double sum256(double v, int tid, double* smem8) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __dadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  const int warp = tid >> 5, lane = tid & 31;
  if (lane == 0) smem8[warp] = v;
  __syncthreads();
  double r = 0.0;
  if (warp == 0) {
    r = lane < 8 ? smem8[lane] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r = __dadd_rn(r, __shfl_xor_sync(0xFFFFFFFFu, r, o));
  }
  __syncthreads();
  return r;
}

// Partial sums of squares of each matrix (blockIdx.y) over its first bpm blocks: G_b is rows x
// cols with leading dimension ld, matrices bs elements apart. `flat` = the matrix is one
// contiguous, 16-byte aligned vector. Threads stride over 8-element vectors, kRound loads in
// flight per round; block x of a matrix writes partial x to its scratch.
template <typename T>
__global__ void __launch_bounds__(kNormThreads) prep_sumsq_kernel(const PrepList L) {
  constexpr int R = kRound<T>;
  __shared__ double red[8];
  tc::pdl_launch_dependents();
  tc::pdl_wait();
  const PrepItem& J = prep_item(L, blockIdx.y);
  if (static_cast<int>(blockIdx.x) >= J.bpm) return;
  const int mb = static_cast<int>(blockIdx.y) - J.first;
  const T* g = static_cast<const T*>(J.g) + mb * J.bs;
  const long long rows = J.rows, cols = J.cols, ld = J.ld;
  double acc = 0.0;
  const long long stride = static_cast<long long>(J.bpm) * blockDim.x;
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  // vector e of the matrix: flat -> g + 8e; rows of c8 vectors -> row e / c8
  const long long c8 = J.flat ? 0 : (J.vec_rows ? cols / 8 : 0);
  const long long nvec = J.flat ? rows * cols / 8 : rows * c8;
  auto at = [&](long long e) -> const T* {
    if (J.flat) return g + 8 * e;
    const long long r = e / c8;
    return g + r * ld + 8 * (e - r * c8);
  };
  long long i = tid;
  for (; i + (R - 1) * stride < nvec; i += R * stride) {
    Raw8<T> r[R];
#pragma unroll
    for (int k = 0; k < R; ++k) ld_raw8(at(i + k * stride), r[k]);
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
  for (; i < nvec; i += stride) {
    float x[8];
    load8(at(i), x);
    acc = __dadd_rn(acc, sumsq8(x));
  }
  if (J.flat) {
    const long long n = rows * cols;
    for (long long k = nvec * 8 + tid; k < n; k += stride) {
      const double d = static_cast<double>(load1(g + k));
      acc = __dadd_rn(acc, __dmul_rn(d, d));
    }
  } else {
    const long long tail = cols - 8 * c8;  // elements of each row past its vectors
    for (long long e = tid; e < rows * tail; e += stride) {
      const long long r = e / tail, c = 8 * c8 + (e - r * tail);
      const double d = static_cast<double>(load1(g + r * ld + c));
      acc = __dadd_rn(acc, __dmul_rn(d, d));
    }
  }
  const double block = sum256(acc, static_cast<int>(threadIdx.x), red);
  if (threadIdx.x == 0) prep_ws(J.ws, mb)->partials[blockIdx.x] = block;
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

// Raw element bits of T (bf16: 16, fp32: 32) and their value.
template <typename T>
using RawOf = typename std::conditional<sizeof(T) == 2, unsigned short, unsigned int>::type;
__device__ __forceinline__ float raw_f32(unsigned short b) { return __uint_as_float(static_cast<unsigned int>(b) << 16); }
__device__ __forceinline__ float raw_f32(unsigned int b) { return __uint_as_float(b); }

// 1 / (||G_b||_F + eps) of matrix mb, valid in thread 0: every block of the matrix reduces its
// bpm partials in the same order (threads stride over them, then the 256-thread tree); block 0
// also keeps the sum in the matrix's stats and zeroes the fused kernel's counters for it.
__device__ __forceinline__ float prep_inv_norm(const PrepItem& J, int mb, double eps, int tid, bool first_block,
                                               double* red) {
  const NormWorkspace* ws = prep_ws(J.ws, mb);
  double a = 0.0;
  for (int i = tid; i < J.bpm; i += 256) a = __dadd_rn(a, __ldcg(ws->partials + i));  // from L2: another kernel wrote them
  const double total = sum256(a, tid, red);
  if (first_block && tid == 0) {
    write_clip_stats(J.stats + mb, total, 0.0f);
    uint32_t* cnt = reinterpret_cast<uint32_t*>(J.ws + static_cast<size_t>(mb) * kPrepWsBytes) + kCntWord;
    cnt[0] = cnt[1] = cnt[2] = 0u;
  }
  return __double2float_rn(__ddiv_rn(1.0, __dadd_rn(__dsqrt_rn(total), eps)));
}

// A matrix already in X0, unnormalised (blockIdx.y, one block each): its norm from its partials
// (the same reduction as prep_inv_norm), kept in its stats; its fused-kernel counters zeroed;
// d = 1 / (||G_b||_F + eps) in fp64, then fp32(d) and fp32(d * d) at words kScaleWord and
// kScaleWord + 1 of its scratch header for the first step's B'X and X X' epilogues.
__global__ void __launch_bounds__(256) prep_finalize_kernel(const PrepList L) {
  __shared__ double red[8];
  tc::pdl_launch_dependents();
  tc::pdl_wait();
  const PrepItem& J = prep_item(L, blockIdx.y);
  const int mb = static_cast<int>(blockIdx.y) - J.first;
  const int tid = static_cast<int>(threadIdx.x);
  const NormWorkspace* ws = prep_ws(J.ws, mb);
  double a = 0.0;
  for (int i = tid; i < J.bpm; i += 256) a = __dadd_rn(a, __ldcg(ws->partials + i));  // from L2: another kernel wrote them
  const double total = sum256(a, tid, red);
  if (tid == 0) {
    write_clip_stats(J.stats + mb, total, 0.0f);
    uint32_t* w = reinterpret_cast<uint32_t*>(J.ws + static_cast<size_t>(mb) * kPrepWsBytes);
    w[kCntWord] = w[kCntWord + 1] = w[kCntWord + 2] = 0u;
    const double d = __ddiv_rn(1.0, __dadd_rn(__dsqrt_rn(total), L.eps));
    float* sc = reinterpret_cast<float*>(w + kScaleWord);
    sc[0] = __double2float_rn(d);
    sc[1] = __double2float_rn(__dmul_rn(d, d));
  }
}

// X0_b = G_b / (||G_b||_F + eps) in the compute dtype U, same orientation (rows <= cols),
// blockIdx.y = matrix across the list, blockIdx.x = a run of kScaleVecs 8-element vectors.
// vec: rows of G are 16-byte aligned with cols % 8 == 0, so each thread moves 8 elements per
// access, kRound loads in flight before their stores (the first round issued before the norm
// is reduced); otherwise one element at a time.
template <typename T, typename U>
__global__ void __launch_bounds__(256) prep_scale_kernel(const PrepList L) {
  constexpr int R = kRound<T>;
  __shared__ double red[8];
  __shared__ float s_inv;
  tc::pdl_launch_dependents();
  tc::pdl_wait();
  const PrepItem& J = prep_item(L, blockIdx.y);
  if (static_cast<long long>(blockIdx.x) >= J.chunks) return;
  const int mb = static_cast<int>(blockIdx.y) - J.first;
  const int tid = static_cast<int>(threadIdx.x);
  const T* g = static_cast<const T*>(J.g) + mb * J.bs;
  U* x = static_cast<U*>(J.x0) + mb * J.x_stride;
  const long long rows = J.rows, cols = J.cols, ld = J.ld, ldx = J.ldx;
  if (J.vec) {
    const long long c8 = cols / 8, nv = rows * c8;
    const long long v0 = static_cast<long long>(blockIdx.x) * kScaleVecs + tid;
    auto g_at = [&](long long e) -> long long {
      if (J.flat_io) return 8 * e;
      const long long r = e / c8;
      return r * ld + 8 * (e - r * c8);
    };
    auto x_at = [&](long long e) -> long long {
      if (J.flat_io) return 8 * e;
      const long long r = e / c8;
      return r * ldx + 8 * (e - r * c8);
    };
    Raw8<T> raw[R];
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const long long e = v0 + static_cast<long long>(k) * 256;
      if (e < nv) ld_raw8(g + g_at(e), raw[k]);
    }
    const float inv_b = prep_inv_norm(J, mb, L.eps, tid, blockIdx.x == 0, red);
    if (tid == 0) s_inv = inv_b;
    __syncthreads();
    const float inv = s_inv;
#pragma unroll 1
    for (int u0 = 0; u0 < kScaleVecs / 256; u0 += R) {
      if (u0 > 0) {
#pragma unroll
        for (int k = 0; k < R; ++k) {
          const long long e = v0 + static_cast<long long>(u0 + k) * 256;
          if (e < nv) ld_raw8(g + g_at(e), raw[k]);
        }
      }
#pragma unroll
      for (int k = 0; k < R; ++k) {
        const long long e = v0 + static_cast<long long>(u0 + k) * 256;
        if (e >= nv) continue;
        float v[8];
        unpack8(raw[k], v);
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] *= inv;
        store8(x + x_at(e), v);
      }
    }
  } else {
    const float inv_b = prep_inv_norm(J, mb, L.eps, tid, blockIdx.x == 0, red);
    if (tid == 0) s_inv = inv_b;
    __syncthreads();
    const float inv = s_inv;
    const long long n = rows * cols, e0 = static_cast<long long>(blockIdx.x) * kScaleVecs * 8;
    const long long e1 = e0 + 8LL * kScaleVecs < n ? e0 + 8LL * kScaleVecs : n;
    for (long long e = e0 + tid; e < e1; e += 256) {
      const long long r = e / cols, c = e - r * cols;
      to_out(to_f32(g[r * ld + c]) * inv, x + r * ldx + c);
    }
  }
}

// X0_b = (G_b / (||G_b||_F + eps))' in fp32 for a tall G (rows > cols): 64 x 64 tiles through
// shared memory, 32 x 8 threads, one tile per block; pair: G's rows allow 2-element accesses.
template <typename T>
__global__ void __launch_bounds__(256) prep_transpose_f32_kernel(const PrepList L) {
  __shared__ double red[8];
  __shared__ float s_inv;
  __shared__ float tile[64][65];
  tc::pdl_launch_dependents();
  tc::pdl_wait();
  const PrepItem& J = prep_item(L, blockIdx.y);
  if (static_cast<long long>(blockIdx.x) >= J.chunks) return;
  const int mb = static_cast<int>(blockIdx.y) - J.first;
  const int lin = static_cast<int>(threadIdx.x + 32 * threadIdx.y);
  const float inv_b = prep_inv_norm(J, mb, L.eps, lin, blockIdx.x == 0, red);
  if (lin == 0) s_inv = inv_b;
  __syncthreads();
  const float inv = s_inv;
  const T* g = static_cast<const T*>(J.g) + mb * J.bs;
  float* x = static_cast<float*>(J.x0) + mb * J.x_stride;
  const long long rows = J.rows, cols = J.cols, ld = J.ld, ldx = J.ldx;
  const int pair = J.pair;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const long long tiles_c = (cols + 63) / 64;
  const long long tt = blockIdx.x;
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
    const int cc = ty + 8 * k;                       // X0 row = G column c0 + cc
    const long long xr = c0 + cc, xc = r0 + 2 * tx;  // X0[c][r] = G[r][c]
    if (full) {
      store2(x + xr * ldx + xc, tile[2 * tx][cc], tile[2 * tx + 1][cc]);
    } else {
      if (xr < cols && xc < rows) to_out(tile[2 * tx][cc], x + xr * ldx + xc);
      if (xr < cols && xc + 1 < rows) to_out(tile[2 * tx + 1][cc], x + xr * ldx + xc + 1);
    }
  }
}

// X0_b = (G_b / (||G_b||_F + eps))' in bf16 for a tall G (rows > cols), one tile per block:
// 64 G rows x 32 16-byte pieces (256 bf16 or 128 fp32 columns). Each warp reads whole 512-byte
// row runs (8 loads in flight per thread, issued before the norm is reduced) into a
// row-swizzled shared tile (piece q of row r at q ^ ((r >> 3) & 7)), then each thread gathers
// 8 consecutive G rows of one G column — 16 bytes of an X0 row, a warp writing four 128-byte
// runs; both sides are bank-conflict free. The value written is bf16(float(g) * inv), as the
// scaling kernel computes it.
template <typename T>
__global__ void __launch_bounds__(256) prep_transpose_bf16_kernel(const PrepList L) {
  constexpr int VT = 16 / static_cast<int>(sizeof(T));  // elements per 16-byte piece
  constexpr int TC = 32 * VT;                             // tile columns
  using Raw = RawOf<T>;
  __shared__ double red[8];
  __shared__ float s_inv;
  __shared__ __align__(16) uint8_t tile[64 * 512];
  tc::pdl_launch_dependents();
  tc::pdl_wait();
  const PrepItem& J = prep_item(L, blockIdx.y);
  if (static_cast<long long>(blockIdx.x) >= J.chunks) return;
  const int mb = static_cast<int>(blockIdx.y) - J.first;
  const int tid = static_cast<int>(threadIdx.x), lane = tid & 31, w = tid >> 5;
  const Raw* g = static_cast<const Raw*>(J.g) + mb * J.bs;
  __nv_bfloat16* x = static_cast<__nv_bfloat16*>(J.x0) + mb * J.x_stride;
  const long long rows = J.rows, cols = J.cols, ld = J.ld, ldx = J.ldx;
  const long long tiles_c = (cols + TC - 1) / TC;
  const long long r0 = (static_cast<long long>(blockIdx.x) / tiles_c) * 64;
  const long long c0 = (static_cast<long long>(blockIdx.x) % tiles_c) * TC;
  uint4 buf[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const long long r = r0 + k * 8 + w, c = c0 + static_cast<long long>(lane) * VT;
    if (J.tvec && r < rows && c + VT <= cols) {
      buf[k] = __ldg(reinterpret_cast<const uint4*>(g + r * ld + c));
    } else {
      Raw e[VT];
#pragma unroll
      for (int i = 0; i < VT; ++i) e[i] = (r < rows && c + i < cols) ? g[r * ld + c + i] : Raw(0);
      memcpy(&buf[k], e, 16);
    }
  }
  const float inv_b = prep_inv_norm(J, mb, L.eps, tid, blockIdx.x == 0, red);
  if (tid == 0) s_inv = inv_b;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    *reinterpret_cast<uint4*>(tile + (k * 8 + w) * 512 + ((lane ^ k) << 4)) = buf[k];
  __syncthreads();
  const float inv = s_inv;
#pragma unroll
  for (int k = 0; k < VT; ++k) {
    const int v = k * 256 + tid, xl = v >> 3, seg = v & 7;  // X0 row c0 + xl, G rows seg*8 ..
    const long long xr = c0 + xl, xc = r0 + seg * 8;
    const uint8_t* col = tile + ((xl % VT) * static_cast<int>(sizeof(T)));
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int rr = seg * 8 + j;
      o[j] = raw_f32(*reinterpret_cast<const Raw*>(col + rr * 512 + (((xl / VT) ^ seg) << 4))) * inv;
    }
    if (xr >= cols) continue;
    __nv_bfloat16* dst = x + xr * ldx + xc;
    if (xc + 8 <= rows) {
      store8(dst, o);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (xc + j < rows) to_out(o[j], dst + j);
    }
  }
}

namespace {

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// Launches one list: K selects the kernel (0 sum of squares, 1 scale, 2 transpose, 3 the scale
// of an X0 that arrived unnormalised).
template <int K, typename T, typename U>
zopt_status launch_list(PrepList& L, int matrices, long long max_x, cudaStream_t s) {
  if (L.n == 0) return ok();
  const dim3 grid(static_cast<unsigned>(max_x), static_cast<unsigned>(matrices));
  zopt_status st = ZOPT_OK;
  if constexpr (K == 0) st = launch_pdl(prep_sumsq_kernel<T>, grid, dim3(kNormThreads), 0, s, L);
  else if constexpr (K == 3) st = launch_pdl(prep_finalize_kernel, grid, dim3(256), 0, s, L);
  else if constexpr (K == 1) st = launch_pdl(prep_scale_kernel<T, U>, grid, dim3(256), 0, s, L);
  else if constexpr (std::is_same<U, float>::value)
    st = launch_pdl(prep_transpose_f32_kernel<T>, grid, dim3(32, 8), 0, s, L);
  else st = launch_pdl(prep_transpose_bf16_kernel<T>, grid, dim3(256), 0, s, L);
  L.n = 0;
  return st;
}

// Builds the lists of kernel K for input dtype T and compute dtype U over the groups that take
// it, and launches them (at most kMaxPrepItems groups and 65535 matrices per launch).
template <int K, typename T, typename U>
zopt_status prep_pass(const Group* groups, int n, float eps, cudaStream_t s) {
  PrepList L{};
  L.eps = static_cast<double>(eps);
  int matrices = 0;
  long long max_x = 1;
  zopt_status st = ZOPT_OK;
  for (int q = 0; q < n; ++q) {
    const Group& G = groups[q];
    const bool t_in = (G.io == ZOPT_F32) == std::is_same<T, float>::value;
    const bool u_out = G.f32c == std::is_same<U, float>::value;
    if (!t_in || (K != 0 && !u_out) || (K == 1 && G.transpose) || (K == 2 && !G.transpose)) continue;
    if (K == 0 && G.norm_ready) continue;  // its partials are already in the scratch
    if ((K == 3) != first_scales(G) && K != 0) continue;  // X0 is in place: only its scale is wanted
    if (L.n == kMaxPrepItems || matrices + G.gs > 65535) {
      if ((st = launch_list<K, T, U>(L, matrices, max_x, s)) != ZOPT_OK) return st;
      matrices = 0;
      max_x = 1;
    }
    const size_t esz = G.esz;
    const long long rows = G.rows, cols = G.cols, ld_g = G.ld_g, bs_g = G.bs_g;
    const bool aligned = (reinterpret_cast<uintptr_t>(G.g) & 15u) == 0 && (bs_g * esz) % 16 == 0;
    const bool rows16 = aligned && (ld_g * esz) % 16 == 0;
    PrepItem& it = L.it[L.n++];
    it.g = G.g;
    it.rows = rows;
    it.cols = cols;
    it.ld = ld_g;
    it.bs = bs_g;
    it.flat = (aligned && ld_g == cols) ? 1 : 0;
    it.vec_rows = rows16 ? 1 : 0;
    it.vec = (rows16 && cols % 8 == 0) ? 1 : 0;
    it.flat_io = (it.vec && ld_g == cols && G.p.ldx == cols) ? 1 : 0;
    it.pair = ((reinterpret_cast<uintptr_t>(G.g) % (2 * esz)) == 0 && ld_g % 2 == 0 && bs_g % 2 == 0) ? 1 : 0;
    it.tvec = rows16 ? 1 : 0;
    // blocks per matrix depend on the matrix size only, so a matrix's sum (and so its result)
    // is bitwise the same whatever group or list it runs in
    const long long bpm = norm_blocks(rows * cols);
    it.bpm = static_cast<int>(bpm);
    if (K == 0) it.chunks = bpm;
    else if (K == 3) it.chunks = 1;
    else if (K == 1) it.chunks = it.vec ? ceil_div(rows * (cols / 8), kScaleVecs) : ceil_div(rows * cols, 8LL * kScaleVecs);
    else if (std::is_same<U, float>::value) it.chunks = ceil_div(rows, 64) * ceil_div(cols, 64);
    else it.chunks = ceil_div(rows, 64) * ceil_div(cols, 32LL * (16 / static_cast<long long>(sizeof(T))));
    it.chunks = std::max(1LL, it.chunks);
    if (it.chunks > 0x7FFFFFFFLL) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: matrix too large");
    it.first = matrices;
    it.ws = G.ws;
    it.stats = G.stats;
    it.x0 = G.xb[0];
    it.ldx = G.p.ldx;
    it.x_stride = G.mat_elems;
    matrices += G.gs;
    max_x = std::max(max_x, it.chunks);
  }
  return launch_list<K, T, U>(L, matrices, max_x, s);
}

}  // namespace

// X0 = G / (||G||_F + eps), oriented, for every matrix of every group: one sum-of-squares launch
// per input dtype, then one scaling and one transpose launch per input and compute dtype that
// occur, and one launch of the first step's scales (each matrix's partial sums are reduced by
// the blocks that normalise it or by its finalize block; block 0 of a matrix also zeroes its
// counters for the fused kernel).
zopt_status group_prep(const Group* groups, int n, float eps, cudaStream_t s) {
  zopt_status st = ZOPT_OK;
  if ((st = prep_pass<0, __nv_bfloat16, float>(groups, n, eps, s)) != ZOPT_OK) return st;
  if ((st = prep_pass<0, float, float>(groups, n, eps, s)) != ZOPT_OK) return st;
  if ((st = prep_pass<1, __nv_bfloat16, __nv_bfloat16>(groups, n, eps, s)) != ZOPT_OK) return st;
  if ((st = prep_pass<1, __nv_bfloat16, float>(groups, n, eps, s)) != ZOPT_OK) return st;
  if ((st = prep_pass<1, float, __nv_bfloat16>(groups, n, eps, s)) != ZOPT_OK) return st;
  if ((st = prep_pass<1, float, float>(groups, n, eps, s)) != ZOPT_OK) return st;
  if ((st = prep_pass<2, __nv_bfloat16, __nv_bfloat16>(groups, n, eps, s)) != ZOPT_OK) return st;
  if ((st = prep_pass<2, __nv_bfloat16, float>(groups, n, eps, s)) != ZOPT_OK) return st;
  if ((st = prep_pass<2, float, __nv_bfloat16>(groups, n, eps, s)) != ZOPT_OK) return st;
  if ((st = prep_pass<2, float, float>(groups, n, eps, s)) != ZOPT_OK) return st;
  if ((st = prep_pass<3, __nv_bfloat16, __nv_bfloat16>(groups, n, eps, s)) != ZOPT_OK) return st;
  ZOPT_CUDA_TRY(cudaGetLastError());
  return ok();
}

}  // namespace ns
}  // namespace zopt
