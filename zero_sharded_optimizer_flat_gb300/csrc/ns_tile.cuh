// Shared definitions of the Newton-Schulz tensor-core kernels: tile geometry, the GEMM
// arguments and tile schedules, the epilogue building blocks (registers and TMA boxes), the
// fused call's work list, and the host-side declarations the kernel files and the entry points
// share.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "internal.h"
#include "launch.cuh"
#include "norm_impl.cuh"
#include "ns_internal.h"
#include "tc.cuh"

namespace zopt {
namespace ns {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int kTileA = BM * BK * 2;          // 16 KiB
constexpr int kTileB = BN * BK * 2;          // 32 KiB
constexpr int kBoxMN = 64 * BK * 2;          // one 64 (MN) x 64 (K) box of an MN-major operand
constexpr int kGemmThreads = 192;            // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kTmemCols = 2 * BN;            // two fp32 accumulators of 128 x 256
constexpr int kStageWarp = 32 * 33;  // floats: one epilogue warp's 32 x 32 transpose tile (padded)
constexpr int kStageBytes = 4 * kStageWarp * 4;
constexpr int kSmemBytes = STAGES * (kTileA + kTileB) + 1024 + 256 + kStageBytes;

// Epilogues of the single-CTA kernel. kEpiRegs: registers and plain stores (any D). The TMA
// epilogues move D, and for a symmetric product its mirror, as 32 x 32 bf16 boxes (64-byte rows,
// 64-byte swizzle) that a warp fills from its 32 TMEM lanes and one lane hands to the TMA:
// kEpiTma (no R term) keeps the ring's four stages and cycles four boxes per warp; kEpiTmaR
// prefetches the warp's 32 x 256 slice of R into eight boxes while the tile's MMAs run, writes D
// over it in place and has two mirror boxes per warp, at the cost of a ring stage.
constexpr int kEpiRegs = 0, kEpiTmaR = 1, kEpiTma = 2;
constexpr int kBox = 32 * 32 * 2;  // 2 KiB
constexpr int kIdentBytes = 2 * 512;  // kEpiTma: two 16 x 16 bf16 identity tiles (32-byte swizzle)
__host__ __device__ constexpr int stages_of(int e) { return e == kEpiTmaR ? 3 : STAGES; }
__host__ __device__ constexpr int epi_bytes(int e) { return e == kEpiTmaR ? 4 * (8 + 2) * kBox : (e == kEpiTma ? 4 * 4 * kBox : 0); }
constexpr int smem_bytes(int e) {
  return stages_of(e) * (kTileA + kTileB) + epi_bytes(e) + 1024 + 256 + (e == kEpiRegs ? kStageBytes : 0) +
         (e == kEpiTma ? kIdentBytes : 0);
}
static_assert(smem_bytes(kEpiTmaR) <= 232448 && smem_bytes(kEpiTma) <= 232448, "shared memory per CTA");
static_assert(smem_bytes(kEpiRegs) == kSmemBytes, "register-epilogue layout");

struct GemmArgs {
  int M, N, K;
  int tiles_m, tiles_n, num_tiles;
  int group;          // matrices processed by this launch (the TMA maps' third coordinate)
  int tiles_per_mat;  // tiles of one matrix
  long long r_stride, d_stride;  // elements between consecutive matrices' R and D
  int symmetric;   // M == N and D symmetric: upper-triangle tiles only, mirrored writes
  int b_mn_major;  // the B-operand is stored [K][N] (N contiguous)
  float alpha, beta;
  const __nv_bfloat16* R;  // D += beta * R[i, j] (bf16, row-major, ldr); may be null if beta == 0
  long long ldr;
  void* D;  // bf16 or fp32
  long long ldd;
  int d_f32;
  int d_trans;  // write D[i, j] to D[j * ldd + i]
  float diag;  // added to D[i, i] (after alpha * acc + beta * R)
  // (single-CTA kernel, kEpiTma, M == N == K) the accumulator also takes (h1 + h2) * P[i, j]:
  // at the k-blocks under the tile's columns the A-operand stage meets a 16 x 16 identity
  int ident;
  float h1, h2;
  // (a Muon call's last product) statistics of the stored output: each epilogue warp writes the
  // sum of squares and the largest magnitude of its part of a tile to its slot of matrix mb
  // (st_stride slots apart; see epi_tile_tma); null when not wanted
  double* st_sum;
  unsigned* st_max;
  long long st_stride;
  // (the first step of a call whose X0 arrives unnormalised) matrix mb's alpha is multiplied by
  // amat[mb * amat_stride], the matrix's 1 / (||X0|| + eps) or its square; null otherwise
  const float* amat;
  long long amat_stride;
  int* err;
};

// Matrix mb's factor on alpha (1 unless a.amat is set); another launch wrote it.
__device__ __forceinline__ float amat_of(const GemmArgs& a, int mb) {
  return a.amat != nullptr ? __ldcg(a.amat + static_cast<long long>(mb) * a.amat_stride) : 1.0f;
}

__device__ __forceinline__ void tile_coords(const GemmArgs& a, int t, int& mb, int& ti, int& tj) {
  mb = t / a.tiles_per_mat;  // matrix-major order: the tiles running together share operands
  t -= mb * a.tiles_per_mat;
  if (!a.symmetric) {
    // column-major raster: the tiles running together share the B-operand columns, and the
    // whole A-operand (m x m) stays in L2
    ti = t % a.tiles_m;
    tj = t / a.tiles_m;
    return;
  }
  // row ti holds tiles tj = ti/2 .. tiles_n-1 (BN = 2 BM): those touching col >= row
  int r = 0;
  for (;;) {
    const int cnt = a.tiles_n - r / 2;
    if (t < cnt) {
      ti = r;
      tj = r / 2 + t;
      return;
    }
    t -= cnt;
    ++r;
  }
}

__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = tc::globaltimer();
  while (!tc::mbar_try_wait(bar, parity)) {
    if (tc::globaltimer() - t0 > tc::kWaitLimitNs) return false;
  }
  return true;
}

__device__ __forceinline__ void store1(const GemmArgs& a, long long off, float v) {
  if (a.d_f32)
    static_cast<float*>(a.D)[off] = v;
  else
    static_cast<__nv_bfloat16*>(a.D)[off] = __float2bfloat16_rn(v);
}

// 32 consecutive outputs of row i starting at column j0 (all < N), row-major.
__device__ __forceinline__ void store_row32(const GemmArgs& a, int i, int j0, const float (&o)[32]) {
  const long long off = static_cast<long long>(i) * a.ldd + j0;
  if (a.d_f32) {
    float* p = static_cast<float*>(a.D) + off;
    if ((reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        reinterpret_cast<float4*>(p)[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) p[k] = o[k];
    }
  } else {
    __nv_bfloat16* p = static_cast<__nv_bfloat16*>(a.D) + off;
    if ((reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 u;
        __nv_bfloat162 h0 = __floats2bfloat162_rn(o[8 * q + 0], o[8 * q + 1]);
        __nv_bfloat162 h1 = __floats2bfloat162_rn(o[8 * q + 2], o[8 * q + 3]);
        __nv_bfloat162 h2 = __floats2bfloat162_rn(o[8 * q + 4], o[8 * q + 5]);
        __nv_bfloat162 h3 = __floats2bfloat162_rn(o[8 * q + 6], o[8 * q + 7]);
        u.x = *reinterpret_cast<uint32_t*>(&h0);
        u.y = *reinterpret_cast<uint32_t*>(&h1);
        u.z = *reinterpret_cast<uint32_t*>(&h2);
        u.w = *reinterpret_cast<uint32_t*>(&h3);
        reinterpret_cast<uint4*>(p)[q] = u;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) p[k] = __float2bfloat16_rn(o[k]);
    }
  }
}

// Epilogue of 32 accumulator columns [j0, j0+32) of row i; the warp's 32 lanes hold rows
// i0 .. i0+31 (i0 = i - lane). `stage` is this warp's 32 x 33 fp32 shared-memory tile.
__device__ __forceinline__ void epilogue32(const GemmArgs& a, int i, int j0, const uint32_t (&v)[32], float* stage,
                                           int lane) {
  const int i0 = i - lane;
  float o[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) o[k] = a.alpha * __uint_as_float(v[k]);
  const bool full = j0 + 32 <= a.N;
  if (a.beta != 0.0f && i < a.M) {
    const __nv_bfloat16* r = a.R + static_cast<long long>(i) * a.ldr + j0;
    if (full && (reinterpret_cast<uintptr_t>(r) & 15u) == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = *reinterpret_cast<const uint4*>(r + 8 * q);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          o[8 * q + 2 * h] += a.beta * __uint_as_float(w[h] << 16);
          o[8 * q + 2 * h + 1] += a.beta * __uint_as_float(w[h] & 0xFFFF0000u);
        }
      }
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (j0 + k < a.N) o[k] += a.beta * __bfloat162float(r[k]);
    }
  }
  if (a.diag != 0.0f && i >= j0 && i < j0 + 32) {
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (j0 + k == i) o[k] += a.diag;
  }
  if (!a.symmetric) {
    if (i >= a.M) return;
    if (!a.d_trans) {
      if (full) {
        store_row32(a, i, j0, o);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (j0 + k < a.N) store1(a, static_cast<long long>(i) * a.ldd + j0 + k, o[k]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (j0 + k < a.N) store1(a, static_cast<long long>(j0 + k) * a.ldd + i, o[k]);
    }
    return;
  }
  // symmetric: upper part (j >= i) written in place, strictly upper part mirrored to (j, i)
  if (i < a.M) {
    if (full && j0 >= i) {
      store_row32(a, i, j0, o);
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int j = j0 + k;
        if (j < a.N && j >= i) store1(a, static_cast<long long>(i) * a.ldd + j, o[k]);
      }
    }
  }
  // The mirror of a whole 32 x 32 block above the diagonal goes through shared memory: lane L
  // writes row j0 + L of the transposed block as four 16-byte stores. (Warp-uniform test.)
  const bool staged = full && j0 >= i0 + 32 && i0 + 32 <= a.M && !a.d_f32 && (a.ldd & 7) == 0 &&
                      (reinterpret_cast<uintptr_t>(a.D) & 15u) == 0;
  if (staged) {
#pragma unroll
    for (int k = 0; k < 32; ++k) stage[lane * 33 + k] = o[k];
    __syncwarp();
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.D) + static_cast<long long>(j0 + lane) * a.ldd + i0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float x[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) x[t] = stage[(8 * q + t) * 33 + lane];
      __nv_bfloat162 h[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) h[t] = __floats2bfloat162_rn(x[2 * t], x[2 * t + 1]);
      reinterpret_cast<uint4*>(dst)[q] = *reinterpret_cast<const uint4*>(h);
    }
    __syncwarp();
  } else if (i < a.M) {
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const int j = j0 + k;
      if (j < a.N && j > i) store1(a, static_cast<long long>(j) * a.ldd + i, o[k]);
    }
  }
}

// ---------------------------------------------------------------------- TMA epilogue
//
// A 32 x 32 bf16 box as the TMA lays it out under the 64-byte swizzle (box 512-byte aligned):
// row r at 64 r, its 16-byte piece q (columns 8q .. 8q + 7) at piece q ^ ((r >> 1) & 3).
__device__ __forceinline__ uint32_t box_piece(int r, int q) {
  return static_cast<uint32_t>(r * 64 + ((q ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Row `lane` of the box <- the lane's 32 values, rounded to bf16.
__device__ __forceinline__ void box_put_row(uint8_t* box, int lane, const float (&o)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = bf16x2_bits(o[8 * q + 0], o[8 * q + 1]);
    u.y = bf16x2_bits(o[8 * q + 2], o[8 * q + 3]);
    u.z = bf16x2_bits(o[8 * q + 4], o[8 * q + 5]);
    u.w = bf16x2_bits(o[8 * q + 6], o[8 * q + 7]);
    *reinterpret_cast<uint4*>(box + box_piece(lane, q)) = u;
  }
}

// The warp's 32 x 32 block transposed into the box: lane L's o[k] lands at row k, column L. Lanes
// pair up so that each writes two neighbouring bf16 of one row (conflict-free).
__device__ __forceinline__ void box_put_transposed(uint8_t* box, int lane, const float (&o)[32]) {
#pragma unroll
  for (int kk = 0; kk < 16; ++kk) {
    const float other = __shfl_xor_sync(0xFFFFFFFFu, (lane & 1) ? o[2 * kk] : o[2 * kk + 1], 1);
    const uint32_t w = (lane & 1) ? bf16x2_bits(other, o[2 * kk + 1]) : bf16x2_bits(o[2 * kk], other);
    const int r = 2 * kk + (lane & 1);
    const uint32_t off = static_cast<uint32_t>(r * 64 + (((lane >> 3) ^ (kk & 3)) << 4) + (lane & 6) * 2);
    *reinterpret_cast<uint32_t*>(box + off) = w;
  }
}

// Row `lane` of a symmetric diagonal block: the lane's own values on and right of the diagonal,
// and left of it row `lane` of `tr`, the block transposed by box_put_transposed (whose column c
// holds row c's value). Written to `box`.
__device__ __forceinline__ void box_put_symmetric_row(uint8_t* box, const uint8_t* tr, int lane,
                                                      const float (&o)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 t = *reinterpret_cast<const uint4*>(tr + box_piece(lane, q));
    const uint32_t tw[4] = {t.x, t.y, t.z, t.w};
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int c = 8 * q + 2 * h;
      const uint32_t own = bf16x2_bits(o[c], o[c + 1]);
      const uint32_t lo = (c >= lane ? own : tw[h]) & 0xFFFFu;
      const uint32_t hi = (c + 1 >= lane ? own : tw[h]) & 0xFFFF0000u;
      w[h] = lo | hi;
    }
    *reinterpret_cast<uint4*>(box + box_piece(lane, q)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// A 32 x 32 fp32 box under the 128-byte swizzle (box 1024-byte aligned): row r at 128 r, its
// 16-byte piece q (columns 4q .. 4q + 3) at piece q ^ (r & 7).
__device__ __forceinline__ uint32_t box32_piece(int r, int q) {
  return static_cast<uint32_t>(r * 128 + ((q ^ (r & 7)) << 4));
}
__device__ __forceinline__ void box32_put_row(uint8_t* box, int lane, const float (&o)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    *reinterpret_cast<float4*>(box + box32_piece(lane, q)) = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
}
// Lane L's o[k] lands at row k, column L: each store of the warp fills one 128-byte row.
__device__ __forceinline__ void box32_put_transposed(uint8_t* box, int lane, const float (&o)[32]) {
#pragma unroll
  for (int k = 0; k < 32; ++k)
    *reinterpret_cast<float*>(box + box32_piece(k, lane >> 2) + (lane & 3) * 4) = o[k];
}

// Where the 32 x 32 block at rows i0, columns j0 stands: 0 out of the matrix, 1 written as is
// (not symmetric), 2 above the diagonal (written and mirrored), 3 on it (its mirror is itself),
// 4 below it (written by the mirror of the block above). i0 and j0 are multiples of 32.
__device__ __forceinline__ int block_kind(const GemmArgs& a, int i0, int j0) {
  if (i0 >= a.M || j0 >= a.N) return 0;
  if (!a.symmetric) return 1;
  return j0 > i0 ? 2 : (j0 == i0 ? 3 : 4);
}

// Lane 0 of an epilogue warp (kEpiTmaR): the R boxes that the warp reads for its rows i0 ..
// i0 + 31 of tile column block tj of matrix mb, into its slice, on bar. Returns whether any
// load was issued.
__device__ __forceinline__ bool epi_load_r(const GemmArgs& a, const CUtensorMap* tmR, uint8_t* slice, uint64_t* bar,
                                           int mb, int i0, int tj) {
  int n = 0;
  for (int c = 0; c < BN / 32; ++c) {
    const int k = block_kind(a, i0, tj * BN + 32 * c);
    n += (k != 0 && k != 4) ? 1 : 0;
  }
  if (n == 0) return false;
  tc::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n * kBox));
  for (int c = 0; c < BN / 32; ++c) {
    const int k = block_kind(a, i0, tj * BN + 32 * c);
    if (k != 0 && k != 4) tc::tma_load_3d(slice + c * kBox, tmR, bar, tj * BN + 32 * c, i0, mb);
  }
  return true;
}

// The first block c >= c of the warp's part of a tile that it writes (neither outside the matrix
// nor below the diagonal), or c_end.
__device__ __forceinline__ int next_written_block(const GemmArgs& a, int i0, int tj, int c, int c_end) {
  for (; c < c_end; ++c) {
    const int k = block_kind(a, i0, tj * BN + 32 * c);
    if (k != 0 && k != 4) break;
  }
  return c;
}

// Lane `lane`'s 32 bf16 values of R (matrix base Rm) at row i0 + lane, columns j0 .. j0 + 31,
// zero outside the M x N matrix as a TMA load would fill them: four 16-byte loads from L2 when
// the whole row piece lies inside the matrix, element by element otherwise.
__device__ __forceinline__ void load_r_piece(const GemmArgs& a, const __nv_bfloat16* Rm, int i0, int j0, int lane,
                                             uint4 (&r)[4]) {
  const int i = i0 + lane;
  const __nv_bfloat16* row = Rm + static_cast<long long>(i) * a.ldr;
  if (i < a.M && j0 + 32 <= a.N) {
    const uint4* p = reinterpret_cast<const uint4*>(row + j0);
#pragma unroll
    for (int q = 0; q < 4; ++q) r[q] = __ldg(p + q);
    return;
  }
  uint32_t w[16];
#pragma unroll
  for (int h = 0; h < 16; ++h) {
    const int c0 = j0 + 2 * h;
    const uint32_t lo = (i < a.M && c0 < a.N) ? __bfloat16_as_ushort(row[c0]) : 0u;
    const uint32_t hi = (i < a.M && c0 + 1 < a.N) ? __bfloat16_as_ushort(row[c0 + 1]) : 0u;
    w[h] = lo | (hi << 16);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) r[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
}

// Loads, into r, R's piece for the first block the warp writes in tile column block tj of
// matrix mb (kRegR epilogues prefetch it before the tile's accumulator is ready).
__device__ __forceinline__ void prefetch_r_first(const GemmArgs& a, int mb, int i0, int tj, int lane, uint4 (&r)[4]) {
  const int c = next_written_block(a, i0, tj, 0, BN / 32);
  if (c < BN / 32) load_r_piece(a, a.R + mb * a.r_stride, i0, tj * BN + 32 * c, lane, r);
}

// One epilogue warp's part of a tile through the TMA: its 32 TMEM lanes (rows i0 .. i0 + 31)
// x 256 columns from taddr (tile column block tj of matrix mb) become alpha * acc + beta * R +
// diag on the diagonal, handed to the TMA as 32 x 32 boxes. kSlice: R sits in the warp's eight
// slice boxes at `mine` (D is written over it) and two mirror boxes follow; otherwise `mine`
// holds four boxes, a D and a mirror box for even blocks and another pair for odd ones (an
// fp32 box takes a pair). kRegR: R comes through registers instead (rfirst holds the piece of
// the first block written, as prefetch_r_first loads it; each block loads the next one's while
// it is processed). last_par: parity of the last block whose boxes went to the TMA.
// Blocks c_begin .. c_end - 1 of the tile; with one pair of boxes (kPairs == 1) every block
// reuses the same D and mirror box. kStreamOut: the product is read by a later launch, not by
// this one, so its stores mark their L2 lines to be evicted first, ahead of the operands that
// this launch's other tiles still read. st_slot >= 0 (with a.st_sum set): the warp also sums the
// squares of the values it stores (as stored: bf16-rounded unless a.d_f32; fp32 pairwise over
// runs of 8, exact fp64 outside the safe range, the runs in fp64) and takes their largest
// magnitude, and writes both to slot st_slot of matrix mb (every block the warp skips adds 0).
// use_amat: alpha takes the matrix's factor amat_of(a, mb) (a persistent launch whose products
// serve every step passes false after the first step).
template <bool kSlice, int kPairs = 2, bool kRegR = false, bool kStreamOut = false>
__device__ __forceinline__ void epi_tile_tma(const GemmArgs& a, const CUtensorMap* tmD, uint8_t* mine, uint32_t taddr,
                                             int i0, int tj, int mb, bool has_r, int lane, int& last_par,
                                             int c_begin = 0, int c_end = BN / 32, const uint4* rfirst = nullptr,
                                             int st_slot = -1, bool use_amat = true) {
  const float alpha = use_amat ? a.alpha * amat_of(a, mb) : a.alpha;
  double st_acc = 0.0;
  unsigned st_mx = 0;
  uint4 rc[4];  // kRegR: R's piece for the block being processed
  const __nv_bfloat16* Rm = nullptr;
  if constexpr (kRegR) {
    if (has_r) {
      Rm = a.R + mb * a.r_stride;
#pragma unroll
      for (int q = 0; q < 4; ++q) rc[q] = rfirst[q];
    }
  }
#pragma unroll 1
  for (int c = c_begin; c < c_end; ++c) {
    const int j0 = tj * BN + 32 * c;
    const int kind = block_kind(a, i0, j0);
    if (kind == 0 || kind == 4) continue;
    uint4 rn[4];  // kRegR: the next written block's piece, loaded while this block is processed
    int cn = c_end;
    if constexpr (kRegR) {
      if (has_r) {
        cn = next_written_block(a, i0, tj, c + 1, c_end);
        if (cn < c_end) load_r_piece(a, Rm, i0, tj * BN + 32 * cn, lane, rn);
      }
    }
    uint32_t v[32];
    tc::tmem_ld32(taddr + static_cast<uint32_t>(32 * c), v);
    tc::tmem_wait_ld();
    float o[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = alpha * __uint_as_float(v[k]);
    const int par = kPairs == 2 ? (c & 1) : 0;
    uint8_t* dbox = kSlice ? mine + c * kBox : mine + 2 * par * kBox;
    uint8_t* mbox = kSlice ? mine + (8 + par) * kBox : dbox + kBox;
    if ((kSlice || kRegR) && has_r) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = kRegR ? rc[q] : *reinterpret_cast<const uint4*>(dbox + box_piece(lane, q));
        const uint32_t x[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          o[8 * q + 2 * h] += a.beta * __uint_as_float(x[h] << 16);
          o[8 * q + 2 * h + 1] += a.beta * __uint_as_float(x[h] & 0xFFFF0000u);
        }
      }
    }
    if constexpr (kRegR) {
      if (has_r && cn < c_end) {
#pragma unroll
        for (int q = 0; q < 4; ++q) rc[q] = rn[q];
      }
    }
    if (a.diag != 0.0f && j0 == i0) {
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (k == lane) o[k] += a.diag;
    }
    if (st_slot >= 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float x[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float v = o[8 * q + k];
          x[k] = a.d_f32 ? v : __bfloat162float(__float2bfloat16_rn(v));
          st_mx = max(st_mx, __float_as_uint(x[k]) & 0x7FFFFFFFu);
        }
        st_acc = __dadd_rn(st_acc, sumsq8(x));
      }
    }
    // the boxes of this parity were last handed to the TMA two blocks ago at the latest: wait
    // until it has read them (all groups but the newest, if that one is the other parity's)
    if (lane == 0) {
      if (last_par == par || last_par < 0)
        tc::bulk_wait_read<0>();
      else
        tc::bulk_wait_read<1>();
    }
    __syncwarp();
    if (!kSlice && a.d_f32) {  // (a last product into the caller's fp32 matrix) one box per pair
      if (a.d_trans)
        box32_put_transposed(dbox, lane, o);
      else
        box32_put_row(dbox, lane, o);
    } else if (a.d_trans) {
      box_put_transposed(dbox, lane, o);
    } else if (kind == 3) {
      box_put_transposed(mbox, lane, o);
      __syncwarp();
      box_put_symmetric_row(dbox, mbox, lane, o);
    } else {
      box_put_row(dbox, lane, o);
      if (kind == 2) box_put_transposed(mbox, lane, o);
    }
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      // D[i, j] goes to row j, column i of the caller's matrix when a.d_trans
      const int x0 = a.d_trans ? i0 : j0, x1 = a.d_trans ? j0 : i0;
      if constexpr (kStreamOut) {
        const uint64_t pol = tc::l2_evict_first();
        tc::tma_store_3d_hint(tmD, dbox, x0, x1, mb, pol);
        if (kind == 2) tc::tma_store_3d_hint(tmD, mbox, i0, j0, mb, pol);
      } else {
        tc::tma_store_3d(tmD, dbox, x0, x1, mb);
        if (kind == 2) tc::tma_store_3d(tmD, mbox, i0, j0, mb);
      }
      tc::bulk_commit();
    }
    last_par = par;
  }
  if (st_slot >= 0) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      st_acc = __dadd_rn(st_acc, __shfl_xor_sync(0xFFFFFFFFu, st_acc, o));
      st_mx = max(st_mx, __shfl_xor_sync(0xFFFFFFFFu, st_mx, o));
    }
    if (lane == 0) {
      a.st_sum[mb * a.st_stride + st_slot] = st_acc;
      a.st_max[mb * a.st_stride + st_slot] = st_mx;
    }
  }
}

// The two 16 x 16 identity tiles (h1, h2) of the B' product, written by the whole block: element
// (n, k) = h if n == k, as the 32-byte swizzle lays it out (row n at 32 (n % 8) + 256 (n / 8),
// its 16-byte halves swapped when bit 2 of n is set).
__device__ __forceinline__ void init_identity(uint8_t* ident, float h1, float h2) {
  for (int w = threadIdx.x; w < kIdentBytes / 4; w += blockDim.x) {
    uint32_t word = 0;
    for (int e = 0; e < 2; ++e) {
      const int byte = 4 * w + 2 * e;
      const int h = byte / 512, bt = byte % 512;
      const int n = (bt / 256) * 8 + (bt % 256) / 32;
      const int k = ((((bt % 32) / 16) ^ ((n >> 2) & 1)) * 8) + (bt % 16) / 2;
      if (n == k) word |= static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(h ? h2 : h1))) << (16 * e);
    }
    *reinterpret_cast<uint32_t*>(ident + 4 * w) = word;
  }
  tc::fence_proxy_async_smem();  // the MMAs read the tiles through the async proxy
}

// ---------------------------------------------------------------------- CTA-pair tiles

// The epilogues are the single-CTA kernel's: each CTA drains its own 128 rows of the tile, except
// that kEpiTmaR reads R from global memory (L2) into registers, a block ahead, rather than
// staging a 64 KiB slice in shared memory: every product keeps the six-stage ring.
constexpr int BM2 = 256, STAGES2 = 6;
constexpr int kHalf = 128 * BK * 2;  // 16 KiB: 128 rows (or columns) of a 64-deep k-block
__host__ __device__ constexpr int stages2_of(int) { return STAGES2; }
__host__ __device__ constexpr int epi_bytes2(int e) { return e == kEpiRegs ? 0 : 4 * 4 * kBox; }
constexpr int smem_bytes2(int e) {
  return stages2_of(e) * 2 * kHalf + epi_bytes2(e) + 1024 + 256 + (e == kEpiRegs ? kStageBytes : 0);
}
static_assert(smem_bytes2(kEpiTma) <= 232448 && smem_bytes2(kEpiTmaR) <= 232448, "shared memory per CTA");

// Products of one kind for several jobs in one CTA-pair launch (a grouped GEMM): job j's tiles
// are [start[j], start[j + 1]) of the launch's tile index, each job with its own maps and
// arguments (its own shape and batch), so the small products fill the large ones' waves.
constexpr int kMaxPairJobs = 4;
struct PairJob {
  CUtensorMap P, Q, R, D;  // R read by kEpiTmaR; D written by the TMA epilogues
  GemmArgs a;
};
struct PairBatch {
  PairJob job[kMaxPairJobs];
  int start[kMaxPairJobs + 1];
  int n;
};
static_assert(sizeof(PairBatch) <= 4096, "kernel parameters");

__device__ __forceinline__ int pair_job_of(const PairBatch& B, int t) {
  int j = 0;
  while (j + 1 < B.n && t >= B.start[j + 1]) ++j;
  return j;
}

__device__ __forceinline__ void tile_coords2(const GemmArgs& a, int t, int& mb, int& tp, int& tj) {
  mb = t / a.tiles_per_mat;
  t -= mb * a.tiles_per_mat;
  if (!a.symmetric) {
    tp = t % a.tiles_m;
    tj = t / a.tiles_m;
    return;
  }
  int r = 0;  // 256 x 256 tiles: row r holds tiles tj = r .. tiles_n - 1
  for (;;) {
    const int cnt = a.tiles_n - r;
    if (t < cnt) {
      tp = r;
      tj = r + t;
      return;
    }
    t -= cnt;
    ++r;
  }
}

// ---------------------------------------------------------------------- prep scratch

// Per-matrix reduction scratch: an arrival counter and up to kPrepBlocks fp64 partials.
constexpr int kPrepBlocks = kNormPartialsMax;
constexpr long long kSumsqElems = 32768;  // elements per sum-of-squares block (before the cap)
constexpr size_t kPrepWsBytes = 256 + sizeof(double) * kPrepBlocks;

__device__ __forceinline__ NormWorkspace* prep_ws(uint8_t* base, int mb) {
  return reinterpret_cast<NormWorkspace*>(base + static_cast<size_t>(mb) * kPrepWsBytes);
}

// ---------------------------------------------------------------------- fused call
//
// Below the pair threshold every product of every step of a call (and of up to kMaxFusedJobs
// jobs of different shapes) can run in one persistent launch of the single-CTA machinery
// (four-stage ring, TMA epilogue, B' by identity MMAs). Its work list is step-major, then
// product (X X', B', B'X), then job, then matrix, then tile; CTA c takes items c, c + G, c + 2G,
// ... Before loading an item, the TMA thread waits until the product the item reads is complete
// for its matrix: each epilogue warp adds one to its matrix's counter for that product once its
// stores of an item have landed (release), and the waiter's acquire load is followed by a proxy
// fence before its TMA loads. Between an item and its input lie the items of the other jobs, so
// one job's waits are filled by another's tiles. An item depends only on earlier items and
// every CTA is resident (one per SM, a grid no larger than the SM count), so the list always
// progresses; each wait is bounded like the barrier waits.
constexpr int kFusedProducts = 4;  // X X', B', B'X, and B'X of the last step (the caller's X)
// warp 0 TMA, warp 1 MMA, warps 2..9 epilogue: two warps per TMEM lane quadrant, each draining
// half of a tile's 32-column blocks through one D and one mirror box
constexpr int kFusedEpiWarps = 8;
constexpr int kFusedThreads = 32 * (2 + kFusedEpiWarps);
constexpr int kCntWord = 16;       // counters at word 16 of each matrix's prep scratch header
// (X0 that arrives unnormalised) 1 / (||X0|| + eps) and its square, fp32, at words 24 and 25
constexpr int kScaleWord = 24;
constexpr int kMaxFusedJobs = 6;

struct FusedJobMaps {
  CUtensorMap xp[2], xq[2], xmn[2], xe[2];  // X (either buffer): operand boxes, epilogue boxes
  CUtensorMap ap, aq, ae, bp, be, oe;       // A, B' and the caller's X
  CUtensorMap gp, gq, gmn;                  // the caller's G as the first step's X (g_in_place)
};
struct FusedMaps {
  FusedJobMaps job[kMaxFusedJobs];
};

struct FusedJob {
  GemmArgs prod[kFusedProducts];
  uint8_t* prep;  // per-matrix prep scratch (kPrepWsBytes apart); counters at kCntWord
  int x0_is_g;    // the first step reads the caller's G in place (maps gp, gq, gmn)
};

struct FusedArgs {
  FusedJob job[kMaxFusedJobs];
  int n_jobs;
  int steps;
  int per_step;                   // items of one step (all products, jobs, matrices)
  int off[3][kMaxFusedJobs + 1];  // within a step, product p's items of job j start at off[p][j]
  int* err;
};

static_assert(sizeof(FusedMaps) + sizeof(FusedArgs) <= 32000, "the fused kernel's parameters fit a launch");

struct Item {
  int s, p, j, mb, ti, tj;
};

__device__ __forceinline__ Item fused_item(const FusedArgs& f, int t) {
  Item it;
  it.s = t / f.per_step;
  const int r = t - it.s * f.per_step;
  it.p = r < f.off[0][f.n_jobs] ? 0 : (r < f.off[1][f.n_jobs] ? 1 : 2);
  it.j = 0;
  while (it.j + 1 < f.n_jobs && r >= f.off[it.p][it.j + 1]) ++it.j;
  tile_coords(f.job[it.j].prod[it.p], r - f.off[it.p][it.j], it.mb, it.ti, it.tj);
  return it;
}

__device__ __forceinline__ const GemmArgs& fused_args(const FusedArgs& f, const Item& it) {
  return f.job[it.j].prod[it.p == 2 && it.s == f.steps - 1 ? 3 : it.p];
}

__device__ __forceinline__ uint32_t* fused_counter(const FusedArgs& f, int j, int mb, int p) {
  return reinterpret_cast<uint32_t*>(f.job[j].prep + static_cast<size_t>(mb) * kPrepWsBytes) + kCntWord + p;
}

// The count the item's input product must reach for its matrix (0: nothing to wait for). Each
// item of a product is counted once by each epilogue warp of its CTA.
__device__ __forceinline__ uint32_t fused_need(const FusedArgs& f, const Item& it, int& dep) {
  if (it.p == 0) {  // X X' of step s reads the X that step s - 1 wrote
    dep = 2;
    return static_cast<uint32_t>(kFusedEpiWarps * it.s * f.job[it.j].prod[2].tiles_per_mat);
  }
  dep = it.p - 1;  // B' reads A, B'X reads B' (and X, complete before A started)
  return static_cast<uint32_t>(kFusedEpiWarps * (it.s + 1) * f.job[it.j].prod[dep].tiles_per_mat);
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Wait (bounded by limit_ns) until *c >= target; then order the caller's later TMA loads after
// it. Gives up like tc::mbar_wait_for: after another thread has reported an error, or at the
// limit, recording error code 1.
__device__ __forceinline__ bool wait_count(const uint32_t* c, uint32_t target, int* err,
                                           unsigned long long limit_ns = tc::kWaitLimitNs) {
  if (ld_acquire(c) < target) {
    const unsigned long long t0 = tc::globaltimer();
    for (uint32_t spin = 1;; ++spin) {
      __nanosleep(32);
      if (ld_acquire(c) >= target) break;
      if ((spin & 15u) == 0) {
        const unsigned long long el = tc::globaltimer() - t0;
        if (el > 1000000ull && *reinterpret_cast<volatile int*>(err) != 0) return false;
        if (el > limit_ns) {
          atomicExch(err, 1);
          return false;
        }
      }
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// ---------------------------------------------------------------------- host-side declarations

// Workspace: a header (per-matrix reduction scratch and stats), then one region per matrix of
// the group holding X0, X1 (m x ldx), A and B (m x lda) in the compute dtype (es bytes).
struct Plan {
  long long m, n, ldx, lda, group;
  size_t off_stats, header, off_x1, off_a, off_b, per_mat, total;
};

Plan plan(long long rows, long long cols, long long es, long long group);
long long round_up(long long x, long long a);
// Tile counts of a single-CTA product (fills tiles_m, tiles_n, tiles_per_mat, num_tiles).
bool tiles_1cta(GemmArgs& a);
// The single-CTA kernel with epilogue `epi` (tensor maps P, Q for the operands; R, D for the
// TMA epilogues).
zopt_status launch_gemm(const CUtensorMap& P, const CUtensorMap& Q, const CUtensorMap* R, const CUtensorMap* D,
                        int epi, GemmArgs a, cudaStream_t stream);
// The CTA-pair kernel over the n jobs of B (each job's maps and arguments filled in; the tile
// counts and starts are set here), all with epilogue `epi`.
zopt_status launch_gemm_pair_batch(PairBatch& B, int epi, cudaStream_t stream);
// The fused kernel over f.n_jobs jobs.
zopt_status launch_fused(const FusedMaps& maps, FusedArgs f, cudaStream_t stream);

// One group of gs same-shape matrices: the caller's matrices, the workspace regions and the
// tensor maps over them.
struct Group {
  const uint8_t* g;  // the group's first input and output matrix
  uint8_t* xo;
  zopt_dtype io;      // the input's dtype
  zopt_dtype out_io;  // the output's dtype
  bool norm_ready;    // the matrices' norm partials are already in the prep scratch
  bool x0_raw;        // the matrices are already in X0, unnormalised (bf16; norm_ready too)
  bool g_in_place;    // the first step reads the caller's G itself as X0 (maps mg_*), unnormalised
  long long rows, cols, ld_g, ld_x, bs_g, bs_x;
  int gs;
  bool f32c, transpose, pair, out_tma;
  long long es, mat_elems;
  size_t esz, osz;  // input and output element sizes
  Plan p;
  uint8_t* ws;  // prep scratch of the group (its matrices' counters live there)
  zopt_clip_stats* stats;
  uint8_t *xb[2], *A, *B;
  CUtensorMap mx_p[2], mx_q[2], mx_mn[2], mx_e[2], ma_p, ma_q, mb_p, ma_e, mb_e, mo_e;
  CUtensorMap mg_p, mg_q, mg_mn;  // g_in_place: G with the boxes of mx_p, mx_q, mx_mn
};

// Whether the group's first step normalises its X0 (X0 unnormalised in the workspace, or the
// caller's G read in place): its X X' and B'X epilogues apply 1 / (||X0|| + eps), squared for
// X X', which the prep scratch holds.
inline bool first_scales(const Group& G) { return G.x0_raw || G.g_in_place; }

// X0 = G / (||G||_F + eps), oriented, for every matrix of n groups, or the scale with which the
// first step normalises an X0 it reads in place (a handful of launches in all).
zopt_status group_prep(const Group* groups, int n, float eps, cudaStream_t s);


}  // namespace ns
}  // namespace zopt
