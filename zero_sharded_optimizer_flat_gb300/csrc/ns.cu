// Muon's quintic Newton-Schulz orthogonalisation on whole matrices, on tcgen05 tensor cores.
//
// bluscript_zero_ckpt.cpp, ShardedMuon design note: U = NewtonSchulz(M), the iterated matrix
// polynomial X <- aX + (bXX' + c(XX')^2)X, in which every output entry depends on the whole
// matrix (so each matrix has one owner rank); 5 steps in the trainer's config.
//
// Per step, with X m x n (m <= n; a taller input is processed as its transpose):
//   A = X X'            (symmetric: only 128x256 tiles touching the upper triangle are
//                        computed, each writes its upper part directly and its strictly upper
//                        part mirrored)
//   B' = c A A' + b A + a I
//                       (A is symmetric, so A^2 = A A': the same symmetric kernel, with the
//                        b*A term and a on the diagonal added in the epilogue)
//   X = B' X            (= aX + BX: the step's aX term rides on B's diagonal, so the largest
//                        product has no second input to read; a plain GEMM whose B-operand X
//                        is read MN-major straight from its row-major layout; the last step
//                        writes the caller's output, in the caller's orientation and dtype)
// Operands and the products A, B', X are bf16; every product accumulates in fp32 in TMEM.
//
// Products with m >= 1024 run on CTA pairs (tcgen05.mma.cta_group::2, 256 x 256 tiles, see
// gemm_bf16_pair_kernel); smaller ones on single CTAs as follows.
// One kernel does all three products: a persistent, warp-specialised tcgen05 GEMM. Warp 0
// streams 128x64 and 256x64 bf16 tiles into a shared-memory ring with TMA (128-byte swizzle);
// one thread of warp 1 issues tcgen05.mma (M=128, N=256, K=16) into one of two TMEM
// accumulators (2 x 256 fp32 columns), committing stage release and accumulator-ready events
// to mbarriers; warps 2-5 drain the other accumulator (tcgen05.ld), apply alpha*acc + beta*R
// (+ the diagonal term) and hand 32 x 32 bf16 boxes to the TMA while the next tile is being
// multiplied. Every mbarrier wait is bounded; a timeout sets an error word that the next call
// reports as ZOPT_ETIMEOUT.
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
  int* err;
};

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

// One epilogue warp's part of a tile through the TMA: its 32 TMEM lanes (rows i0 .. i0 + 31)
// x 256 columns from taddr (tile column block tj of matrix mb) become alpha * acc + beta * R +
// diag on the diagonal, handed to the TMA as 32 x 32 boxes. kSlice: R sits in the warp's eight
// slice boxes at `mine` (D is written over it) and two mirror boxes follow; otherwise `mine`
// holds four boxes, a D and a mirror box for even blocks and another pair for odd ones (an
// fp32 box takes a pair). last_par: parity of the last block whose boxes went to the TMA.
// Blocks c_begin .. c_end - 1 of the tile; with one pair of boxes (kPairs == 1) every block
// reuses the same D and mirror box.
template <bool kSlice, int kPairs = 2>
__device__ __forceinline__ void epi_tile_tma(const GemmArgs& a, const CUtensorMap* tmD, uint8_t* mine, uint32_t taddr,
                                             int i0, int tj, int mb, bool has_r, int lane, int& last_par,
                                             int c_begin = 0, int c_end = BN / 32) {
#pragma unroll 1
  for (int c = c_begin; c < c_end; ++c) {
    const int j0 = tj * BN + 32 * c;
    const int kind = block_kind(a, i0, j0);
    if (kind == 0 || kind == 4) continue;
    uint32_t v[32];
    tc::tmem_ld32(taddr + static_cast<uint32_t>(32 * c), v);
    tc::tmem_wait_ld();
    float o[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = a.alpha * __uint_as_float(v[k]);
    const int par = kPairs == 2 ? (c & 1) : 0;
    uint8_t* dbox = kSlice ? mine + c * kBox : mine + 2 * par * kBox;
    uint8_t* mbox = kSlice ? mine + (8 + par) * kBox : dbox + kBox;
    if (kSlice && has_r) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = *reinterpret_cast<const uint4*>(dbox + box_piece(lane, q));
        const uint32_t x[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          o[8 * q + 2 * h] += a.beta * __uint_as_float(x[h] << 16);
          o[8 * q + 2 * h + 1] += a.beta * __uint_as_float(x[h] & 0xFFFF0000u);
        }
      }
    }
    if (a.diag != 0.0f && j0 == i0) {
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (k == lane) o[k] += a.diag;
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
      if (a.d_trans)  // D[i, j] goes to row j, column i of the caller's matrix
        tc::tma_store_3d(tmD, dbox, i0, j0, mb);
      else
        tc::tma_store_3d(tmD, dbox, j0, i0, mb);
      if (kind == 2) tc::tma_store_3d(tmD, mbox, i0, j0, mb);
      tc::bulk_commit();
    }
    last_par = par;
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

// The single-CTA persistent GEMM with the epilogue kEpi (kEpiRegs, kEpiTmaR or kEpiTma). The TMA
// epilogues store D, and a symmetric product's mirror, through tmD (32 x 32 boxes, 64-byte
// swizzle; D a bf16 row-major matrix the TMA can address); kEpiTmaR reads R through tmR (the same
// boxes). Unused maps may be any valid map.
template <int kEpi>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmD,
                     const GemmArgs a) {
  constexpr int S = stages_of(kEpi);
  constexpr bool kTma = kEpi != kEpiRegs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * kTileA;
  uint8_t* sEpi = sB + S * kTileB;  // the TMA epilogue's boxes
  uint64_t* full = reinterpret_cast<uint64_t*>(sEpi + epi_bytes(kEpi));
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* rbar = drain + 1;  // kEpiTmaR: one R barrier per epilogue warp
  uint32_t* tslot = reinterpret_cast<uint32_t*>(rbar + 4);
  float* stage_base = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 256);
  uint8_t* ident = reinterpret_cast<uint8_t*>(full) + 256;  // kEpiTma (256-byte aligned)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (kEpi == kEpiTma && a.ident) init_identity(ident, a.h1, a.h2);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(tfull + b, 1);
      tc::mbar_init(tempty + b, 128);
    }
    tc::mbar_init(drain, 1);
    if (kEpi == kEpiTmaR)
      for (int q = 0; q < 4; ++q) tc::mbar_init(rbar + q, 1);
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmP);
    tc::prefetch_tmap(&tmQ);
    if (kEpi == kEpiTmaR) tc::prefetch_tmap(&tmR);
    if (kTma) tc::prefetch_tmap(&tmD);
  }
  if (warp == 1) {
    tc::tmem_alloc(tslot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  const int nk = (a.K + BK - 1) / BK;
  tc::pdl_launch_dependents();
  tc::pdl_wait();  // the previous product's outputs are complete and visible

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      int s = 0;
      uint32_t ph = 0;
      int armed[S];
      for (int q = 0; q < S; ++q) armed[q] = -1;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < a.num_tiles; t += gridDim.x) {
        int mb, ti, tj;
        tile_coords(a, t, mb, ti, tj);
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(empty + s, ph ^ 1u, a.err)) {
            ok = false;
            break;
          }
          tc::mbar_arrive_expect_tx(full + s, kTileA + kTileB);
          armed[s] = static_cast<int>(ph);
          tc::tma_load_3d(sA + s * kTileA, &tmP, full + s, kb * BK, ti * BM, mb);
          if (!a.b_mn_major) {
            tc::tma_load_3d(sB + s * kTileB, &tmQ, full + s, kb * BK, tj * BN, mb);
          } else {
#pragma unroll
            for (int q = 0; q < BN / 64; ++q)
              tc::tma_load_3d(sB + s * kTileB + q * kBoxMN, &tmQ, full + s, tj * BN + 64 * q, kb * BK, mb);
          }
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {  // leave no copy in flight: wait (bounded) for every stage armed last
        for (int q = 0; q < S; ++q)
          if (armed[q] >= 0) mbar_wait_drain(full + q, static_cast<uint32_t>(armed[q]));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      const uint32_t idesc = tc::idesc_bf16_f32(BM, BN, false, a.b_mn_major != 0);
      const uint32_t idesc16 = tc::idesc_bf16_f32(BM, 16, false, false);
      const bool ident_on = kEpi == kEpiTma && a.ident != 0;
      const uint64_t id_desc[2] = {tc::smem_desc(tc::smem_u32(ident), 16u, 256u, 6u),
                                   tc::smem_desc(tc::smem_u32(ident + 512), 16u, 256u, 6u)};
      int s = 0, it = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < a.num_tiles; t += gridDim.x, ++it) {
        const int b = it & 1;
        const uint32_t tph = static_cast<uint32_t>(it >> 1) & 1u;
        int mb, ti, tj;
        tile_coords(a, t, mb, ti, tj);
        if (!tc::mbar_wait(tempty + b, tph ^ 1u, a.err)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + static_cast<uint32_t>(b * BN);
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(full + s, ph, a.err)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t abase = tc::smem_u32(sA + s * kTileA);
          const uint32_t bbase = tc::smem_u32(sB + s * kTileB);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = tc::smem_desc_sw128(abase + 32u * kk, 16u, 1024u);
            const uint64_t bd = a.b_mn_major ? tc::smem_desc_sw128(bbase + 2048u * kk, kBoxMN, 1024u)
                                             : tc::smem_desc_sw128(bbase + 32u * kk, 16u, 1024u);
            tc::umma_bf16(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          const int c0 = kb * BK - tj * BN;  // accumulator column of this k-block's first k
          if (ident_on && c0 >= 0 && c0 < BN) {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = tc::smem_desc_sw128(abase + 32u * kk, 16u, 1024u);
              tc::umma_bf16(d + static_cast<uint32_t>(c0 + 16 * kk), ad, id_desc[0], idesc16, 1u);
              tc::umma_bf16(d + static_cast<uint32_t>(c0 + 16 * kk), ad, id_desc[1], idesc16, 1u);
            }
          }
          tc::umma_commit(empty + s);  // the stage is free once these MMAs have read it
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc::umma_commit(tfull + b);  // accumulator b is complete
      }
      tc::umma_commit(drain);  // no MMA may still be running when TMEM is released
      mbar_wait_drain(drain, 0);
    }
  } else if constexpr (kTma) {
    // ------------------------------------------------------- epilogue through the TMA (warps 2..5)
    const int quad = warp & 3;  // this warp may read TMEM lanes [32 quad, 32 quad + 32)
    uint8_t* mine = sEpi + quad * (epi_bytes(kEpi) / 4);
    uint64_t* rb = rbar + quad;
    const bool has_r = kEpi == kEpiTmaR && a.beta != 0.0f;
    bool rpend = false;  // (warp-uniform) R boxes of the current tile are in flight on rb
    uint32_t rph = 0;
    int last_par = -1;
    int t = blockIdx.x;
    if (has_r && t < a.num_tiles) {
      int mb, ti, tj;
      tile_coords(a, t, mb, ti, tj);
      int l = 0;
      if (lane == 0) l = epi_load_r(a, &tmR, mine, rb, mb, ti * BM + 32 * quad, tj) ? 1 : 0;
      rpend = __shfl_sync(0xFFFFFFFFu, l, 0) != 0;
    }
    for (int it = 0; t < a.num_tiles; t += gridDim.x, ++it) {
      const int b = it & 1;
      const uint32_t tph = static_cast<uint32_t>(it >> 1) & 1u;
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait(tfull + b, tph, a.err) ? 1 : 0;
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
      if (rpend) {  // every lane waits, so that each sees the TMA's writes
        if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(rb, rph, a.err) ? 1 : 0)) break;
        rph ^= 1u;
        rpend = false;
      }
      tc::fence_after_sync();
      int mb, ti, tj;
      tile_coords(a, t, mb, ti, tj);
      epi_tile_tma<kEpi == kEpiTmaR>(a, &tmD, mine,
                                     tmem + (static_cast<uint32_t>(32 * quad) << 16) + static_cast<uint32_t>(b * BN),
                                     ti * BM + 32 * quad, tj, mb, has_r, lane, last_par);
      tc::fence_before_sync();
      tc::mbar_arrive(tempty + b);  // the MMA warp may reuse this accumulator
      if (has_r) {
        // the slice is free once the TMA has read it: then prefetch the next tile's R
        if (lane == 0) tc::bulk_wait_read<0>();
        __syncwarp();
        const int tn = t + static_cast<int>(gridDim.x);
        if (tn < a.num_tiles) {
          tile_coords(a, tn, mb, ti, tj);
          int l = 0;
          if (lane == 0) l = epi_load_r(a, &tmR, mine, rb, mb, ti * BM + 32 * quad, tj) ? 1 : 0;
          rpend = __shfl_sync(0xFFFFFFFFu, l, 0) != 0;
        }
      }
    }
    if (lane == 0) {
      tc::bulk_wait_all();                  // every store has reached global memory
      if (rpend) mbar_wait_drain(rb, rph);  // (after a failed wait) no load left in flight
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2..5)
    const int quad = warp & 3;  // this warp may read TMEM lanes [32 quad, 32 quad + 32)
    const int row = 32 * quad + lane;
    int it = 0;
    for (int t = blockIdx.x; t < a.num_tiles; t += gridDim.x, ++it) {
      const int b = it & 1;
      const uint32_t tph = static_cast<uint32_t>(it >> 1) & 1u;
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait(tfull + b, tph, a.err) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc::fence_after_sync();
      int mb, ti, tj;
      tile_coords(a, t, mb, ti, tj);
      GemmArgs am = a;  // this matrix's R and D
      am.R = a.R + mb * a.r_stride;
      am.D = static_cast<uint8_t*>(a.D) + mb * a.d_stride * (a.d_f32 ? 4 : 2);
      const int i = ti * BM + row;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tc::tmem_ld32(tmem + (static_cast<uint32_t>(32 * quad) << 16) + static_cast<uint32_t>(b * BN + 32 * c), v);
        tc::tmem_wait_ld();
        if (c == BN / 32 - 1) {
          tc::fence_before_sync();
          tc::mbar_arrive(tempty + b);  // the MMA warp may reuse this accumulator
        }
        epilogue32(am, i, tj * BN + 32 * c, v, stage_base + (warp - 2) * kStageWarp, lane);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------- CTA-pair GEMM
//
// The same three products with tcgen05.mma.cta_group::2: a cluster of two CTAs on two SMs
// computes a 256 x 256 tile, each CTA holding its 128 rows of the A-operand and its 128
// columns of the B-operand, so a CTA streams 32 KiB per 64-deep k-block instead of 48 and the
// ring holds 6 stages. Both CTAs' TMA loads complete on the leader's (rank 0) stage barrier;
// the leader's single thread issues the M=256 MMAs, whose commits reach both CTAs; each CTA
// drains its own 128 TMEM lanes; the epilogue warps of both CTAs release an accumulator on the
// leader's barrier.
// The epilogues are the single-CTA kernel's: each CTA drains its own 128 rows of the tile.
// With R prefetched (kEpiTmaR) the ring keeps four stages, otherwise six.
constexpr int BM2 = 256, STAGES2 = 6;
constexpr int kHalf = 128 * BK * 2;  // 16 KiB: 128 rows (or columns) of a 64-deep k-block
__host__ __device__ constexpr int stages2_of(int e) { return e == kEpiTmaR ? 4 : STAGES2; }
constexpr int smem_bytes2(int e) {
  return stages2_of(e) * 2 * kHalf + epi_bytes(e) + 1024 + 256 + (e == kEpiRegs ? kStageBytes : 0);
}
static_assert(smem_bytes2(kEpiTma) <= 232448 && smem_bytes2(kEpiTmaR) <= 232448, "shared memory per CTA");

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

// tmR, tmD: as for the single-CTA kernel (unused by kEpiRegs).
template <int kEpi>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmD,
                          const GemmArgs a) {
  constexpr int S2 = stages2_of(kEpi);
  constexpr bool kTma = kEpi != kEpiRegs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S2 * kHalf;
  uint8_t* sEpi = sB + S2 * kHalf;  // the TMA epilogue's boxes
  uint64_t* full = reinterpret_cast<uint64_t*>(sEpi + epi_bytes(kEpi));
  uint64_t* empty = full + S2;
  uint64_t* tfull = empty + S2;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* rbar = drain + 1;  // kEpiTmaR: one R barrier per epilogue warp
  uint32_t* tslot = reinterpret_cast<uint32_t*>(rbar + 4);
  float* stage_base = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_rank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  if (threadIdx.x == 0) {
    for (int q = 0; q < S2; ++q) {
      tc::mbar_init(full + q, 1);
      tc::mbar_init(empty + q, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(tfull + b, 1);
      tc::mbar_init(tempty + b, 256);  // the epilogue threads of both CTAs (used in the leader)
    }
    tc::mbar_init(drain, 1);
    if (kEpi == kEpiTmaR)
      for (int q = 0; q < 4; ++q) tc::mbar_init(rbar + q, 1);
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmP);
    tc::prefetch_tmap(&tmQ);
    if (kEpi == kEpiTmaR) tc::prefetch_tmap(&tmR);
    if (kTma) tc::prefetch_tmap(&tmD);
  }
  if (warp == 1) {
    tc::tmem_alloc_pair(tslot, kTmemCols);
    tc::tmem_relinquish_pair();
  }
  tc::fence_before_sync();
  tc::cluster_sync();  // the peer's barriers exist before anyone arrives on them
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  const int nk = (a.K + BK - 1) / BK;
  tc::pdl_launch_dependents();
  tc::pdl_wait();  // the previous product's outputs are complete and visible

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer (both CTAs)
      int s = 0;
      uint32_t ph = 0;
      int armed[S2];
      for (int q = 0; q < S2; ++q) armed[q] = -1;
      bool ok = true;
      for (int t = pair; ok && t < a.num_tiles; t += npairs) {
        int mb, tp, tj;
        tile_coords2(a, t, mb, tp, tj);
        const int row0 = tp * BM2 + static_cast<int>(rank) * 128;  // this CTA's A rows
        const int col0 = tj * BN + static_cast<int>(rank) * 128;    // this CTA's B columns
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(empty + s, ph ^ 1u, a.err)) {
            ok = false;
            break;
          }
          if (leader) tc::mbar_arrive_expect_tx(full + s, 4 * kHalf);  // both CTAs' A and B halves
          armed[s] = static_cast<int>(ph);
          const uint32_t bar = tc::map_to_rank(tc::smem_u32(full + s), 0);
          tc::tma_load_3d_pair(sA + s * kHalf, &tmP, bar, kb * BK, row0, mb);
          if (!a.b_mn_major) {
            tc::tma_load_3d_pair(sB + s * kHalf, &tmQ, bar, kb * BK, col0, mb);
          } else {
            tc::tma_load_3d_pair(sB + s * kHalf, &tmQ, bar, col0, kb * BK, mb);
            tc::tma_load_3d_pair(sB + s * kHalf + kBoxMN, &tmQ, bar, col0 + 64, kb * BK, mb);
          }
          if (++s == S2) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok && leader) {  // the leader's stage barriers count both CTAs' copies
        for (int q = 0; q < S2; ++q)
          if (armed[q] >= 0) mbar_wait_drain(full + q, static_cast<uint32_t>(armed[q]));
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------------- MMA issuer (leader)
      const uint32_t idesc = tc::idesc_bf16_f32(BM2, BN, false, a.b_mn_major != 0);
      int s = 0, it = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = pair; ok && t < a.num_tiles; t += npairs, ++it) {
        const int b = it & 1;
        const uint32_t tph = static_cast<uint32_t>(it >> 1) & 1u;
        if (!tc::mbar_wait(tempty + b, tph ^ 1u, a.err)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + static_cast<uint32_t>(b * BN);
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(full + s, ph, a.err)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t abase = tc::smem_u32(sA + s * kHalf);
          const uint32_t bbase = tc::smem_u32(sB + s * kHalf);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = tc::smem_desc_sw128(abase + 32u * kk, 16u, 1024u);
            const uint64_t bd = a.b_mn_major ? tc::smem_desc_sw128(bbase + 2048u * kk, kBoxMN, 1024u)
                                             : tc::smem_desc_sw128(bbase + 32u * kk, 16u, 1024u);
            tc::umma_bf16_pair(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc::umma_commit_pair(empty + s, 3);  // both CTAs' stage s is free
          if (++s == S2) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc::umma_commit_pair(tfull + b, 3);  // both CTAs' accumulator b is complete
      }
      tc::umma_commit_pair(drain, 1);
      mbar_wait_drain(drain, 0);
    }
  } else if constexpr (kTma) {
    // ------------------------------------------------------- epilogue through the TMA (warps 2..5)
    const int quad = warp & 3;
    uint8_t* mine = sEpi + quad * (epi_bytes(kEpi) / 4);
    uint64_t* rb = rbar + quad;
    const bool has_r = kEpi == kEpiTmaR && a.beta != 0.0f;
    const uint32_t tempty_leader[2] = {tc::map_to_rank(tc::smem_u32(tempty), 0),
                                       tc::map_to_rank(tc::smem_u32(tempty + 1), 0)};
    const int rows0 = static_cast<int>(rank) * 128 + 32 * quad;  // this warp's rows within a tile
    bool rpend = false;  // (warp-uniform) R boxes of the current tile are in flight on rb
    uint32_t rph = 0;
    int last_par = -1;
    int t = pair;
    if (has_r && t < a.num_tiles) {
      int mb, tp, tj;
      tile_coords2(a, t, mb, tp, tj);
      int l = 0;
      if (lane == 0) l = epi_load_r(a, &tmR, mine, rb, mb, tp * BM2 + rows0, tj) ? 1 : 0;
      rpend = __shfl_sync(0xFFFFFFFFu, l, 0) != 0;
    }
    for (int it = 0; t < a.num_tiles; t += npairs, ++it) {
      const int b = it & 1;
      const uint32_t tph = static_cast<uint32_t>(it >> 1) & 1u;
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait(tfull + b, tph, a.err) ? 1 : 0;
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
      if (rpend) {  // every lane waits, so that each sees the TMA's writes
        if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(rb, rph, a.err) ? 1 : 0)) break;
        rph ^= 1u;
        rpend = false;
      }
      tc::fence_after_sync();
      int mb, tp, tj;
      tile_coords2(a, t, mb, tp, tj);
      epi_tile_tma<kEpi == kEpiTmaR>(a, &tmD, mine,
                                     tmem + (static_cast<uint32_t>(32 * quad) << 16) + static_cast<uint32_t>(b * BN),
                                     tp * BM2 + rows0, tj, mb, has_r, lane, last_par);
      tc::fence_before_sync();
      tc::mbar_arrive_cluster(tempty_leader[b]);  // the leader's MMA thread may reuse this accumulator
      if (has_r) {
        // the slice is free once the TMA has read it: then prefetch the next tile's R
        if (lane == 0) tc::bulk_wait_read<0>();
        __syncwarp();
        const int tn = t + npairs;
        if (tn < a.num_tiles) {
          tile_coords2(a, tn, mb, tp, tj);
          int l = 0;
          if (lane == 0) l = epi_load_r(a, &tmR, mine, rb, mb, tp * BM2 + rows0, tj) ? 1 : 0;
          rpend = __shfl_sync(0xFFFFFFFFu, l, 0) != 0;
        }
      }
    }
    if (lane == 0) {
      tc::bulk_wait_all();                  // every store has reached global memory
      if (rpend) mbar_wait_drain(rb, rph);  // (after a failed wait) no load left in flight
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2..5)
    const int quad = warp & 3;
    const int row = 32 * quad + lane;
    const uint32_t tempty_leader[2] = {tc::map_to_rank(tc::smem_u32(tempty), 0),
                                       tc::map_to_rank(tc::smem_u32(tempty + 1), 0)};
    int it = 0;
    for (int t = pair; t < a.num_tiles; t += npairs, ++it) {
      const int b = it & 1;
      const uint32_t tph = static_cast<uint32_t>(it >> 1) & 1u;
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait(tfull + b, tph, a.err) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc::fence_after_sync();
      int mb, tp, tj;
      tile_coords2(a, t, mb, tp, tj);
      GemmArgs am = a;
      am.R = a.R + mb * a.r_stride;
      am.D = static_cast<uint8_t*>(a.D) + mb * a.d_stride * (a.d_f32 ? 4 : 2);
      const int i = tp * BM2 + static_cast<int>(rank) * 128 + row;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tc::tmem_ld32(tmem + (static_cast<uint32_t>(32 * quad) << 16) + static_cast<uint32_t>(b * BN + 32 * c), v);
        tc::tmem_wait_ld();
        if (c == BN / 32 - 1) {
          tc::fence_before_sync();
          tc::mbar_arrive_cluster(tempty_leader[b]);
        }
        epilogue32(am, i, tj * BN + 32 * c, v, stage_base + (warp - 2) * kStageWarp, lane);
      }
    }
  }
  tc::fence_before_sync();
  tc::cluster_sync();  // every MMA, copy and remote arrival of the pair is done
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------- prep kernels

// Per-matrix reduction scratch: an arrival counter and up to kPrepBlocks fp64 partials.
constexpr int kPrepBlocks = 512;
constexpr size_t kPrepWsBytes = 256 + sizeof(double) * kPrepBlocks;

__device__ __forceinline__ NormWorkspace* prep_ws(uint8_t* base, int mb) {
  return reinterpret_cast<NormWorkspace*>(base + static_cast<size_t>(mb) * kPrepWsBytes);
}

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
constexpr int kMaxFusedJobs = 6;

struct FusedJobMaps {
  CUtensorMap xp[2], xq[2], xmn[2], xe[2];  // X (either buffer): operand boxes, epilogue boxes
  CUtensorMap ap, aq, ae, bp, be, oe;       // A, B' and the caller's X
};
struct FusedMaps {
  FusedJobMaps job[kMaxFusedJobs];
};

struct FusedJob {
  GemmArgs prod[kFusedProducts];
  uint8_t* prep;  // per-matrix prep scratch (kPrepWsBytes apart); counters at kCntWord
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

// Wait (bounded) until *c >= target; then order the caller's later TMA loads after it.
__device__ __forceinline__ bool wait_count(const uint32_t* c, uint32_t target, int* err) {
  if (ld_acquire(c) < target) {
    const unsigned long long t0 = tc::globaltimer();
    for (uint32_t spin = 1;; ++spin) {
      __nanosleep(32);
      if (ld_acquire(c) >= target) break;
      if ((spin & 15u) == 0) {
        const unsigned long long el = tc::globaltimer() - t0;
        if (el > 1000000ull && *reinterpret_cast<volatile int*>(err) != 0) return false;
        if (el > tc::kWaitLimitNs) {
          atomicExch(err, 1);
          return false;
        }
      }
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

__global__ void __launch_bounds__(kFusedThreads, 1)
    ns_fused_kernel(const __grid_constant__ FusedMaps mp, const FusedArgs f) {
  constexpr int S = STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * kTileA;
  uint8_t* sEpi = sB + S * kTileB;
  uint64_t* full = reinterpret_cast<uint64_t*>(sEpi + epi_bytes(kEpiTma));
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
  uint8_t* ident = reinterpret_cast<uint8_t*>(full) + 256;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = f.steps * f.per_step;
  init_identity(ident, f.job[0].prod[1].h1, f.job[0].prod[1].h2);  // every job has the call's b / c
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(tfull + b, 1);
      tc::mbar_init(tempty + b, 32 * kFusedEpiWarps);
    }
    tc::mbar_init(drain, 1);
    tc::fence_mbar_init();
    for (int j = 0; j < f.n_jobs; ++j) {
      const FusedJobMaps& m = mp.job[j];
      for (int q = 0; q < 2; ++q) {
        tc::prefetch_tmap(&m.xp[q]);
        tc::prefetch_tmap(&m.xq[q]);
        tc::prefetch_tmap(&m.xmn[q]);
        tc::prefetch_tmap(&m.xe[q]);
      }
      tc::prefetch_tmap(&m.ap);
      tc::prefetch_tmap(&m.aq);
      tc::prefetch_tmap(&m.ae);
      tc::prefetch_tmap(&m.bp);
      tc::prefetch_tmap(&m.be);
      tc::prefetch_tmap(&m.oe);
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(tslot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  tc::pdl_launch_dependents();
  tc::pdl_wait();  // X0 (the normalised input) is complete and visible

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      int s = 0;
      uint32_t ph = 0;
      int armed[S];
      for (int q = 0; q < S; ++q) armed[q] = -1;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        const Item it = fused_item(f, t);
        const GemmArgs& a = fused_args(f, it);
        int dep = 0;
        const uint32_t need = fused_need(f, it, dep);
        if (need > 0 && !wait_count(fused_counter(f, it.j, it.mb, dep), need, f.err)) {
          ok = false;
          break;
        }
        const int cur = it.s & 1;
        const FusedJobMaps& m = mp.job[it.j];
        const CUtensorMap* P = it.p == 0 ? &m.xp[cur] : (it.p == 1 ? &m.ap : &m.bp);
        const CUtensorMap* Q = it.p == 0 ? &m.xq[cur] : (it.p == 1 ? &m.aq : &m.xmn[cur]);
        const int nk = (a.K + BK - 1) / BK;
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(empty + s, ph ^ 1u, f.err)) {
            ok = false;
            break;
          }
          tc::mbar_arrive_expect_tx(full + s, kTileA + kTileB);
          armed[s] = static_cast<int>(ph);
          tc::tma_load_3d(sA + s * kTileA, P, full + s, kb * BK, it.ti * BM, it.mb);
          if (!a.b_mn_major) {
            tc::tma_load_3d(sB + s * kTileB, Q, full + s, kb * BK, it.tj * BN, it.mb);
          } else {
#pragma unroll
            for (int q = 0; q < BN / 64; ++q)
              tc::tma_load_3d(sB + s * kTileB + q * kBoxMN, Q, full + s, it.tj * BN + 64 * q, kb * BK, it.mb);
          }
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {  // leave no copy in flight: wait (bounded) for every stage armed last
        for (int q = 0; q < S; ++q)
          if (armed[q] >= 0) mbar_wait_drain(full + q, static_cast<uint32_t>(armed[q]));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      const uint32_t idesc_k = tc::idesc_bf16_f32(BM, BN, false, false);
      const uint32_t idesc_mn = tc::idesc_bf16_f32(BM, BN, false, true);
      const uint32_t idesc16 = tc::idesc_bf16_f32(BM, 16, false, false);
      const uint64_t id_desc[2] = {tc::smem_desc(tc::smem_u32(ident), 16u, 256u, 6u),
                                   tc::smem_desc(tc::smem_u32(ident + 512), 16u, 256u, 6u)};
      int s = 0, n = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x, ++n) {
        const Item it = fused_item(f, t);
        const GemmArgs& a = fused_args(f, it);
        const int b = n & 1;
        const uint32_t tph = static_cast<uint32_t>(n >> 1) & 1u;
        if (!tc::mbar_wait(tempty + b, tph ^ 1u, f.err)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + static_cast<uint32_t>(b * BN);
        const bool mn = a.b_mn_major != 0;
        const bool ident_on = a.ident != 0;
        const int nk = (a.K + BK - 1) / BK;
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(full + s, ph, f.err)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t abase = tc::smem_u32(sA + s * kTileA);
          const uint32_t bbase = tc::smem_u32(sB + s * kTileB);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = tc::smem_desc_sw128(abase + 32u * kk, 16u, 1024u);
            const uint64_t bd = mn ? tc::smem_desc_sw128(bbase + 2048u * kk, kBoxMN, 1024u)
                                   : tc::smem_desc_sw128(bbase + 32u * kk, 16u, 1024u);
            tc::umma_bf16(d, ad, bd, mn ? idesc_mn : idesc_k, (kb | kk) != 0 ? 1u : 0u);
          }
          const int c0 = kb * BK - it.tj * BN;
          if (ident_on && c0 >= 0 && c0 < BN) {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = tc::smem_desc_sw128(abase + 32u * kk, 16u, 1024u);
              tc::umma_bf16(d + static_cast<uint32_t>(c0 + 16 * kk), ad, id_desc[0], idesc16, 1u);
              tc::umma_bf16(d + static_cast<uint32_t>(c0 + 16 * kk), ad, id_desc[1], idesc16, 1u);
            }
          }
          tc::umma_commit(empty + s);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc::umma_commit(tfull + b);
      }
      tc::umma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ------------------------------------------------------- epilogue through the TMA (warps 2..5)
    const int quad = warp & 3;        // this warp may read TMEM lanes [32 quad, 32 quad + 32)
    const int half = (warp - 2) >> 2;  // and drains blocks [4 half, 4 half + 4) of a tile
    uint8_t* mine = sEpi + (warp - 2) * (epi_bytes(kEpiTma) / kFusedEpiWarps);
    int last_par = -1;
    int n = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++n) {
      const Item it = fused_item(f, t);
      const GemmArgs& a = fused_args(f, it);
      const int b = n & 1;
      const uint32_t tph = static_cast<uint32_t>(n >> 1) & 1u;
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait(tfull + b, tph, f.err) ? 1 : 0;
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
      tc::fence_after_sync();
      const int cur = it.s & 1;
      const FusedJobMaps& m = mp.job[it.j];
      const CUtensorMap* D = it.p == 0 ? &m.ae : (it.p == 1 ? &m.be : (it.s == f.steps - 1 ? &m.oe : &m.xe[cur ^ 1]));
      epi_tile_tma<false, 1>(a, D, mine, tmem + (static_cast<uint32_t>(32 * quad) << 16) + static_cast<uint32_t>(b * BN),
                             it.ti * BM + 32 * quad, it.tj, it.mb, false, lane, last_par, 4 * half, 4 * half + 4);
      tc::fence_before_sync();
      tc::mbar_arrive(tempty + b);  // the MMA warp may reuse this accumulator
      if (lane == 0) {
        // this warp's part of the item has landed: count it for the item's matrix and product
        tc::bulk_wait_all();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(fused_counter(f, it.j, it.mb, it.p))
                     : "memory");
      }
      __syncwarp();
    }
    if (lane == 0) tc::bulk_wait_all();
    __syncwarp();
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A 3-D bf16 (or fp32) tensor map over `group` row-major [outer][inner] matrices with `pitch`
// elements per row, `mat_bytes` apart; boxes of box_inner x box_outer x 1 under the given swizzle.
zopt_status make_map(CUtensorMap* m, const void* base, long long inner, long long outer, long long pitch,
                     long long group, long long mat_bytes, int box_inner, int box_outer,
                     CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B, bool f32 = false) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(ZOPT_ECUDA, "zopt_ns_orthogonalize: cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer),
                              static_cast<cuuint64_t>(group)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(pitch) * (f32 ? 4 : 2), static_cast<cuuint64_t>(mat_bytes)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(ZOPT_ECUDA, "zopt_ns_orthogonalize: cuTensorMapEncodeTiled failed (" + std::to_string(r) + ")");
  return ok();
}

// Error word written by timed-out kernels: mapped pinned host memory, so the next call can
// read it without synchronising the device. Shared by every kernel with bounded waits.
zopt_status error_word(int** host, int** dev) {
  static int* h = nullptr;
  static int* d = nullptr;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (h == nullptr) {
    void* p = nullptr;
    ZOPT_CUDA_TRY(cudaHostAlloc(&p, 64, cudaHostAllocMapped | cudaHostAllocPortable));
    h = static_cast<int*>(p);
    *h = 0;
    void* dp = nullptr;
    ZOPT_CUDA_TRY(cudaHostGetDevicePointer(&dp, p, 0));
    d = static_cast<int*>(dp);
  }
  *host = h;
  *dev = d;
  return ok();
}

long long round_up(long long x, long long a) { return (x + a - 1) / a * a; }

// A finite float rounded to the nearest bf16 (ties to even), as a float.
float bf16_round(float x) {
  uint32_t u;
  std::memcpy(&u, &x, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  u &= 0xFFFF0000u;
  float r;
  std::memcpy(&r, &u, 4);
  return r;
}

// Workspace: a header (per-matrix reduction scratch and stats), then one region per matrix of
// the group holding X0, X1 (m x ldx), A and B (m x lda) in the compute dtype (es bytes).
struct Plan {
  long long m, n, ldx, lda, group;
  size_t off_stats, header, off_x1, off_a, off_b, per_mat, total;
};

Plan plan(long long rows, long long cols, long long es, long long group) {
  Plan p;
  p.m = rows < cols ? rows : cols;
  p.n = rows < cols ? cols : rows;
  p.group = group;
  p.ldx = round_up(p.n, 8);
  p.lda = round_up(p.m, 8);
  p.off_stats = static_cast<size_t>(round_up(group * static_cast<long long>(kPrepWsBytes), 256));
  p.header = static_cast<size_t>(round_up(static_cast<long long>(p.off_stats) + group * 32, 1024));
  const size_t xbytes = static_cast<size_t>(round_up(p.m * p.ldx * es, 1024));
  const size_t abytes = static_cast<size_t>(round_up(p.m * p.lda * es, 1024));
  p.off_x1 = xbytes;
  p.off_a = 2 * xbytes;
  p.off_b = 2 * xbytes + abytes;
  p.per_mat = 2 * xbytes + 2 * abytes;
  p.total = p.header + static_cast<size_t>(group) * p.per_mat;
  return p;
}

// Launches `kernel` on `stream` with programmatic stream serialisation: it may start while
// the previous kernel finishes (every kernel here waits with griddepcontrol.wait before it
// touches global memory).
template <typename... KArgs, typename... Args>
zopt_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ZOPT_CUDA_TRY(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...));
  return ok();
}

// The CTA-pair kernel for products with at least 256 rows: P is read with 128-row boxes, Q
// with 128-row (K-major) or 64 x 64 (MN-major) boxes.
// The CTA-pair kernel with epilogue `epi` (maps as for launch_gemm; kEpiTmaR reads R through *R).
zopt_status launch_gemm_pair(const CUtensorMap& P, const CUtensorMap& Q, const CUtensorMap* R, const CUtensorMap* D,
                             int epi, GemmArgs a, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    ZOPT_CUDA_TRY(cudaFuncSetAttribute(gemm_bf16_pair_kernel<kEpiRegs>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_bytes2(kEpiRegs)));
    ZOPT_CUDA_TRY(cudaFuncSetAttribute(gemm_bf16_pair_kernel<kEpiTmaR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_bytes2(kEpiTmaR)));
    ZOPT_CUDA_TRY(cudaFuncSetAttribute(gemm_bf16_pair_kernel<kEpiTma>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_bytes2(kEpiTma)));
    attr_set = true;
  }
  a.tiles_m = static_cast<int>((a.M + BM2 - 1) / BM2);
  a.tiles_n = static_cast<int>((a.N + BN - 1) / BN);
  long long per = 0;
  if (a.symmetric) {
    for (int r = 0; r < a.tiles_m; ++r) per += a.tiles_n - r;
  } else {
    per = static_cast<long long>(a.tiles_m) * a.tiles_n;
  }
  const long long total = per * a.group;
  if (total < 1 || total > 0x7FFFFFFFLL) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: too many tiles");
  a.tiles_per_mat = static_cast<int>(per);
  a.num_tiles = static_cast<int>(total);
  const int sms = sm_count();
  if (sms < 2) return fail(ZOPT_ECUDA, "zopt_ns_orthogonalize: no CUDA device");
  const int pairs = a.num_tiles < sms / 2 ? a.num_tiles : sms / 2;
  const dim3 grid(static_cast<unsigned>(2 * pairs));
  if (epi == kEpiRegs)
    return launch_pdl(gemm_bf16_pair_kernel<kEpiRegs>, grid, dim3(kGemmThreads),
                      static_cast<size_t>(smem_bytes2(kEpiRegs)), stream, P, Q, P, P, a);
  if (D == nullptr || (epi == kEpiTmaR && (a.beta != 0.0f && R == nullptr)) ||
      (epi == kEpiTmaR && (a.d_f32 || a.d_trans)) || (epi == kEpiTma && a.beta != 0.0f) ||
      (a.symmetric && (a.d_f32 || a.d_trans)))
    return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: internal: TMA epilogue without its maps");
  if (epi == kEpiTmaR)
    return launch_pdl(gemm_bf16_pair_kernel<kEpiTmaR>, grid, dim3(kGemmThreads),
                      static_cast<size_t>(smem_bytes2(kEpiTmaR)), stream, P, Q, R != nullptr ? *R : P, *D, a);
  return launch_pdl(gemm_bf16_pair_kernel<kEpiTma>, grid, dim3(kGemmThreads), static_cast<size_t>(smem_bytes2(kEpiTma)),
                    stream, P, Q, P, *D, a);
}

// The single-CTA kernel's tiles of a product (128 x 256; a symmetric product only those that
// touch the upper triangle). False if the group has 2^31 tiles or more.
bool tiles_1cta(GemmArgs& a) {
  a.tiles_m = static_cast<int>((a.M + BM - 1) / BM);
  a.tiles_n = static_cast<int>((a.N + BN - 1) / BN);
  long long per = 0;
  if (a.symmetric) {
    for (int r = 0; r < a.tiles_m; ++r) per += a.tiles_n - r / 2;
  } else {
    per = static_cast<long long>(a.tiles_m) * a.tiles_n;
  }
  const long long total = per * a.group;
  if (total < 1 || total > 0x7FFFFFFFLL) return false;
  a.tiles_per_mat = static_cast<int>(per);
  a.num_tiles = static_cast<int>(total);
  return true;
}

// The single-CTA kernel with epilogue `epi`: kEpiTmaR reads R through *R, the TMA epilogues store
// D through *D (32 x 32 boxes, 64-byte swizzle).
zopt_status launch_gemm(const CUtensorMap& P, const CUtensorMap& Q, const CUtensorMap* R, const CUtensorMap* D,
                        int epi, GemmArgs a, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    ZOPT_CUDA_TRY(cudaFuncSetAttribute(gemm_bf16_kernel<kEpiRegs>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_bytes(kEpiRegs)));
    ZOPT_CUDA_TRY(cudaFuncSetAttribute(gemm_bf16_kernel<kEpiTmaR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_bytes(kEpiTmaR)));
    ZOPT_CUDA_TRY(cudaFuncSetAttribute(gemm_bf16_kernel<kEpiTma>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_bytes(kEpiTma)));
    attr_set = true;
  }
  if (!tiles_1cta(a)) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: too many tiles");
  const int sms = sm_count();
  if (sms <= 0) return fail(ZOPT_ECUDA, "zopt_ns_orthogonalize: no CUDA device");
  const int grid = a.num_tiles < sms ? a.num_tiles : sms;
  if (epi == kEpiRegs)
    return launch_pdl(gemm_bf16_kernel<kEpiRegs>, dim3(grid), dim3(kGemmThreads), static_cast<size_t>(kSmemBytes),
                      stream, P, Q, P, P, a);
  if (D == nullptr || (epi == kEpiTmaR && (a.beta != 0.0f && R == nullptr)) ||
      (epi == kEpiTmaR && (a.d_f32 || a.d_trans)) || (epi == kEpiTma && a.beta != 0.0f) ||
      (a.symmetric && (a.d_f32 || a.d_trans)))
    return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: internal: TMA epilogue without its maps");
  if (epi == kEpiTmaR)
    return launch_pdl(gemm_bf16_kernel<kEpiTmaR>, dim3(grid), dim3(kGemmThreads),
                      static_cast<size_t>(smem_bytes(kEpiTmaR)), stream, P, Q, R != nullptr ? *R : P, *D, a);
  return launch_pdl(gemm_bf16_kernel<kEpiTma>, dim3(grid), dim3(kGemmThreads), static_cast<size_t>(smem_bytes(kEpiTma)),
                    stream, P, Q, P, *D, a);
}


// One launch of the fused kernel for every step of f.n_jobs groups (see ns_fused_kernel): each
// job's prod[0..3] hold X X', B', B'X and the last step's B'X with everything but their tile
// counts.
zopt_status launch_fused(const FusedMaps& maps, FusedArgs f, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    ZOPT_CUDA_TRY(cudaFuncSetAttribute(ns_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_bytes(kEpiTma)));
    attr_set = true;
  }
  if (f.n_jobs < 1 || f.n_jobs > kMaxFusedJobs) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: internal: job count");
  long long at = 0;
  for (int p = 0; p < 3; ++p) {
    for (int j = 0; j < f.n_jobs; ++j) {
      if (p == 0)
        for (int q = 0; q < kFusedProducts; ++q)
          if (!tiles_1cta(f.job[j].prod[q])) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: too many tiles");
      if (at > 0x7FFFFFFFLL) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: too many tiles");
      f.off[p][j] = static_cast<int>(at);
      at += f.job[j].prod[p].num_tiles;
    }
    f.off[p][f.n_jobs] = static_cast<int>(at);
  }
  if (at * f.steps > 0x7FFFFFFFLL) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: too many tiles");
  f.per_step = static_cast<int>(at);
  const int sms = sm_count();
  if (sms <= 0) return fail(ZOPT_ECUDA, "zopt_ns_orthogonalize: no CUDA device");
  const long long total = at * f.steps;
  const int grid = total < sms ? static_cast<int>(total) : sms;
  return launch_pdl(ns_fused_kernel, dim3(grid), dim3(kFusedThreads), static_cast<size_t>(smem_bytes(kEpiTma)),
                    stream, maps, f);
}

// The call's coefficients: (a, b, c) and b / c split into two bf16 values for B' on single CTAs.
struct Coef {
  float a, b, c, h1, h2;
  bool id_ok;  // the identity MMAs can carry b A (c != 0, b / c representable)
};

Coef coef_of(const float* abc) {
  Coef k;
  k.a = abc[0];
  k.b = abc[1];
  k.c = abc[2];
  const double bc = k.c != 0.0f ? static_cast<double>(k.b) / static_cast<double>(k.c) : 0.0;
  k.h1 = bf16_round(static_cast<float>(bc));
  k.h2 = bf16_round(static_cast<float>(bc - static_cast<double>(k.h1)));
  k.id_ok = k.c != 0.0f && std::isfinite(bc) && std::isfinite(k.h1) && std::isfinite(k.h2) && std::fabs(bc) < 1e30;
  return k;
}

// One group of gs same-shape matrices: the caller's matrices, the workspace regions and the
// tensor maps over them.
struct Group {
  const uint8_t* g;  // the group's first input and output matrix
  uint8_t* xo;
  zopt_dtype io;
  long long rows, cols, ld_g, ld_x, bs_g, bs_x;
  int gs;
  bool f32c, transpose, pair, out_tma;
  long long es, mat_elems;
  size_t esz;
  Plan p;
  uint8_t* ws;  // prep scratch of the group (its matrices' counters live there)
  zopt_clip_stats* stats;
  uint8_t *xb[2], *A, *B;
  CUtensorMap mx_p[2], mx_q[2], mx_mn[2], mx_e[2], ma_p, ma_q, mb_p, ma_e, mb_e, mo_e;
};

// Fill the derived fields and encode the maps of a group whose workspace is at ws (plan p).
zopt_status group_init(Group& G, const Plan& p, uint8_t* ws) {
  zopt_status st = ZOPT_OK;
  G.p = p;
  G.es = G.f32c ? 4 : 2;
  G.esz = G.io == ZOPT_F32 ? 4 : 2;
  G.transpose = G.rows > G.cols;
  G.pair = p.m >= 1024;
  G.ws = ws;
  G.stats = reinterpret_cast<zopt_clip_stats*>(ws + p.off_stats);
  uint8_t* mat0 = ws + p.header;  // matrix 0's region; matrix b at + b * per_mat
  G.xb[0] = mat0;
  G.xb[1] = mat0 + p.off_x1;
  G.A = mat0 + p.off_a;
  G.B = mat0 + p.off_b;
  G.mat_elems = static_cast<long long>(p.per_mat) / G.es;
  // the last product writes the caller's X through the TMA (32 x 32 boxes, transposed for a
  // tall matrix) when the TMA can address it: 16-byte aligned rows and matrices
  const long long esz = static_cast<long long>(G.esz);
  G.out_tma = !G.f32c && (reinterpret_cast<uintptr_t>(G.xo) & 15u) == 0 && (G.ld_x * esz) % 16 == 0 &&
              (G.gs == 1 || (G.bs_x * esz) % 16 == 0);
  if (G.f32c) return ok();
  const long long mb = static_cast<long long>(p.per_mat), grp = p.group;
  for (int q = 0; q < 2; ++q) {
    if ((st = make_map(&G.mx_p[q], G.xb[q], p.n, p.m, p.ldx, grp, mb, 64, BM)) != ZOPT_OK) return st;
    if ((st = make_map(&G.mx_q[q], G.xb[q], p.n, p.m, p.ldx, grp, mb, 64, BN)) != ZOPT_OK) return st;
    if ((st = make_map(&G.mx_mn[q], G.xb[q], p.n, p.m, p.ldx, grp, mb, 64, BK)) != ZOPT_OK) return st;
    if ((st = make_map(&G.mx_e[q], G.xb[q], p.n, p.m, p.ldx, grp, mb, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B)) != ZOPT_OK)
      return st;
  }
  if ((st = make_map(&G.ma_p, G.A, p.m, p.m, p.lda, grp, mb, 64, BM)) != ZOPT_OK) return st;
  if ((st = make_map(&G.ma_q, G.A, p.m, p.m, p.lda, grp, mb, 64, BN)) != ZOPT_OK) return st;
  if ((st = make_map(&G.mb_p, G.B, p.m, p.m, p.lda, grp, mb, 64, BM)) != ZOPT_OK) return st;
  if ((st = make_map(&G.ma_e, G.A, p.m, p.m, p.lda, grp, mb, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B)) != ZOPT_OK) return st;
  if ((st = make_map(&G.mb_e, G.B, p.m, p.m, p.lda, grp, mb, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B)) != ZOPT_OK) return st;
  if (G.out_tma) {
    const long long xrows = G.transpose ? p.n : p.m, xcols = G.transpose ? p.m : p.n;  // the caller's shape
    const long long ob = (G.gs == 1 ? xrows * G.ld_x : G.bs_x) * esz;
    const bool of32 = G.io == ZOPT_F32;
    if ((st = make_map(&G.mo_e, G.xo, xcols, xrows, G.ld_x, G.gs, ob, 32, 32,
                       of32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, of32)) != ZOPT_OK)
      return st;
  }
  return ok();
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

// Whether every product of the group can run in the fused kernel.
bool group_fusable(const Group& G, const Coef& k) { return !G.f32c && !G.pair && G.out_tma && k.id_ok; }

// The group as one job of the fused kernel.
void group_job(const Group& G, const Coef& k, int* err, FusedJob& job, FusedJobMaps& m) {
  for (int q = 0; q < 2; ++q) {
    m.xp[q] = G.mx_p[q];
    m.xq[q] = G.mx_q[q];
    m.xmn[q] = G.mx_mn[q];
    m.xe[q] = G.mx_e[q];
  }
  m.ap = G.ma_p;
  m.aq = G.ma_q;
  m.ae = G.ma_e;
  m.bp = G.mb_p;
  m.be = G.mb_e;
  m.oe = G.mo_e;
  const int mm = static_cast<int>(G.p.m), n = static_cast<int>(G.p.n);
  GemmArgs g0{};
  g0.group = G.gs;
  g0.err = err;
  g0.alpha = 1.0f;
  GemmArgs& pa = job.prod[0];  // A = X X'
  pa = g0;
  pa.M = mm; pa.N = mm; pa.K = n; pa.symmetric = 1;
  GemmArgs& pb = job.prod[1];  // B' = c A A' + b A + a I (b A by identity MMAs)
  pb = g0;
  pb.M = mm; pb.N = mm; pb.K = mm; pb.symmetric = 1;
  pb.alpha = k.c; pb.diag = k.a; pb.ident = 1; pb.h1 = k.h1; pb.h2 = k.h2;
  GemmArgs& px = job.prod[2];  // X = B' X
  px = g0;
  px.M = mm; px.N = n; px.K = mm; px.b_mn_major = 1;
  job.prod[3] = px;  // the last step's, into the caller's X
  job.prod[3].d_f32 = G.io == ZOPT_F32 ? 1 : 0;
  job.prod[3].d_trans = G.transpose ? 1 : 0;
  job.prep = G.ws;
}

// The group's products one launch at a time (the fp32 mode, the CTA-pair kernel, outputs the
// TMA cannot address).
zopt_status group_products(const Group& G, const Coef& k, int steps, int* err, cudaStream_t s) {
  zopt_status st = ZOPT_OK;
  const int m = static_cast<int>(G.p.m), n = static_cast<int>(G.p.n), gs = G.gs;
  const long long mat_elems = G.mat_elems;
  const Plan& p = G.p;
  const bool pair = G.pair;
  int cur = 0;
  for (int it = 0; it < steps; ++it) {
    const bool last = it == steps - 1;
    void* xnext = last ? static_cast<void*>(G.xo) : static_cast<void*>(G.xb[cur ^ 1]);
    const long long ldnext = last ? G.ld_x : p.ldx;
    const long long dstr_next = last ? G.bs_x : mat_elems;
    const int next_f32 = last ? (G.io == ZOPT_F32 ? 1 : 0) : (G.f32c ? 1 : 0);
    const int next_trans = last && G.transpose ? 1 : 0;
    if (G.f32c) {
      float* X0 = reinterpret_cast<float*>(G.xb[cur]);
      float* Af = reinterpret_cast<float*>(G.A);
      float* Bf = reinterpret_cast<float*>(G.B);
      // A = X X'
      GemmF32Args fa{m, m, n, gs, X0, p.ldx, mat_elems, X0, p.ldx, mat_elems, 0, 1, 1.0f, 0.0f, nullptr, 0, 0,
                     Af, p.lda, mat_elems, 1, 0};
      if ((st = launch_gemm_f32(fa, s)) != ZOPT_OK) return st;
      // B = c A A' + b A
      GemmF32Args fb{m, m, m, gs, Af, p.lda, mat_elems, Af, p.lda, mat_elems, 0, 1, k.c, k.b, Af, p.lda,
                     mat_elems, Bf, p.lda, mat_elems, 1, 0};
      if ((st = launch_gemm_f32(fb, s)) != ZOPT_OK) return st;
      // X = B X + a X
      GemmF32Args fx{m, n, m, gs, Bf, p.lda, mat_elems, X0, p.ldx, mat_elems, 1, 0, 1.0f, k.a, X0, p.ldx,
                     mat_elems, xnext, ldnext, dstr_next, next_f32, next_trans};
      if ((st = launch_gemm_f32(fx, s)) != ZOPT_OK) return st;
    } else {
      GemmArgs ga{};
      ga.err = err;
      ga.group = gs;
      // A = X X'
      ga.M = m; ga.N = m; ga.K = n;
      ga.symmetric = 1; ga.b_mn_major = 0; ga.alpha = 1.0f; ga.beta = 0.0f; ga.diag = 0.0f; ga.R = nullptr;
      ga.ldr = 0; ga.r_stride = 0; ga.D = G.A; ga.ldd = p.lda; ga.d_stride = mat_elems; ga.d_f32 = 0; ga.d_trans = 0;
      if ((st = pair ? launch_gemm_pair(G.mx_p[cur], G.mx_p[cur], nullptr, &G.ma_e, kEpiTma, ga, s)
                     : launch_gemm(G.mx_p[cur], G.mx_q[cur], nullptr, &G.ma_e, kEpiTma, ga, s)) != ZOPT_OK)
        return st;
      // B' = c A A' + b A + a I: the step's a X term joins the last product as (B + a I) X.
      // On single CTAs b A rides in the accumulator as c (h1 + h2) A (identity MMAs, h1 + h2 =
      // b / c to about 2^-18), so B' needs no second input and keeps the four-stage ring.
      ga.K = m;
      ga.alpha = k.c; ga.beta = k.b; ga.diag = k.a;
      ga.R = reinterpret_cast<const __nv_bfloat16*>(G.A); ga.ldr = p.lda; ga.r_stride = mat_elems;
      ga.D = G.B; ga.ldd = p.lda; ga.d_stride = mat_elems;
      if (!pair && k.id_ok) {
        GemmArgs gi = ga;
        gi.beta = 0.0f; gi.R = nullptr; gi.ident = 1; gi.h1 = k.h1; gi.h2 = k.h2;
        st = launch_gemm(G.ma_p, G.ma_q, nullptr, &G.mb_e, kEpiTma, gi, s);
      } else {
        st = pair ? launch_gemm_pair(G.ma_p, G.ma_p, &G.ma_e, &G.mb_e, kEpiTmaR, ga, s)
                  : launch_gemm(G.ma_p, G.ma_q, &G.ma_e, &G.mb_e, kEpiTmaR, ga, s);
      }
      if (st != ZOPT_OK) return st;
      // X = B' X
      ga.M = m; ga.N = n; ga.K = m;
      ga.symmetric = 0; ga.b_mn_major = 1; ga.alpha = 1.0f; ga.beta = 0.0f; ga.diag = 0.0f;
      ga.R = nullptr; ga.ldr = 0; ga.r_stride = 0;
      ga.D = xnext; ga.ldd = ldnext; ga.d_stride = dstr_next; ga.d_f32 = next_f32; ga.d_trans = next_trans;
      const int x_epi = (!last || G.out_tma) ? kEpiTma : kEpiRegs;
      const CUtensorMap* xd = last ? &G.mo_e : &G.mx_e[cur ^ 1];
      if ((st = pair ? launch_gemm_pair(G.mb_p, G.mx_mn[cur], nullptr, xd, x_epi, ga, s)
                     : launch_gemm(G.mb_p, G.mx_mn[cur], nullptr, xd, x_epi, ga, s)) != ZOPT_OK)
        return st;
    }
    cur ^= 1;
  }
  return ok();
}

// The error word, reporting (and clearing) a timeout of an earlier call.
zopt_status take_error_word(const char* fn, int** dev) {
  int* h = nullptr;
  zopt_status st = error_word(&h, dev);
  if (st != ZOPT_OK) return st;
  if (*reinterpret_cast<volatile int*>(h) != 0) {
    *reinterpret_cast<volatile int*>(h) = 0;
    return fail(ZOPT_ETIMEOUT, std::string(fn) + ": a tensor-core kernel of an earlier call timed out on a wait");
  }
  return ok();
}

// The checks shared by both entry points for one shape's arguments.
zopt_status check_job(const char* fn, const void* G, const void* X, zopt_dtype io, long long rows, long long cols,
                      long long ld_g, long long ld_x, long long bs_g, long long bs_x, long long batch) {
  const std::string f(fn);
  if (G == nullptr || X == nullptr) return fail(ZOPT_EINVAL, f + ": NULL pointer");
  if (rows < 1 || cols < 1 || batch < 1) return fail(ZOPT_EINVAL, f + ": empty matrix or batch");
  if (rows > (1LL << 31) || cols > (1LL << 31)) return fail(ZOPT_EINVAL, f + ": dimension >= 2^31");
  if (ld_g < cols || ld_x < cols) return fail(ZOPT_EINVAL, f + ": leading dimension < cols");
  if (batch > 1 && (bs_g < rows * ld_g || bs_x < rows * ld_x))
    return fail(ZOPT_EINVAL, f + ": batch strides overlap the matrices");
  if (io != ZOPT_F32 && io != ZOPT_BF16) return fail(ZOPT_EUNSUPPORTED, f + ": input/output dtype must be fp32 or bf16");
  return ok();
}

}  // namespace ns
}  // namespace zopt

extern "C" size_t zopt_ns_workspace(int64_t rows, int64_t cols, int32_t group, zopt_dtype compute_dtype) {
  if (rows < 1 || cols < 1 || group < 1 || (compute_dtype != ZOPT_BF16 && compute_dtype != ZOPT_F32)) return 0;
  return zopt::ns::plan(rows, cols, compute_dtype == ZOPT_F32 ? 4 : 2, group).total;
}

extern "C" zopt_status zopt_ns_orthogonalize(const void* G, void* X, zopt_dtype io_dtype, int64_t rows, int64_t cols,
                                             int64_t ld_g, int64_t ld_x, int64_t batch_stride_g,
                                             int64_t batch_stride_x, int32_t batch, zopt_dtype compute_dtype,
                                             int32_t steps, const float* abc, float eps, void* d_ws,
                                             size_t ws_bytes, zopt_stream stream) {
  using namespace zopt;
  using namespace zopt::ns;
  const char* fn = "zopt_ns_orthogonalize";
  if (d_ws == nullptr || abc == nullptr) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: NULL pointer");
  zopt_status st = check_job(fn, G, X, io_dtype, rows, cols, ld_g, ld_x, batch_stride_g, batch_stride_x, batch);
  if (st != ZOPT_OK) return st;
  if (steps < 1) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: steps < 1");
  if (compute_dtype != ZOPT_BF16 && compute_dtype != ZOPT_F32)
    return fail(ZOPT_EUNSUPPORTED, "zopt_ns_orthogonalize: compute dtype must be bf16 or fp32");
  if (!std::isfinite(abc[0]) || !std::isfinite(abc[1]) || !std::isfinite(abc[2]) || !std::isfinite(eps) || eps < 0)
    return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: coefficients and eps must be finite (eps >= 0)");
  if (!aligned16(d_ws)) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: workspace is not 16-byte aligned");
  const bool f32c = compute_dtype == ZOPT_F32;
  const long long es = f32c ? 4 : 2;
  // the largest group of matrices the workspace holds, at most the batch
  long long group = 0;
  {
    const Plan one = plan(rows, cols, es, 1);
    if (ws_bytes >= one.total) {
      group = static_cast<long long>((ws_bytes - one.header) / one.per_mat);
      if (group > batch) group = batch;
      if (group > 65535) group = 65535;  // the matrix index is a grid's y coordinate
      while (group > 1 && plan(rows, cols, es, group).total > ws_bytes) --group;
    }
  }
  if (group < 1) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: workspace smaller than zopt_ns_workspace");
  const Plan p = plan(rows, cols, es, group);
  int* err_dev = nullptr;
  if ((st = take_error_word(fn, &err_dev)) != ZOPT_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int sms = sm_count();
  if (sms <= 0) return fail(ZOPT_ECUDA, "zopt_ns_orthogonalize: no CUDA device");
  const Coef k = coef_of(abc);
  const size_t esz = io_dtype == ZOPT_F32 ? 4 : 2;
  for (long long g0i = 0; g0i < batch; g0i += group) {
    Group Gr;
    Gr.g = static_cast<const uint8_t*>(G) + static_cast<size_t>(g0i) * batch_stride_g * esz;
    Gr.xo = static_cast<uint8_t*>(X) + static_cast<size_t>(g0i) * batch_stride_x * esz;
    Gr.io = io_dtype;
    Gr.rows = rows; Gr.cols = cols; Gr.ld_g = ld_g; Gr.ld_x = ld_x; Gr.bs_g = batch_stride_g; Gr.bs_x = batch_stride_x;
    Gr.gs = static_cast<int>(batch - g0i < group ? batch - g0i : group);
    Gr.f32c = f32c;
    if ((st = group_init(Gr, p, static_cast<uint8_t*>(d_ws))) != ZOPT_OK) return st;
    if ((st = group_prep(Gr, eps, sms, s)) != ZOPT_OK) return st;
    if (group_fusable(Gr, k)) {
      // every product of every step in one persistent launch
      FusedMaps fm;
      FusedArgs fa{};
      fa.n_jobs = 1;
      fa.steps = steps;
      fa.err = err_dev;
      group_job(Gr, k, err_dev, fa.job[0], fm.job[0]);
      if ((st = launch_fused(fm, fa, s)) != ZOPT_OK) return st;
    } else if ((st = group_products(Gr, k, steps, err_dev, s)) != ZOPT_OK) {
      return st;
    }
  }
  return ok();
}

static_assert(sizeof(zopt_ns_job) == 72, "zopt_ns_job layout");

extern "C" size_t zopt_ns_workspace_many(const zopt_ns_job* jobs, int32_t n_jobs) {
  if (jobs == nullptr || n_jobs < 1) return 0;
  size_t total = 0;
  for (int32_t j = 0; j < n_jobs; ++j) {
    const zopt_ns_job& b = jobs[j];
    if (b.rows < 1 || b.cols < 1 || b.batch < 1 || b.batch > 65535) return 0;
    total += static_cast<size_t>(zopt::ns::round_up(
        static_cast<long long>(zopt::ns::plan(b.rows, b.cols, 2, b.batch).total), 1024));
  }
  return total;
}

extern "C" zopt_status zopt_ns_orthogonalize_many(const zopt_ns_job* jobs, int32_t n_jobs, int32_t steps,
                                                  const float* abc, float eps, void* d_ws, size_t ws_bytes,
                                                  zopt_stream stream) {
  using namespace zopt;
  using namespace zopt::ns;
  const char* fn = "zopt_ns_orthogonalize_many";
  if (jobs == nullptr || d_ws == nullptr || abc == nullptr) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize_many: NULL pointer");
  if (n_jobs < 1) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize_many: no jobs");
  if (steps < 1) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize_many: steps < 1");
  if (!std::isfinite(abc[0]) || !std::isfinite(abc[1]) || !std::isfinite(abc[2]) || !std::isfinite(eps) || eps < 0)
    return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize_many: coefficients and eps must be finite (eps >= 0)");
  if (!aligned16(d_ws)) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize_many: workspace is not 16-byte aligned");
  zopt_status st = ZOPT_OK;
  for (int32_t j = 0; j < n_jobs; ++j) {
    const zopt_ns_job& b = jobs[j];
    if ((st = check_job(fn, b.G, b.X, static_cast<zopt_dtype>(b.io_dtype), b.rows, b.cols, b.ld_g, b.ld_x,
                        b.batch_stride_g, b.batch_stride_x, b.batch)) != ZOPT_OK)
      return st;
    if (b.batch > 65535) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize_many: a job's batch exceeds 65535");
  }
  const size_t need = zopt_ns_workspace_many(jobs, n_jobs);
  if (need == 0 || ws_bytes < need) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize_many: workspace smaller than zopt_ns_workspace_many");
  int* err_dev = nullptr;
  if ((st = take_error_word(fn, &err_dev)) != ZOPT_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int sms = sm_count();
  if (sms <= 0) return fail(ZOPT_ECUDA, "zopt_ns_orthogonalize_many: no CUDA device");
  const Coef k = coef_of(abc);
  // every job's whole batch is one group in its own slice of the workspace; all normalise first,
  // then the fusable jobs go kMaxFusedJobs to a launch and the others run product by product
  std::vector<Group> groups(static_cast<size_t>(n_jobs));
  size_t at = 0;
  for (int32_t j = 0; j < n_jobs; ++j) {
    const zopt_ns_job& b = jobs[j];
    Group& Gr = groups[static_cast<size_t>(j)];
    Gr.g = static_cast<const uint8_t*>(b.G);
    Gr.xo = static_cast<uint8_t*>(b.X);
    Gr.io = static_cast<zopt_dtype>(b.io_dtype);
    Gr.rows = b.rows; Gr.cols = b.cols; Gr.ld_g = b.ld_g; Gr.ld_x = b.ld_x;
    Gr.bs_g = b.batch_stride_g; Gr.bs_x = b.batch_stride_x;
    Gr.gs = b.batch;
    Gr.f32c = false;
    const Plan p = plan(b.rows, b.cols, 2, b.batch);
    if ((st = group_init(Gr, p, static_cast<uint8_t*>(d_ws) + at)) != ZOPT_OK) return st;
    at += static_cast<size_t>(round_up(static_cast<long long>(p.total), 1024));
    if ((st = group_prep(Gr, eps, sms, s)) != ZOPT_OK) return st;
  }
  FusedMaps fm;
  FusedArgs fa{};
  fa.steps = steps;
  fa.err = err_dev;
  for (int32_t j = 0; j <= n_jobs; ++j) {
    const bool flush = fa.n_jobs == kMaxFusedJobs || (j == n_jobs && fa.n_jobs > 0);
    if (flush) {
      if ((st = launch_fused(fm, fa, s)) != ZOPT_OK) return st;
      fa.n_jobs = 0;
    }
    if (j == n_jobs) break;
    const Group& Gr = groups[static_cast<size_t>(j)];
    if (group_fusable(Gr, k)) {
      group_job(Gr, k, err_dev, fa.job[fa.n_jobs], fm.job[fa.n_jobs]);
      ++fa.n_jobs;
    }
  }
  for (int32_t j = 0; j < n_jobs; ++j) {
    const Group& Gr = groups[static_cast<size_t>(j)];
    if (!group_fusable(Gr, k) && (st = group_products(Gr, k, steps, err_dev, s)) != ZOPT_OK) return st;
  }
  return ok();
}

namespace zopt {
namespace ns {
namespace {
// One thread waits, with the given limit, for an mbarrier phase that nothing completes: the
// bounded-wait path of the tensor-core kernels, run on purpose.
__global__ void wait_selftest_kernel(int* err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
    tc::mbar_wait_for(&bar, 0, err, limit_ns);
  }
}
}  // namespace
}  // namespace ns
}  // namespace zopt

extern "C" zopt_status zopt_selftest_wait_timeout(int64_t limit_ns, zopt_stream stream) {
  using namespace zopt;
  if (limit_ns < 1 || limit_ns > 2000000000LL)
    return fail(ZOPT_EINVAL, "zopt_selftest_wait_timeout: limit must lie in (0, 2 s]");
  int* h = nullptr;
  int* d = nullptr;
  zopt_status st = ns::error_word(&h, &d);
  if (st != ZOPT_OK) return st;
  ns::wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      d, static_cast<unsigned long long>(limit_ns));
  ZOPT_CUDA_TRY(cudaGetLastError());
  return ok();
}

extern "C" int32_t zopt_take_device_error(void) {
  int* h = nullptr;
  int* d = nullptr;
  if (zopt::ns::error_word(&h, &d) != ZOPT_OK) return -1;
  const int v = *reinterpret_cast<volatile int*>(h);
  *reinterpret_cast<volatile int*>(h) = 0;
  return v;
}
