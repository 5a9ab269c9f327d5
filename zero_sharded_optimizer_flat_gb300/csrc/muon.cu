// Muon's update around Newton-Schulz, for the matrices a rank owns whole.
//
// bluscript_zero_ckpt.cpp, ShardedMuon: each matrix has one owner rank holding its fp32 master
// and momentum; momentum 0.95 with Nesterov, decoupled weight decay, U = NewtonSchulz(u);
// adjust_lr "match_rms_adamw" lifts the update's RMS to 0.2 (scale 0.2*sqrt(max(rows, cols)))
// and "original" uses sqrt(max(1, rows/cols)); diagnostics nsratio = ||U||_F/sqrt(min(rows,
// cols)) and a divergence guard that rejects an update with an element above 1000.
//
// Four steps on the caller's stream, each one launch for every job of a call (for a single
// shape: per group of matrices, as many as the workspace holds):
//   1. momentum:  buf = mu*buf + g;  u = g + mu*buf (Nesterov) or buf      (fp32, 12-14 B/elem);
//      u leaves rounded to bf16 (the dtype Newton-Schulz computes in), straight into
//      Newton-Schulz's input buffer where the shape allows (not tall, cols a multiple of 8),
//      and each block sums its share of the bf16 u^2 into the Newton-Schulz norm's partial
//      sums, so no pass reads u a second time
//   2. U = NewtonSchulz(u): bf16 u in, bf16 tensor cores, U written in bf16 (the bf16 method
//      rounds every product, its last one included, to bf16); the first step's products apply
//      the normalisation of an input written in place, and the last product's epilogue writes
//      U's per-warp sums of squares and largest magnitudes
//   3. only for a job whose last product ran elsewhere: those statistics from a pass over U
//      (2 B/elem)
//   4. p = p*fp32(1 - lr*wd) - fp32(lr*scale)*U unless rejected; bf16 round-out (12 B/elem);
//      each block first reduces its matrix's statistics slots in a fixed order (no atomics,
//      no memset)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <memory>
#include <string>
#include <vector>

#include "internal.h"
#include "norm_impl.cuh"
#include "ns_internal.h"

namespace zopt {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxBlocksPerMat = 512;
static_assert(kMaxBlocksPerMat >= ns::kNormPartialsMax, "a matrix's statistics blocks are its norm blocks");
constexpr int kMaxItems = 8;         // jobs per element-wise launch
constexpr long long kMaxCallElems = 1LL << 46;  // elements of one shape's batch

long long round_up(long long x, long long a) { return (x + a - 1) / a * a; }

// Statistics slots per matrix: one fp64 partial sum of squares and one max |U| bit pattern each,
// written by the statistics pass (a block each) or by the epilogue of Newton-Schulz's last
// product (an epilogue warp's part of a tile each).
long long red_cap(long long rows, long long cols) {
  const long long b = ns::stats_slots_bound(rows, cols);
  return b > kMaxBlocksPerMat ? b : kMaxBlocksPerMat;
}

struct MuonPlan {
  size_t off_u, off_o, off_ns, ns_bytes, total;
};

// Workspace of `group` matrices: the reduction area (the group's red_cap partial sums per matrix,
// then as many maxima), u and U (both bf16), then the Newton-Schulz workspace.
MuonPlan muon_plan(long long rows, long long cols, long long group) {
  MuonPlan p;
  const long long n = rows * cols;
  p.off_u = static_cast<size_t>(round_up(group * red_cap(rows, cols) * 12, 1024));
  p.off_o = p.off_u + static_cast<size_t>(round_up(group * n * 2, 1024));
  p.off_ns = p.off_o + static_cast<size_t>(round_up(group * n * 2, 1024));
  p.ns_bytes = static_cast<size_t>(
      round_up(static_cast<long long>(zopt_ns_workspace(rows, cols, static_cast<int32_t>(group), ZOPT_BF16)), 1024));
  p.total = p.off_ns + p.ns_bytes;
  return p;
}

// One job of an element-wise launch: `batch` matrices of n elements, back to back.
struct MuonItem {
  float* master;
  float* momentum;
  const void* grad;
  uint16_t* u_in;           // momentum's output in bf16, Newton-Schulz's input; matrix b at + b * u_stride
  long long u_stride;
  const uint16_t* u_out;    // Newton-Schulz's output U (bf16)
  double* npart;            // the Newton-Schulz norm partials of matrix 0; matrix b's at + b * npart_stride
  long long npart_stride;
  uint16_t* out;        // bf16 round-out (may be null)
  zopt_muon_stats* stats;
  double* rsum;         // matrix b's statistics slots: sums at rsum + b * rcap, maxima at rmax + b * rcap
  unsigned* rmax;
  long long rcap;
  int nred;             // slots of each matrix the update reduces (bpm, or the Newton-Schulz epilogue's)
  int ns_stats;         // the Newton-Schulz epilogue wrote the slots: no statistics pass
  long long n;          // elements per matrix
  long long u0;         // blocks of the launch before this job
  int batch;
  int bpm;              // blocks per matrix of every pass (the norm's partial count: depends on n only)
  int out8;             // the bf16 output allows 8-byte stores
  float decay, step, sqrt_min;
};

struct MuonList {
  MuonItem it[kMaxItems];
  int n;
  float mu;
  int nesterov;
  float guard;
};

__device__ __forceinline__ int item_of(const MuonList& L, long long u) {
  int k = 0;
  while (k + 1 < L.n && u >= L.it[k + 1].u0) ++k;
  return k;
}

__device__ __forceinline__ float4 fma4_momentum(float mu, const float4& b, const float4& g) {
  return make_float4(__fadd_rn(__fmul_rn(mu, b.x), g.x), __fadd_rn(__fmul_rn(mu, b.y), g.y),
                     __fadd_rn(__fmul_rn(mu, b.z), g.z), __fadd_rn(__fmul_rn(mu, b.w), g.w));
}

__device__ __forceinline__ float bf16r(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
__device__ __forceinline__ float4 bf16r4(const float4& x) {
  return make_float4(bf16r(x.x), bf16r(x.y), bf16r(x.z), bf16r(x.w));
}
// Four bf16-exact floats as 4 bf16 (their high halves).
__device__ __forceinline__ uint2 pack_bf16x4(const float4& r) {
  return make_uint2((__float_as_uint(r.x) >> 16) | (__float_as_uint(r.y) & 0xFFFF0000u),
                    (__float_as_uint(r.z) >> 16) | (__float_as_uint(r.w) & 0xFFFF0000u));
}

// Step 1: block u takes part c = (u - u0) % bpm of matrix mb = (u - u0) / bpm of its job; threads
// stride over the matrix's 4-element vectors with stride bpm * 256, four vectors' loads in flight
// per round; the matrix's n % 4 last elements go to part 0 element by element. u goes out rounded
// to bf16, the dtype Newton-Schulz computes in (where the job allows, straight into its X0). The block's sum of squares of those bf16 values
// (fp32 pairwise over runs of 8, exact fp64 outside the safe range, the runs in fp64) is the
// matrix's norm partial c, which the Newton-Schulz normalisation reads in place of a pass over u.
template <typename T>
__global__ void __launch_bounds__(kThreads) momentum_kernel(const MuonList L) {
  __shared__ double red[32];
  const MuonItem& J = L.it[item_of(L, blockIdx.x)];
  const long long v = static_cast<long long>(blockIdx.x) - J.u0;
  const long long mb = v / J.bpm, c = v - mb * J.bpm;
  const long long n = J.n;
  const T* g = static_cast<const T*>(J.grad) + mb * n;
  float* buf = J.momentum + mb * n;
  uint16_t* u = J.u_in + mb * J.u_stride;
  float4* b4 = reinterpret_cast<float4*>(buf);
  uint2* u4 = reinterpret_cast<uint2*>(u);
  const float mu = L.mu;
  const int64_t n4 = n / 4;
  const int64_t stride = static_cast<int64_t>(J.bpm) * blockDim.x;
  double acc = 0.0;
  int64_t j = c * blockDim.x + threadIdx.x;
  for (; j + 3 * stride < n4; j += 4 * stride) {  // four vectors' loads in flight before any store
    float4 gv[4], bv[4], uv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      gv[k] = load4(g + 4 * (j + k * stride));
      bv[k] = b4[j + k * stride];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 nb = fma4_momentum(mu, bv[k], gv[k]);
      b4[j + k * stride] = nb;
      uv[k] = bf16r4(L.nesterov ? fma4_momentum(mu, nb, gv[k]) : nb);  // g + mu*buf, as the same two roundings
      u4[j + k * stride] = pack_bf16x4(uv[k]);
    }
    acc = __dadd_rn(acc, sumsq44(uv[0], uv[1]));
    acc = __dadd_rn(acc, sumsq44(uv[2], uv[3]));
  }
  for (; j < n4; j += stride) {
    const float4 gv = load4(g + 4 * j);
    const float4 nb = fma4_momentum(mu, b4[j], gv);
    b4[j] = nb;
    const float4 uv = bf16r4(L.nesterov ? fma4_momentum(mu, nb, gv) : nb);
    u4[j] = pack_bf16x4(uv);
    acc = __dadd_rn(acc, sumsq44(uv, make_float4(0.f, 0.f, 0.f, 0.f)));
  }
  if (c == 0 && threadIdx.x == 0) {
    for (int64_t k = n4 * 4; k < n; ++k) {
      const float gv = load1(g + k);
      const float b = __fadd_rn(__fmul_rn(mu, buf[k]), gv);
      buf[k] = b;
      const float x = bf16r(L.nesterov ? __fadd_rn(__fmul_rn(mu, b), gv) : b);
      u[k] = static_cast<uint16_t>(__float_as_uint(x) >> 16);
      acc = __dadd_rn(acc, __dmul_rn(static_cast<double>(x), static_cast<double>(x)));
    }
  }
  const double block = block_sum(acc, red);
  if (threadIdx.x == 0 && J.npart != nullptr) J.npart[mb * J.npart_stride + c] = block;
}

__device__ __forceinline__ float4 bf16x4(const uint2 w) {
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                     __uint_as_float(w.y & 0xFFFF0000u));
}
__device__ __forceinline__ float bf16x1(const uint16_t h) { return __uint_as_float(static_cast<unsigned>(h) << 16); }

// Step 3: block u is block c = (u - u0) % bpm of matrix mb = (u - u0) / bpm; threads stride over
// the matrix's 4-element bf16 vectors with stride bpm * 256, 8 loads (64 bytes) in flight per round;
// squares are summed in fp32 over runs of 32 (sumsq32: exact fp64 outside the safe range) and
// the runs in fp64. The block's sum and its max |U| (the fp32 bit patterns of non-negative
// values order as unsigned integers; NaN sorts above inf) go to slot c of the matrix's area.
__global__ void __launch_bounds__(kThreads) ustats_kernel(const MuonList L) {
  __shared__ double red[32];
  __shared__ unsigned smax[kThreads / 32];
  const MuonItem& J = L.it[item_of(L, blockIdx.x)];
  const long long v = static_cast<long long>(blockIdx.x) - J.u0;
  const long long mb = v / J.bpm, c = v - mb * J.bpm;
  const long long n = J.n;
  const uint16_t* U = J.u_out + mb * n;
  const uint2* U4 = reinterpret_cast<const uint2*>(U);
  const int64_t n4 = n / 4;
  const int64_t stride = static_cast<int64_t>(J.bpm) * blockDim.x;
  double acc = 0.0;
  unsigned mx = 0;
  auto amax = [](unsigned m, const float4& x) {
    return max(m, max(max(__float_as_uint(x.x) & 0x7FFFFFFFu, __float_as_uint(x.y) & 0x7FFFFFFFu),
                      max(__float_as_uint(x.z) & 0x7FFFFFFFu, __float_as_uint(x.w) & 0x7FFFFFFFu)));
  };
  int64_t j = c * blockDim.x + threadIdx.x;
  for (; j + 7 * stride < n4; j += 8 * stride) {
    float4 x[8];
    uint2 w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = __ldg(U4 + j + k * stride);
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = bf16x4(w[k]);
    float r[4][8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float* d = r[k >> 1] + 4 * (k & 1);
      d[0] = x[k].x; d[1] = x[k].y; d[2] = x[k].z; d[3] = x[k].w;
      mx = amax(mx, x[k]);
    }
    acc = __dadd_rn(acc, sumsq32(r[0], r[1], r[2], r[3]));
  }
  for (; j < n4; j += stride) {
    const float4 x = bf16x4(__ldg(U4 + j));
    acc = __dadd_rn(acc, sumsq44(x, make_float4(0.f, 0.f, 0.f, 0.f)));
    mx = amax(mx, x);
  }
  if (c == 0 && threadIdx.x == 0) {
    for (int64_t k = n4 * 4; k < n; ++k) {
      const float x = bf16x1(U[k]);
      acc = __dadd_rn(acc, __dmul_rn(static_cast<double>(x), static_cast<double>(x)));
      mx = max(mx, __float_as_uint(x) & 0x7FFFFFFFu);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  if ((threadIdx.x & 31) == 0) smax[threadIdx.x >> 5] = mx;
  const double block = block_sum(acc, red);  // (its barriers also publish smax)
  if (threadIdx.x == 0) {
    unsigned m = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) m = max(m, smax[w]);
    J.rsum[mb * J.rcap + c] = block;
    J.rmax[mb * J.rcap + c] = m;
  }
}

// Step 4: block u updates block c of matrix mb (as step 3 splits it). It first reduces the
// matrix's nred maxima (every block) and partial sums (block 0, which writes the stats; threads
// stride over the slots, then the block tree). Rejected (max |U| above the guard, or NaN): the
// master is kept, the bf16 round-out is written either way.
__global__ void __launch_bounds__(kThreads) update_kernel(const MuonList L) {
  __shared__ double red[32];
  __shared__ unsigned smax[kThreads / 32];
  __shared__ unsigned s_max;
  const MuonItem& J = L.it[item_of(L, blockIdx.x)];
  const long long v = static_cast<long long>(blockIdx.x) - J.u0;
  const long long mb = v / J.bpm, c = v - mb * J.bpm;
  const long long n = J.n;
  const double* rs = J.rsum + mb * J.rcap;
  const unsigned* rm = J.rmax + mb * J.rcap;
  double a = 0.0;
  unsigned m = 0;
  for (int i = threadIdx.x; i < J.nred; i += kThreads) {  // from L2: another kernel wrote them
    if (c == 0) a = __dadd_rn(a, __ldcg(rs + i));
    m = max(m, __ldcg(rm + i));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) smax[threadIdx.x >> 5] = m;
  const double ss = block_sum(a, red);  // valid in thread 0 (its barriers also publish smax)
  if (threadIdx.x == 0) {
    unsigned mm = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) mm = max(mm, smax[w]);
    s_max = mm;
    if (c == 0) {
      const double norm64 = (ss >= 0.0) ? __dsqrt_rn(ss) : __longlong_as_double(0x7FF8000000000000LL);
      const float fro = __double2float_rn(norm64);
      const float max_abs = __uint_as_float(mm);
      J.stats[mb] = zopt_muon_stats{fro, __fdiv_rn(fro, J.sqrt_min), max_abs, !(max_abs <= L.guard) ? 1u : 0u};
    }
  }
  __syncthreads();
  const bool rejected = !(__uint_as_float(s_max) <= L.guard);
  float* p = J.master + mb * n;
  const uint16_t* U = J.u_out + mb * n;
  uint16_t* out = J.out ? J.out + mb * n : nullptr;
  const float decay = J.decay, step = J.step;
  auto one = [&](float x, float u) { return __fsub_rn(__fmul_rn(x, decay), __fmul_rn(step, u)); };
  auto put = [&](int64_t k, const float4& x) {
    const unsigned short b0 = __bfloat16_as_ushort(__float2bfloat16_rn(x.x)),
                         b1 = __bfloat16_as_ushort(__float2bfloat16_rn(x.y)),
                         b2 = __bfloat16_as_ushort(__float2bfloat16_rn(x.z)),
                         b3 = __bfloat16_as_ushort(__float2bfloat16_rn(x.w));
    if (J.out8) {
      *reinterpret_cast<uint2*>(out + 4 * k) =
          make_uint2(b0 | (static_cast<unsigned>(b1) << 16), b2 | (static_cast<unsigned>(b3) << 16));
    } else {
      out[4 * k] = b0; out[4 * k + 1] = b1; out[4 * k + 2] = b2; out[4 * k + 3] = b3;
    }
  };
  const int64_t n4 = n / 4;
  const int64_t stride = static_cast<int64_t>(J.bpm) * blockDim.x;
  float4* p4 = reinterpret_cast<float4*>(p);
  const uint2* U4 = reinterpret_cast<const uint2*>(U);
  int64_t j = c * blockDim.x + threadIdx.x;
  for (; j + stride < n4; j += 2 * stride) {
    float4 x = p4[j], y = p4[j + stride];
    if (!rejected) {
      const float4 ux = bf16x4(__ldg(U4 + j)), uy = bf16x4(__ldg(U4 + j + stride));
      x = make_float4(one(x.x, ux.x), one(x.y, ux.y), one(x.z, ux.z), one(x.w, ux.w));
      y = make_float4(one(y.x, uy.x), one(y.y, uy.y), one(y.z, uy.z), one(y.w, uy.w));
      p4[j] = x;
      p4[j + stride] = y;
    }
    if (out) {
      put(j, x);
      put(j + stride, y);
    }
  }
  for (; j < n4; j += stride) {
    float4 x = p4[j];
    if (!rejected) {
      const float4 ux = bf16x4(__ldg(U4 + j));
      x = make_float4(one(x.x, ux.x), one(x.y, ux.y), one(x.z, ux.z), one(x.w, ux.w));
      p4[j] = x;
    }
    if (out) put(j, x);
  }
  if (c == 0 && threadIdx.x == 0) {
    for (int64_t k = n4 * 4; k < n; ++k) {
      float x = p[k];
      if (!rejected) {
        x = one(x, bf16x1(U[k]));
        p[k] = x;
      }
      if (out) out[k] = __bfloat16_as_ushort(__float2bfloat16_rn(x));
    }
  }
}

// One shape's matrices of a Muon step.
struct Job {
  float* master;
  float* momentum;
  const void* grad;
  zopt_dtype gdt;
  uint16_t* out;
  long long rows, cols;
  long long batch;
  zopt_muon_stats* stats;
};

zopt_status check_job(const char* fn, const Job& j) {
  const std::string f(fn);
  if (j.master == nullptr || j.momentum == nullptr || j.grad == nullptr || j.stats == nullptr)
    return fail(ZOPT_EINVAL, f + ": NULL pointer");
  if (j.rows < 1 || j.cols < 1 || j.batch < 1) return fail(ZOPT_EINVAL, f + ": empty matrix or batch");
  if (j.rows > ZOPT_NS_MAX_DIM || j.cols > ZOPT_NS_MAX_DIM || j.rows * j.cols > ZOPT_NS_MAX_ELEMS)
    return fail(ZOPT_EINVAL, f + ": a dimension above 2^30 or a matrix above 2^36 elements");
  if (j.batch > kMaxCallElems / (j.rows * j.cols))
    return fail(ZOPT_EINVAL, f + ": the batch holds more than 2^46 elements");
  if (!aligned16(j.master) || !aligned16(j.momentum) || !aligned16(j.grad) ||
      (j.out != nullptr && (reinterpret_cast<uintptr_t>(j.out) & 1u) != 0) ||
      (reinterpret_cast<uintptr_t>(j.stats) & 3u) != 0)
    return fail(ZOPT_EINVAL, f + ": a device pointer is misaligned");
  if (((j.rows * j.cols) & 3) != 0 && j.batch > 1)
    return fail(ZOPT_EINVAL, f + ": a batch needs rows*cols to be a multiple of 4 (16-byte matrices)");
  if (j.gdt != ZOPT_F32 && j.gdt != ZOPT_BF16) return fail(ZOPT_EUNSUPPORTED, f + ": gradient dtype must be fp32 or bf16");
  return ok();
}

zopt_status check_hparams(const char* fn, const zopt_muon_hparams* hp) {
  if (!std::isfinite(hp->lr) || hp->lr < 0 || !(hp->momentum >= 0 && hp->momentum < 1) ||
      !std::isfinite(hp->weight_decay) || hp->ns_steps < 1 ||
      (hp->adjust != ZOPT_MUON_MATCH_RMS_ADAMW && hp->adjust != ZOPT_MUON_ORIGINAL) || !(hp->guard > 0))
    return fail(ZOPT_EINVAL, std::string(fn) + ": hyper-parameters out of range");
  return ok();
}

// The element-wise item for matrices b0 .. b0 + gs - 1 of job j, whose workspace slice (plan P)
// starts at ws.
MuonItem item_of_job(const Job& j, long long b0, int gs, uint8_t* ws, const MuonPlan& P, const zopt_muon_hparams* hp) {
  const long long rows = j.rows, cols = j.cols, n = rows * cols;
  const size_t gsz = j.gdt == ZOPT_F32 ? 4 : 2;
  const double scale = hp->adjust == ZOPT_MUON_MATCH_RMS_ADAMW
                           ? 0.2 * std::sqrt(static_cast<double>(rows > cols ? rows : cols))
                           : std::sqrt(rows > cols ? static_cast<double>(rows) / static_cast<double>(cols) : 1.0);
  MuonItem it{};
  it.master = j.master + b0 * n;
  it.momentum = j.momentum + b0 * n;
  it.grad = static_cast<const uint8_t*>(j.grad) + static_cast<size_t>(b0 * n) * gsz;
  it.u_in = reinterpret_cast<uint16_t*>(ws + P.off_u);  // unless the Newton-Schulz X0 takes u (attach_ns)
  it.u_stride = n;
  it.u_out = reinterpret_cast<const uint16_t*>(ws + P.off_o);
  it.npart = nullptr;  // set once the Newton-Schulz workspace is known
  it.npart_stride = 0;
  it.out = j.out ? j.out + b0 * n : nullptr;
  it.stats = j.stats + b0;
  it.rcap = red_cap(rows, cols);
  it.rsum = reinterpret_cast<double*>(ws);
  it.rmax = reinterpret_cast<unsigned*>(ws + gs * it.rcap * 8);
  it.n = n;
  it.batch = gs;
  // depends on n only (a matrix's stats are the same in any call), and equals the Newton-Schulz
  // norm's partial count, which the momentum pass fills
  it.bpm = ns::norm_blocks(n);
  it.nred = it.bpm;  // until the Newton-Schulz call says its epilogue writes the slots
  it.ns_stats = 0;
  // 8-byte bf16 stores need the first matrix 8-byte aligned and every matrix a multiple of 4
  it.out8 = it.out != nullptr && (reinterpret_cast<uintptr_t>(it.out) & 7u) == 0 && (n & 3) == 0 ? 1 : 0;
  it.decay = static_cast<float>(1.0 - hp->lr * hp->weight_decay);
  it.step = static_cast<float>(hp->lr * scale);
  it.sqrt_min = static_cast<float>(std::sqrt(static_cast<double>(rows < cols ? rows : cols)));
  return it;
}

enum Pass { kMomentumBf16, kMomentumF32, kStats, kUpdate };

// One pass over every item that takes it (momentum: those with the pass's gradient dtype),
// kMaxItems to a launch, one block per chunk (momentum) or per matrix block (stats, update).
zopt_status launch_pass(Pass pass, const std::vector<MuonItem>& items, const std::vector<zopt_dtype>& gdt,
                        const zopt_muon_hparams* hp, cudaStream_t s) {
  MuonList L{};
  L.mu = static_cast<float>(hp->momentum);
  L.nesterov = hp->nesterov ? 1 : 0;
  L.guard = hp->guard;
  long long units = 0;
  auto flush = [&]() -> zopt_status {
    if (L.n == 0) return ok();
    if (units > 0x7FFFFFFFLL) return fail(ZOPT_EINVAL, "zopt_muon_step: too many blocks for one launch");
    const dim3 grid(static_cast<unsigned>(units)), block(kThreads);
    if (pass == kMomentumBf16) momentum_kernel<__nv_bfloat16><<<grid, block, 0, s>>>(L);
    else if (pass == kMomentumF32) momentum_kernel<float><<<grid, block, 0, s>>>(L);
    else if (pass == kStats) ustats_kernel<<<grid, block, 0, s>>>(L);
    else update_kernel<<<grid, block, 0, s>>>(L);
    ZOPT_CUDA_TRY(cudaGetLastError());
    L.n = 0;
    units = 0;
    return ok();
  };
  zopt_status st = ZOPT_OK;
  for (size_t k = 0; k < items.size(); ++k) {
    if (pass == kMomentumBf16 && gdt[k] != ZOPT_BF16) continue;
    if (pass == kMomentumF32 && gdt[k] != ZOPT_F32) continue;
    if (pass == kStats && items[k].ns_stats) continue;
    if (L.n == kMaxItems && (st = flush()) != ZOPT_OK) return st;
    MuonItem it = items[k];
    it.u0 = units;
    units += static_cast<long long>(it.batch) * it.bpm;
    L.it[L.n++] = it;
  }
  return flush();
}

zopt_status launch_momentum(const std::vector<MuonItem>& items, const std::vector<zopt_dtype>& gdt,
                            const zopt_muon_hparams* hp, cudaStream_t s) {
  zopt_status st = launch_pass(kMomentumBf16, items, gdt, hp, s);
  return st != ZOPT_OK ? st : launch_pass(kMomentumF32, items, gdt, hp, s);
}

zopt_status launch_update(const std::vector<MuonItem>& items, const std::vector<zopt_dtype>& gdt,
                          const zopt_muon_hparams* hp, cudaStream_t s) {
  zopt_status st = launch_pass(kStats, items, gdt, hp, s);
  return st != ZOPT_OK ? st : launch_pass(kUpdate, items, gdt, hp, s);
}

Job job_of(const zopt_muon_job& b) {
  return Job{b.master, b.momentum, b.grad, static_cast<zopt_dtype>(b.grad_dtype), b.out_bf16,
             b.rows, b.cols, b.batch, b.d_stats};
}

// The Newton-Schulz job of a Muon job: u -> U, both bf16, contiguous matrices.
zopt_ns_job ns_job_of(const Job& j, const uint16_t* U_in, uint16_t* U_out) {
  const long long n = j.rows * j.cols;
  zopt_ns_job q;
  q.G = U_in;
  q.X = U_out;
  q.rows = j.rows;
  q.cols = j.cols;
  q.ld_g = j.cols;
  q.ld_x = j.cols;
  q.batch_stride_g = n;
  q.batch_stride_x = n;
  q.batch = static_cast<int32_t>(j.batch);
  q.io_dtype = ZOPT_BF16;
  return q;
}

// Points each item's momentum pass at its Newton-Schulz job's norm partials (ns[] in the
// Newton-Schulz workspace nws), which the pass fills in place of a sum-of-squares launch, and,
// where the job can take it (raw[k] set), at the job's X0 itself: u goes there unnormalised
// and the first step's products normalise it, so no preparation pass reads u.
void attach_ns(const std::vector<zopt_ns_job>& ns, uint8_t* nws, std::vector<MuonItem>& items, bool* raw) {
  const size_t n = ns.size();
  std::vector<double*> base(n);
  std::vector<long long> stride(n), xs(n);
  std::vector<uint16_t*> x0(n);
  ns::many_norm_partials(ns.data(), static_cast<int32_t>(n), nws, base.data(), stride.data());
  ns::many_x0(ns.data(), static_cast<int32_t>(n), nws, x0.data(), xs.data(), raw);
  for (size_t k = 0; k < n; ++k) {
    items[k].npart = base[k];
    items[k].npart_stride = stride[k];
    if (raw[k]) {
      items[k].u_in = x0[k];
      items[k].u_stride = xs[k];
    }
  }
}

// Step 2: U = NewtonSchulz(u) for every job in one many-call, its norms taken from the partials
// the momentum pass wrote and U written in bf16. Where the last product's epilogue is a TMA one,
// it also writes U's statistics slots (step 3 then skips the item).
zopt_status muon_ns(const char* fn, const std::vector<zopt_ns_job>& ns, const zopt_muon_hparams* hp, uint8_t* nws,
                    size_t nws_bytes, cudaStream_t s, std::vector<MuonItem>& items, const bool* raw) {
  const size_t n = ns.size();
  const std::vector<zopt_dtype> out(n, ZOPT_BF16);
  std::unique_ptr<bool[]> ready(new bool[n]);
  std::vector<ns::StatsSink> sinks(n);
  std::vector<int> slots(n, 0);
  for (size_t k = 0; k < n; ++k) {
    ready[k] = true;
    sinks[k] = ns::StatsSink{items[k].rsum, items[k].rmax, items[k].rcap, items[k].rcap};
  }
  const zopt_status st = ns::orthogonalize_many(fn, ns.data(), static_cast<int32_t>(n), hp->ns_steps, hp->abc, hp->eps,
                                                nws, nws_bytes, s, out.data(), ready.get(), sinks.data(), slots.data(),
                                                raw);
  for (size_t k = 0; k < n; ++k) {
    items[k].ns_stats = slots[k] > 0 ? 1 : 0;
    items[k].nred = slots[k] > 0 ? slots[k] : items[k].bpm;
  }
  return st;
}

}  // namespace
}  // namespace zopt

extern "C" size_t zopt_muon_workspace(int64_t rows, int64_t cols, int32_t group) {
  if (rows < 1 || cols < 1 || group < 1) return 0;
  if (rows > ZOPT_NS_MAX_DIM || cols > ZOPT_NS_MAX_DIM || rows * cols > ZOPT_NS_MAX_ELEMS) return 0;
  return zopt::muon_plan(rows, cols, group).total;
}

extern "C" zopt_status zopt_muon_step(float* master, float* momentum, const void* grad, zopt_dtype grad_dtype,
                                      uint16_t* out_bf16, int64_t rows, int64_t cols, int32_t batch,
                                      const zopt_muon_hparams* hp, zopt_muon_stats* d_stats, void* d_ws,
                                      size_t ws_bytes, zopt_stream stream) {
  using namespace zopt;
  const char* fn = "zopt_muon_step";
  if (hp == nullptr || d_ws == nullptr) return fail(ZOPT_EINVAL, "zopt_muon_step: NULL pointer");
  const Job j{master, momentum, grad, grad_dtype, out_bf16, rows, cols, batch, d_stats};
  zopt_status st = check_job(fn, j);
  if (st != ZOPT_OK) return st;
  if (!aligned16(d_ws)) return fail(ZOPT_EINVAL, "zopt_muon_step: a device pointer is misaligned");
  if ((st = check_hparams(fn, hp)) != ZOPT_OK) return st;
  long long group = 0;
  {
    const MuonPlan one = muon_plan(rows, cols, 1);
    if (ws_bytes >= one.total) {
      group = batch;
      if (group > 65535) group = 65535;
      while (group > 1 && muon_plan(rows, cols, group).total > ws_bytes) --group;
    }
  }
  if (group < 1) return fail(ZOPT_EINVAL, "zopt_muon_step: workspace smaller than zopt_muon_workspace(rows, cols, 1)");
  const MuonPlan P = muon_plan(rows, cols, group);
  uint8_t* ws = static_cast<uint8_t*>(d_ws);
  uint16_t* U_in = reinterpret_cast<uint16_t*>(ws + P.off_u);
  uint16_t* U_out = reinterpret_cast<uint16_t*>(ws + P.off_o);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int sms = sm_count();
  if (sms <= 0) return fail(ZOPT_ECUDA, "zopt_muon_step: no CUDA device");
  const std::vector<zopt_dtype> gdt{grad_dtype};
  for (long long b0 = 0; b0 < batch; b0 += group) {
    const int gs = static_cast<int>(batch - b0 < group ? batch - b0 : group);
    std::vector<MuonItem> items{item_of_job(j, b0, gs, ws, P, hp)};
    Job jg = j;
    jg.batch = gs;
    const std::vector<zopt_ns_job> ns{ns_job_of(jg, U_in, U_out)};
    bool raw[1];
    attach_ns(ns, ws + P.off_ns, items, raw);
    // 1. momentum over the group's matrices (contiguous), u and its norm partials into the workspace
    if ((st = launch_momentum(items, gdt, hp, s)) != ZOPT_OK) return st;
    // 2. U = NewtonSchulz(u), bf16 in and out, bf16 tensor cores
    if ((st = muon_ns(fn, ns, hp, ws + P.off_ns, P.ns_bytes, s, items, raw)) != ZOPT_OK) return st;
    // 3, 4. per-matrix statistics, the guarded update and bf16 round-out
    if ((st = launch_update(items, gdt, hp, s)) != ZOPT_OK) return st;
  }
  return ok();
}

static_assert(sizeof(zopt_muon_job) == 64, "zopt_muon_job layout");

extern "C" size_t zopt_muon_workspace_many(const zopt_muon_job* jobs, int32_t n_jobs) {
  using namespace zopt;
  if (jobs == nullptr || n_jobs < 1) return 0;
  size_t total = 0;
  std::vector<zopt_ns_job> ns(static_cast<size_t>(n_jobs));
  for (int32_t k = 0; k < n_jobs; ++k) {
    const zopt_muon_job& b = jobs[k];
    if (b.rows < 1 || b.cols < 1 || b.batch < 1 || b.batch > 65535) return 0;
    if (b.rows > ZOPT_NS_MAX_DIM || b.cols > ZOPT_NS_MAX_DIM || b.rows * b.cols > ZOPT_NS_MAX_ELEMS) return 0;
    total += static_cast<size_t>(round_up(static_cast<long long>(muon_plan(b.rows, b.cols, b.batch).off_ns), 1024));
    ns[static_cast<size_t>(k)] = ns_job_of(job_of(b), nullptr, nullptr);
  }
  const size_t nsb = zopt_ns_workspace_many(ns.data(), n_jobs);
  return nsb == 0 ? 0 : total + nsb;
}

extern "C" zopt_status zopt_muon_step_many(const zopt_muon_job* jobs, int32_t n_jobs, const zopt_muon_hparams* hp,
                                           void* d_ws, size_t ws_bytes, zopt_stream stream) {
  using namespace zopt;
  const char* fn = "zopt_muon_step_many";
  if (jobs == nullptr || hp == nullptr || d_ws == nullptr) return fail(ZOPT_EINVAL, "zopt_muon_step_many: NULL pointer");
  if (n_jobs < 1) return fail(ZOPT_EINVAL, "zopt_muon_step_many: no jobs");
  if (!aligned16(d_ws)) return fail(ZOPT_EINVAL, "zopt_muon_step_many: a device pointer is misaligned");
  zopt_status st = check_hparams(fn, hp);
  if (st != ZOPT_OK) return st;
  for (int32_t k = 0; k < n_jobs; ++k) {
    if ((st = check_job(fn, job_of(jobs[k]))) != ZOPT_OK) return st;
    if (jobs[k].batch > 65535) return fail(ZOPT_EINVAL, "zopt_muon_step_many: a job's batch exceeds 65535");
  }
  const size_t need = zopt_muon_workspace_many(jobs, n_jobs);
  if (need == 0 || ws_bytes < need)
    return fail(ZOPT_EINVAL, "zopt_muon_step_many: workspace smaller than zopt_muon_workspace_many");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int sms = sm_count();
  if (sms <= 0) return fail(ZOPT_ECUDA, "zopt_muon_step_many: no CUDA device");
  // every job's whole batch in its own slice of the workspace: momentum for all, Newton-Schulz
  // for all in one call (the shapes below 1024 share fused launches), then the updates
  uint8_t* ws = static_cast<uint8_t*>(d_ws);
  std::vector<zopt_ns_job> ns(static_cast<size_t>(n_jobs));
  std::vector<MuonItem> items(static_cast<size_t>(n_jobs));
  std::vector<zopt_dtype> gdt(static_cast<size_t>(n_jobs));
  size_t at = 0;
  for (int32_t k = 0; k < n_jobs; ++k) {
    const Job j = job_of(jobs[k]);
    const MuonPlan P = muon_plan(j.rows, j.cols, j.batch);
    items[static_cast<size_t>(k)] = item_of_job(j, 0, static_cast<int>(j.batch), ws + at, P, hp);
    gdt[static_cast<size_t>(k)] = j.gdt;
    ns[static_cast<size_t>(k)] = ns_job_of(j, items[static_cast<size_t>(k)].u_in,
                                           const_cast<uint16_t*>(items[static_cast<size_t>(k)].u_out));
    at += static_cast<size_t>(round_up(static_cast<long long>(P.off_ns), 1024));
  }
  std::unique_ptr<bool[]> raw(new bool[static_cast<size_t>(n_jobs)]);
  attach_ns(ns, ws + at, items, raw.get());
  if ((st = launch_momentum(items, gdt, hp, s)) != ZOPT_OK) return st;
  if ((st = muon_ns(fn, ns, hp, ws + at, ws_bytes - at, s, items, raw.get())) != ZOPT_OK) return st;
  return launch_update(items, gdt, hp, s);
}
