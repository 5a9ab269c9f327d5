// Muon's update around Newton-Schulz, for the matrices a rank owns whole.
//
// bluscript_zero_ckpt.cpp, ShardedMuon: each matrix has one owner rank holding its fp32 master
// and momentum; momentum 0.95 with Nesterov, decoupled weight decay, U = NewtonSchulz(u);
// adjust_lr "match_rms_adamw" lifts the update's RMS to 0.2 (scale 0.2*sqrt(max(rows, cols)))
// and "original" uses sqrt(max(1, rows/cols)); diagnostics nsratio = ||U||_F/sqrt(min(rows,
// cols)) and a divergence guard that rejects an update with an element above 1000.
//
// Per group of matrices (as many as the workspace holds), four steps on the caller's stream:
//   1. momentum:  buf = mu*buf + g;  u = g + mu*buf (Nesterov) or buf      (fp32, 14-16 B/elem)
//   2. U = NewtonSchulz(u) through zopt_ns_orthogonalize (fp32 in/out, bf16 tensor cores)
//   3. per matrix: sum of squares and largest magnitude of U                 (4 B/elem)
//   4. p = p*fp32(1 - lr*wd) - fp32(lr*scale)*U unless rejected; bf16 round-out (14 B/elem)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <string>
#include <vector>

#include "internal.h"
#include "norm_impl.cuh"

namespace zopt {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxBlocksPerMat = 512;
constexpr size_t kRedBytes = 256 + sizeof(double) * kMaxBlocksPerMat;  // one NormWorkspace per matrix

long long round_up(long long x, long long a) { return (x + a - 1) / a * a; }

struct MuonPlan {
  size_t off_max, off_cs, off_u, off_o, off_ns, ns_bytes, total;
};

MuonPlan muon_plan(long long rows, long long cols, long long group) {
  MuonPlan p;
  const long long n = rows * cols;
  p.off_max = static_cast<size_t>(round_up(group * static_cast<long long>(kRedBytes), 256));
  p.off_cs = static_cast<size_t>(round_up(static_cast<long long>(p.off_max) + group * 4, 256));
  p.off_u = static_cast<size_t>(round_up(static_cast<long long>(p.off_cs) + group * 32, 1024));
  p.off_o = p.off_u + static_cast<size_t>(round_up(group * n * 4, 1024));
  p.off_ns = p.off_o + static_cast<size_t>(round_up(group * n * 4, 1024));
  p.ns_bytes = zopt_ns_workspace(rows, cols, static_cast<int32_t>(group), ZOPT_BF16);
  p.total = p.off_ns + p.ns_bytes;
  return p;
}

__device__ __forceinline__ float4 fma4_momentum(float mu, const float4& b, const float4& g) {
  return make_float4(__fadd_rn(__fmul_rn(mu, b.x), g.x), __fadd_rn(__fmul_rn(mu, b.y), g.y),
                     __fadd_rn(__fmul_rn(mu, b.z), g.z), __fadd_rn(__fmul_rn(mu, b.w), g.w));
}

template <typename T>
__global__ void __launch_bounds__(kThreads) momentum_kernel(float* __restrict__ buf, const T* __restrict__ g,
                                                             float* __restrict__ u, int64_t n, float mu, int nesterov) {
  const int64_t n4 = n / 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  float4* b4 = reinterpret_cast<float4*>(buf);
  float4* u4 = reinterpret_cast<float4*>(u);
  int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; j + stride < n4; j += 2 * stride) {  // two vectors' loads in flight before any store
    const float4 ga = load4(g + 4 * j), gb = load4(g + 4 * (j + stride));
    const float4 ba = b4[j], bb = b4[j + stride];
    const float4 na = fma4_momentum(mu, ba, ga), nb = fma4_momentum(mu, bb, gb);
    b4[j] = na;
    b4[j + stride] = nb;
    u4[j] = nesterov ? fma4_momentum(mu, na, ga) : na;  // g + mu*buf, as the same two roundings
    u4[j + stride] = nesterov ? fma4_momentum(mu, nb, gb) : nb;
  }
  for (; j < n4; j += stride) {
    const float4 gv = load4(g + 4 * j);
    const float4 b = fma4_momentum(mu, b4[j], gv);
    b4[j] = b;
    u4[j] = nesterov ? fma4_momentum(mu, b, gv) : b;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    for (int64_t k = n4 * 4; k < n; ++k) {
      const float gv = load1(g + k);
      const float b = __fadd_rn(__fmul_rn(mu, buf[k]), gv);
      buf[k] = b;
      u[k] = nesterov ? __fadd_rn(__fmul_rn(mu, b), gv) : b;
    }
  }
}

// Per matrix (blockIdx.y): sum of squares of U and max |U| (the fp32 bit patterns of
// non-negative values order as unsigned integers; NaN sorts above inf). Threads stride over
// 4-element vectors, 8 loads (128 bytes) in flight per round; squares are summed in fp32 over
// runs of 32 (sumsq32: exact fp64 outside the safe range) and the runs in fp64; one partial per
// block, the last block of the matrix adding them in a fixed order.
__global__ void __launch_bounds__(kThreads) ustats_kernel(const float* __restrict__ U0, int64_t n, uint8_t* red,
                                                           unsigned* maxbits, zopt_clip_stats* cs) {
  const int mb = blockIdx.y;
  const float* U = U0 + mb * n;
  const int64_t n4 = n / 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  double acc = 0.0;
  unsigned mx = 0;
  auto amax = [](unsigned m, const float4& x) {
    return max(m, max(max(__float_as_uint(x.x) & 0x7FFFFFFFu, __float_as_uint(x.y) & 0x7FFFFFFFu),
                      max(__float_as_uint(x.z) & 0x7FFFFFFFu, __float_as_uint(x.w) & 0x7FFFFFFFu)));
  };
  int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; j + 7 * stride < n4; j += 8 * stride) {
    float4 x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = __ldg(reinterpret_cast<const float4*>(U) + j + k * stride);
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
    const float4 x = __ldg(reinterpret_cast<const float4*>(U) + j);
    acc = __dadd_rn(acc, sumsq44(x, make_float4(0.f, 0.f, 0.f, 0.f)));
    mx = amax(mx, x);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    for (int64_t k = n4 * 4; k < n; ++k) {
      const float x = U[k];
      acc = __dadd_rn(acc, __dmul_rn(static_cast<double>(x), static_cast<double>(x)));
      mx = max(mx, __float_as_uint(x) & 0x7FFFFFFFu);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  if ((threadIdx.x & 31) == 0) atomicMax(maxbits + mb, mx);
  finish_sumsq(acc, reinterpret_cast<NormWorkspace*>(red + mb * kRedBytes), cs + mb, 0.0f);
}

// p = p * decay - step * U unless the matrix is rejected; the bf16 round-out of p either way.
// Threads stride over 4-element vectors, two in flight per round (master and U: 64 bytes);
// `out8`: the bf16 rows allow 8-byte stores.
__global__ void __launch_bounds__(kThreads)
    update_kernel(float* __restrict__ p0, const float* __restrict__ U0, uint16_t* __restrict__ out0, int64_t n,
                  int out8, const zopt_clip_stats* cs, const unsigned* maxbits, float decay, float step, float guard,
                  float sqrt_min_dim, zopt_muon_stats* st) {
  const int mb = blockIdx.y;
  float* p = p0 + mb * n;
  const float* U = U0 + mb * n;
  uint16_t* out = out0 ? out0 + mb * n : nullptr;
  const float max_abs = __uint_as_float(maxbits[mb]);
  const bool rejected = !(max_abs <= guard);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const float fro = cs[mb].norm;
    st[mb] = zopt_muon_stats{fro, __fdiv_rn(fro, sqrt_min_dim), max_abs, rejected ? 1u : 0u};
  }
  auto one = [&](float v, float u) { return __fsub_rn(__fmul_rn(v, decay), __fmul_rn(step, u)); };
  auto put = [&](int64_t k, const float4& v) {
    const unsigned short b0 = __bfloat16_as_ushort(__float2bfloat16_rn(v.x)),
                         b1 = __bfloat16_as_ushort(__float2bfloat16_rn(v.y)),
                         b2 = __bfloat16_as_ushort(__float2bfloat16_rn(v.z)),
                         b3 = __bfloat16_as_ushort(__float2bfloat16_rn(v.w));
    if (out8) {
      *reinterpret_cast<uint2*>(out + 4 * k) =
          make_uint2(b0 | (static_cast<unsigned>(b1) << 16), b2 | (static_cast<unsigned>(b3) << 16));
    } else {
      out[4 * k] = b0; out[4 * k + 1] = b1; out[4 * k + 2] = b2; out[4 * k + 3] = b3;
    }
  };
  const int64_t n4 = n / 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  float4* p4 = reinterpret_cast<float4*>(p);
  const float4* U4 = reinterpret_cast<const float4*>(U);
  int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; j + stride < n4; j += 2 * stride) {
    float4 a = p4[j], b = p4[j + stride];
    if (!rejected) {
      const float4 ua = __ldg(U4 + j), ub = __ldg(U4 + j + stride);
      a = make_float4(one(a.x, ua.x), one(a.y, ua.y), one(a.z, ua.z), one(a.w, ua.w));
      b = make_float4(one(b.x, ub.x), one(b.y, ub.y), one(b.z, ub.z), one(b.w, ub.w));
      p4[j] = a;
      p4[j + stride] = b;
    }
    if (out) {
      put(j, a);
      put(j + stride, b);
    }
  }
  for (; j < n4; j += stride) {
    float4 a = p4[j];
    if (!rejected) {
      const float4 ua = __ldg(U4 + j);
      a = make_float4(one(a.x, ua.x), one(a.y, ua.y), one(a.z, ua.z), one(a.w, ua.w));
      p4[j] = a;
    }
    if (out) put(j, a);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    for (int64_t k = n4 * 4; k < n; ++k) {
      float v = p[k];
      if (!rejected) {
        v = one(v, U[k]);
        p[k] = v;
      }
      if (out) out[k] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
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

// Step 1 for matrices b0 .. b0 + gs - 1 of a job (contiguous): momentum, u into U_in.
zopt_status launch_momentum(const Job& j, long long b0, int gs, float* U_in, const zopt_muon_hparams* hp, int sms,
                            cudaStream_t s) {
  const long long n = j.rows * j.cols, ng = n * gs;
  const size_t gsz = j.gdt == ZOPT_F32 ? 4 : 2;
  float* bm = j.momentum + b0 * n;
  const uint8_t* gm = static_cast<const uint8_t*>(j.grad) + static_cast<size_t>(b0 * n) * gsz;
  const float mu = static_cast<float>(hp->momentum);
  long long blocks = (ng / 4 + kThreads - 1) / kThreads;
  if (blocks > static_cast<long long>(sms) * 8) blocks = static_cast<long long>(sms) * 8;
  if (blocks < 1) blocks = 1;
  if (j.gdt == ZOPT_F32)
    momentum_kernel<float><<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(
        bm, reinterpret_cast<const float*>(gm), U_in, ng, mu, hp->nesterov ? 1 : 0);
  else
    momentum_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(
        bm, reinterpret_cast<const __nv_bfloat16*>(gm), U_in, ng, mu, hp->nesterov ? 1 : 0);
  ZOPT_CUDA_TRY(cudaGetLastError());
  return ok();
}

// Steps 3 and 4 for matrices b0 .. b0 + gs - 1: per-matrix ||U|| and max |U| into the plan's
// reduction area at ws, then the guarded update and bf16 round-out.
zopt_status launch_update(const Job& j, long long b0, int gs, uint8_t* ws, const MuonPlan& P, const float* U_out,
                          const zopt_muon_hparams* hp, cudaStream_t s) {
  const long long rows = j.rows, cols = j.cols, n = rows * cols;
  const double scale = hp->adjust == ZOPT_MUON_MATCH_RMS_ADAMW
                           ? 0.2 * std::sqrt(static_cast<double>(rows > cols ? rows : cols))
                           : std::sqrt(rows > cols ? static_cast<double>(rows) / static_cast<double>(cols) : 1.0);
  const float decay = static_cast<float>(1.0 - hp->lr * hp->weight_decay);
  const float step = static_cast<float>(hp->lr * scale);
  const float sqrt_min = static_cast<float>(std::sqrt(static_cast<double>(rows < cols ? rows : cols)));
  unsigned* maxbits = reinterpret_cast<unsigned*>(ws + P.off_max);
  zopt_clip_stats* cs = reinterpret_cast<zopt_clip_stats*>(ws + P.off_cs);
  ZOPT_CUDA_TRY(cudaMemsetAsync(ws, 0, P.off_cs, s));  // reduction counters and maxima start at zero
  long long bpm = (n + 32767) / 32768;
  bpm = bpm < 1 ? 1 : (bpm > kMaxBlocksPerMat ? kMaxBlocksPerMat : bpm);
  const dim3 grid(static_cast<unsigned>(bpm), static_cast<unsigned>(gs));
  ustats_kernel<<<grid, kThreads, 0, s>>>(U_out, n, ws, maxbits, cs);
  ZOPT_CUDA_TRY(cudaGetLastError());
  uint16_t* out = j.out ? j.out + b0 * n : nullptr;
  // 8-byte bf16 stores need the first matrix 8-byte aligned and every matrix a multiple of 4
  const int out8 = out != nullptr && (reinterpret_cast<uintptr_t>(out) & 7u) == 0 && (n & 3) == 0 ? 1 : 0;
  update_kernel<<<grid, kThreads, 0, s>>>(j.master + b0 * n, U_out, out, n, out8, cs, maxbits, decay, step, hp->guard,
                                          sqrt_min, j.stats + b0);
  ZOPT_CUDA_TRY(cudaGetLastError());
  return ok();
}

Job job_of(const zopt_muon_job& b) {
  return Job{b.master, b.momentum, b.grad, static_cast<zopt_dtype>(b.grad_dtype), b.out_bf16,
             b.rows, b.cols, b.batch, b.d_stats};
}

// The Newton-Schulz job of a Muon job: u -> U, fp32 in and out, contiguous matrices.
zopt_ns_job ns_job_of(const Job& j, const float* U_in, float* U_out) {
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
  q.io_dtype = ZOPT_F32;
  return q;
}

}  // namespace
}  // namespace zopt

extern "C" size_t zopt_muon_workspace(int64_t rows, int64_t cols, int32_t group) {
  if (rows < 1 || cols < 1 || group < 1) return 0;
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
  float* U_in = reinterpret_cast<float*>(ws + P.off_u);
  float* U_out = reinterpret_cast<float*>(ws + P.off_o);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int sms = sm_count();
  if (sms <= 0) return fail(ZOPT_ECUDA, "zopt_muon_step: no CUDA device");
  const long long n = rows * cols;
  for (long long b0 = 0; b0 < batch; b0 += group) {
    const int gs = static_cast<int>(batch - b0 < group ? batch - b0 : group);
    // 1. momentum over the group's matrices (contiguous), u into the workspace
    if ((st = launch_momentum(j, b0, gs, U_in, hp, sms, s)) != ZOPT_OK) return st;
    // 2. U = NewtonSchulz(u), fp32 in and out, bf16 tensor cores
    st = zopt_ns_orthogonalize(U_in, U_out, ZOPT_F32, rows, cols, cols, cols, n, n, gs, ZOPT_BF16, hp->ns_steps,
                               hp->abc, hp->eps, ws + P.off_ns, P.ns_bytes, stream);
    if (st != ZOPT_OK) return st;
    // 3, 4. per-matrix statistics, the guarded update and bf16 round-out
    if ((st = launch_update(j, b0, gs, ws, P, U_out, hp, s)) != ZOPT_OK) return st;
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
  std::vector<size_t> off(static_cast<size_t>(n_jobs));
  size_t at = 0;
  for (int32_t k = 0; k < n_jobs; ++k) {
    const Job j = job_of(jobs[k]);
    const MuonPlan P = muon_plan(j.rows, j.cols, j.batch);
    off[static_cast<size_t>(k)] = at;
    float* U_in = reinterpret_cast<float*>(ws + at + P.off_u);
    float* U_out = reinterpret_cast<float*>(ws + at + P.off_o);
    if ((st = launch_momentum(j, 0, static_cast<int>(j.batch), U_in, hp, sms, s)) != ZOPT_OK) return st;
    ns[static_cast<size_t>(k)] = ns_job_of(j, U_in, U_out);
    at += static_cast<size_t>(round_up(static_cast<long long>(P.off_ns), 1024));
  }
  if ((st = zopt_ns_orthogonalize_many(ns.data(), n_jobs, hp->ns_steps, hp->abc, hp->eps, ws + at, ws_bytes - at,
                                       stream)) != ZOPT_OK)
    return st;
  for (int32_t k = 0; k < n_jobs; ++k) {
    const Job j = job_of(jobs[k]);
    const MuonPlan P = muon_plan(j.rows, j.cols, j.batch);
    uint8_t* wj = ws + off[static_cast<size_t>(k)];
    if ((st = launch_update(j, 0, static_cast<int>(j.batch), wj, P, reinterpret_cast<const float*>(wj + P.off_o), hp,
                            s)) != ZOPT_OK)
      return st;
  }
  return ok();
}
