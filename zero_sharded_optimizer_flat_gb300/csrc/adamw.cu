// Fused AdamW over the flat fp32 master shard.
//
// dmuon PR #16, foreach AdamW commit: decoupled weight decay, then the moments, then the
// bias-corrected addcdiv; bias corrections are per-step scalars. DeepSpeed PR #9021: the
// gradient is scaled as it is loaded (after the bf16 -> fp32 promotion). deg/zero.py: flat
// AdamW is the same arithmetic as per tensor; the updated shard is rounded to bf16 compute
// weights (gather_params). bluscript_zero_ckpt.cpp: fp32 master and moments, 1-D parameters
// excluded from weight decay.
//
// Design (HBM-bound, 28-30 algorithmic bytes per element):
//   * one launch per shard; each block owns a contiguous run of 2048-element tiles; a thread
//     moves 2 x 4 elements per tile with 128-bit loads and stores, every warp instruction
//     covering 512 contiguous bytes of each fp32 array;
//   * the weight-decay flag comes from the layout's sorted no-decay runs: each thread keeps
//     a cursor that only moves forward, so a tile without a run boundary costs one compare;
//   * t-dependent scalars are formed once per block by thread 0 in fp64 (IEEE mul/sub/div/
//     sqrt, no contraction) from the device step counter, so a skipped step (found_inf)
//     needs no host round trip; the last block to finish advances the counter;
//   * every per-element operation is an explicitly rounded fp32 intrinsic, so the result
//     is bitwise the exact-order definition.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "adam_common.cuh"
#include "internal.h"
#include "launch.cuh"
#include "norm_impl.cuh"
#include "ns_internal.h"

namespace zopt {
namespace {

using namespace adam;

struct HostScalars {
  float b1, omb1, b2, omb2, eps, decay;  // fp64 -> fp32 once
  double lr, beta1, beta2;               // for the t-dependent scalars
  int skip_on_inf;
};

struct StepScalars {
  float coef, b1, omb1, b2, omb2, eps, decay, step_size, bc2s;
};

// One element, every operation rounded on its own, in the documented order.
__device__ __forceinline__ void adamw_elem(float& p, float& m, float& v, float gin, bool decays,
                                           const StepScalars& s) {
  const float g = __fmul_rn(gin, s.coef);
  if (decays) p = __fmul_rn(p, s.decay);
  m = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
  v = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
  const float d = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), s.bc2s), s.eps);
  p = __fsub_rn(p, __fmul_rn(s.step_size, __fdiv_rn(m, d)));
}

// Is shard slot x inside one of the no-decay runs [runs[2k], runs[2k+1]) with k >= cur
// whose begin is below `limit`?
__device__ __forceinline__ bool in_nodecay(const int64_t* __restrict__ runs, int64_t nruns, int64_t cur,
                                           int64_t limit, int64_t x) {
  for (int64_t k = cur; k < nruns; ++k) {
    const int64_t b = __ldg(runs + 2 * k);
    if (b >= limit) break;
    if (x >= b && x < __ldg(runs + 2 * k + 1)) return true;
  }
  return false;
}

// Thread 0's per-launch scalars: the clip coefficient and found_inf as given, the step
// t = state->step + 1 and its bias corrections (fp64, rounded once to fp32).
__device__ __forceinline__ void step_scalars(const HostScalars& hs, float coef, int found,
                                             const zopt_adam_state* state, StepScalars& sc, int& skip,
                                             long long& t_out) {
  const long long t = *reinterpret_cast<const volatile long long*>(&state->step) + 1;
  const double bc1 = __dsub_rn(1.0, pow_sq_mul(hs.beta1, t));
  const double bc2 = __dsub_rn(1.0, pow_sq_mul(hs.beta2, t));
  sc = StepScalars{coef,   hs.b1,  hs.omb1, hs.b2, hs.omb2, hs.eps, hs.decay,
                   __double2float_rn(__ddiv_rn(hs.lr, bc1)), __double2float_rn(__dsqrt_rn(bc2))};
  skip = (hs.skip_on_inf && found) ? 1 : 0;
  t_out = t;
}

// The block's run of whole 2048-element tiles, updated in place, then the step counter: the
// last block to finish advances it (every block has read it by now).
template <typename G, bool kOut>
__device__ __forceinline__ void adamw_tiles(float* __restrict__ P, float* __restrict__ M, float* __restrict__ V,
                                            const G* __restrict__ Gr, uint16_t* __restrict__ out, int64_t n,
                                            const int64_t* __restrict__ runs, int64_t nruns, const StepScalars& sc,
                                            zopt_adam_state* state, long long t_new) {
  const int64_t ntiles = (n + kTile - 1) / kTile;
  const int64_t t_begin = ntiles * blockIdx.x / gridDim.x;
  const int64_t t_end = ntiles * (blockIdx.x + 1) / gridDim.x;

  // First no-decay run that ends after this block's first slot (runs are sorted, so their
  // ends are sorted too).
  int64_t cur = 0;
  {
    int64_t lo = 0, hi = nruns;
    const int64_t x0 = t_begin * kTile;
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (__ldg(runs + 2 * mid + 1) <= x0) lo = mid + 1; else hi = mid;
    }
    cur = lo;
  }

  for (int64_t tile = t_begin; tile < t_end; ++tile) {
    const int64_t tb = tile * kTile;
    const int64_t te = (tb + kTile < n) ? tb + kTile : n;
    while (cur < nruns && __ldg(runs + 2 * cur + 1) <= tb) ++cur;
    const bool mixed = cur < nruns && __ldg(runs + 2 * cur) < te;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t x = tb + h * (kThreads * kGroup) + kGroup * threadIdx.x;
      if (x + kGroup <= n) {
        Vec4 p = ld4(P + x), m = ld4(M + x), v = ld4(V + x);
        const Vec4 g = ldg4(Gr + x);
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
          const bool dec = !mixed || !in_nodecay(runs, nruns, cur, te, x + k);
          adamw_elem(p.x[k], m.x[k], v.x[k], g.x[k], dec, sc);
        }
        st4(P + x, p);
        st4(M + x, m);
        st4(V + x, v);
        if (kOut) {
          const uint2 o = make_uint2(static_cast<unsigned int>(bf16_bits(p.x[0])) |
                                         (static_cast<unsigned int>(bf16_bits(p.x[1])) << 16),
                                     static_cast<unsigned int>(bf16_bits(p.x[2])) |
                                         (static_cast<unsigned int>(bf16_bits(p.x[3])) << 16));
          *reinterpret_cast<uint2*>(out + x) = o;
        }
      } else {
        for (int64_t y = x; y < n && y < x + kGroup; ++y) {
          float p = P[y], m = M[y], v = V[y];
          const bool dec = !mixed || !in_nodecay(runs, nruns, cur, te, y);
          adamw_elem(p, m, v, ldg1(Gr + y), dec, sc);
          P[y] = p;
          M[y] = m;
          V[y] = v;
          if (kOut) out[y] = bf16_bits(p);
        }
      }
    }
  }

  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int ticket = atomicAdd(&state->arrive, 1u);
    if (ticket == gridDim.x - 1) {
      state->step = t_new;
      state->arrive = 0u;
      __threadfence();
    }
  }
}

template <typename G, bool kOut>
__global__ void __launch_bounds__(kThreads) adamw_kernel(float* __restrict__ P, float* __restrict__ M,
                                                          float* __restrict__ V, const G* __restrict__ Gr,
                                                          uint16_t* __restrict__ out, int64_t n,
                                                          const int64_t* __restrict__ runs, int64_t nruns,
                                                          HostScalars hs, const zopt_clip_stats* clip,
                                                          zopt_adam_state* state) {
  __shared__ StepScalars s_sc;
  __shared__ int s_skip;
  __shared__ long long s_t;
  if (threadIdx.x == 0) {
    float coef = 1.0f;
    int found = 0;
    if (clip != nullptr) {
      coef = *reinterpret_cast<const volatile float*>(&clip->clip_coef);
      found = *reinterpret_cast<const volatile uint8_t*>(&clip->found_inf);
    }
    step_scalars(hs, coef, found, state, s_sc, s_skip, s_t);
  }
  __syncthreads();
  if (s_skip) return;  // uniform over the grid: nothing is written, the counter stays
  const StepScalars sc = s_sc;
  adamw_tiles<G, kOut>(P, M, V, Gr, out, n, runs, nruns, sc, state, s_t);
}

// ---- the norm / clip reduction and the step in one launch (zopt_adamw_clip_step)
//
// A cooperative launch of one wave: each block sums the squares of its own run of tiles (the
// run it then updates; fp32 pairwise over runs of 32 squares, exact fp64 outside the safe
// range, the runs in fp64, as the norm pass does), publishes the sum, and waits at a grid-wide
// barrier; then every block adds all the blocks' sums in the same fixed order, so every block
// holds the same sum of squares, norm, clip coefficient and found_inf (block 0 also writes them
// out), and the step runs as adamw_kernel's. The gradient is read twice; the second read finds
// it in L2 only where the update's own stream has not evicted it first (a small shard).
constexpr int64_t kClipMaxBlocks = 4096;  // partial sums the workspace holds

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Sum of squares of g[e0, e1) over the block (per thread; e0 16-byte aligned).
template <typename G>
__device__ __forceinline__ double range_sumsq(const G* __restrict__ g, int64_t e0, int64_t e1) {
  const int64_t nv = (e1 - e0) / 8;
  const G* base = g + e0;
  double acc = 0.0;
  int64_t j = threadIdx.x;
  for (; j + 3 * kThreads < nv; j += 4 * kThreads) {
    Raw8<G> r[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) ld_raw8(base + 8 * (j + k * kThreads), r[k]);
    float x0[8], x1[8], x2[8], x3[8];
    unpack8(r[0], x0);
    unpack8(r[1], x1);
    unpack8(r[2], x2);
    unpack8(r[3], x3);
    acc = __dadd_rn(acc, sumsq32(x0, x1, x2, x3));
  }
  for (; j < nv; j += kThreads) {
    float x[8];
    load8(base + 8 * j, x);
    acc = __dadd_rn(acc, sumsq8(x));
  }
  if (threadIdx.x == 0)
    for (int64_t k = e0 + 8 * nv; k < e1; ++k) {
      const double d = static_cast<double>(load1(g + k));
      acc = __dadd_rn(acc, __dmul_rn(d, d));
    }
  return acc;
}

template <typename G, bool kOut>
__global__ void __launch_bounds__(kThreads) adamw_clip_kernel(float* __restrict__ P, float* __restrict__ M,
                                                               float* __restrict__ V, const G* __restrict__ Gr,
                                                               uint16_t* __restrict__ out, int64_t n,
                                                               const int64_t* __restrict__ runs, int64_t nruns,
                                                               HostScalars hs, float max_norm, NormWorkspace* ws,
                                                               zopt_clip_stats* clip, zopt_adam_state* state,
                                                               int* err) {
  __shared__ double red[32];
  __shared__ int s_ok;
  __shared__ StepScalars s_sc;
  __shared__ int s_skip;
  __shared__ long long s_t;
  const int64_t ntiles = (n + kTile - 1) / kTile;
  const int64_t e0 = kTile * (ntiles * blockIdx.x / gridDim.x);
  const int64_t e1c = kTile * (ntiles * (blockIdx.x + 1) / gridDim.x);
  const int64_t e1 = e1c < n ? e1c : n;
  const double block = block_sum(range_sumsq(Gr, e0, e1), red);
  unsigned* depart = &ws->reserved[0];
  if (threadIdx.x == 0) {
    ws->partials[blockIdx.x] = block;
    __threadfence();
    atomicAdd(&ws->arrive, 1u);
    // every block is resident (cooperative launch); the wait is bounded all the same
    int ok = 1;
    if (ld_acquire_u32(&ws->arrive) < gridDim.x) {
      const unsigned long long t0 = global_ns();
      for (unsigned spin = 1;; ++spin) {
        __nanosleep(64);
        if (ld_acquire_u32(&ws->arrive) >= gridDim.x) break;
        if ((spin & 63u) == 0 && global_ns() - t0 > 4000000000ull) {
          atomicExch(err, 1);
          ok = 0;
          break;
        }
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  if (!s_ok) return;  // the error word reports it; this block updates nothing
  double a = 0.0;
  const volatile double* parts = ws->partials;
  for (unsigned int i = threadIdx.x; i < gridDim.x; i += blockDim.x) a = __dadd_rn(a, parts[i]);
  const double ss = block_sum(a, red);
  if (threadIdx.x == 0) {
    // the partials have been read: the last block past this point re-zeroes both counters
    if (atomicAdd(depart, 1u) == gridDim.x - 1) {
      ws->arrive = 0u;
      *depart = 0u;
      __threadfence();
    }
    zopt_clip_stats st;
    write_clip_stats(&st, ss, max_norm);
    if (blockIdx.x == 0) *clip = st;
    step_scalars(hs, st.clip_coef, st.found_inf, state, s_sc, s_skip, s_t);
  }
  __syncthreads();
  if (s_skip) return;  // uniform over the grid: nothing is written, the counter stays
  const StepScalars sc = s_sc;
  adamw_tiles<G, kOut>(P, M, V, Gr, out, n, runs, nruns, sc, state, s_t);
}

template <typename G, bool kOut>
zopt_status launch_clip(const HostScalars& hs, float* P, float* M, float* V, const void* g, uint16_t* out, int64_t n,
                        const int64_t* runs, int64_t nruns, float max_norm, NormWorkspace* ws, zopt_clip_stats* clip,
                        zopt_adam_state* state, int* err, cudaStream_t stream) {
  const int occ = once([] {  // resident blocks per SM for this instantiation
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, adamw_clip_kernel<G, kOut>, kThreads, 0) != cudaSuccess ||
        o < 1)
      o = 1;
    return o < kBlocksPerSm ? o : kBlocksPerSm;
  });
  const int sms = sm_count();
  if (sms <= 0) return fail(ZOPT_ECUDA, "zopt_adamw_clip_step: no CUDA device");
  const int64_t ntiles = (n + kTile - 1) / kTile;
  int64_t blocks = static_cast<int64_t>(sms) * occ;  // one wave: every block resident
  if (blocks > ntiles) blocks = ntiles;
  if (blocks > kClipMaxBlocks) blocks = kClipMaxBlocks;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ZOPT_CUDA_TRY(cudaLaunchKernelEx(&cfg, adamw_clip_kernel<G, kOut>, P, M, V, static_cast<const G*>(g), out, n, runs,
                                   nruns, hs, max_norm, ws, clip, state, err));
  return ok();
}

template <typename G, bool kOut>
zopt_status launch(const HostScalars& hs, float* P, float* M, float* V, const void* g, uint16_t* out, int64_t n,
                   const int64_t* runs, int64_t nruns, const zopt_clip_stats* clip, zopt_adam_state* state,
                   cudaStream_t stream) {
  const int occ = once([] {  // resident blocks per SM for this instantiation
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, adamw_kernel<G, kOut>, kThreads, 0) != cudaSuccess || o < 1)
      o = kBlocksPerSm;
    return o < kBlocksPerSm ? o : kBlocksPerSm;
  });
  const int sms = sm_count();
  if (sms <= 0) return fail(ZOPT_ECUDA, "zopt_adamw_step: no CUDA device");
  const int64_t ntiles = (n + kTile - 1) / kTile;
  int64_t blocks = static_cast<int64_t>(sms) * occ;
  if (blocks > ntiles) blocks = ntiles;
  adamw_kernel<G, kOut><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
      P, M, V, static_cast<const G*>(g), out, n, runs, nruns, hs, clip, state);
  ZOPT_CUDA_TRY(cudaGetLastError());
  return ok();
}

}  // namespace
}  // namespace zopt

namespace zopt {
namespace {

// Checks the arguments shared by zopt_adamw_step and zopt_adamw_clip_step and forms the
// step-independent scalars: fp64 expressions rounded once to fp32 (the host build uses
// -ffp-contract=off, so 1 - lr*wd is two roundings, as written).
zopt_status prepare_step(const char* fn, const zopt_layout* layout, const int64_t* d_nodecay_runs, float* master,
                         float* exp_avg, float* exp_avg_sq, const void* grad, zopt_dtype grad_dtype,
                         uint16_t* out_bf16, const zopt_adamw_hparams* hp, const zopt_clip_stats* d_clip,
                         zopt_adam_state* d_state, HostScalars& hs, int64_t& nruns) {
  const std::string f(fn);
  if (layout == nullptr || hp == nullptr) return fail(ZOPT_EINVAL, f + ": layout or hparams is NULL");
  if (master == nullptr || exp_avg == nullptr || exp_avg_sq == nullptr || grad == nullptr || d_state == nullptr)
    return fail(ZOPT_EINVAL, f + ": NULL device pointer");
  if (!aligned16(master) || !aligned16(exp_avg) || !aligned16(exp_avg_sq) || !aligned16(grad) ||
      (out_bf16 != nullptr && !aligned16(out_bf16)) || !aligned16(d_state) ||
      (d_clip != nullptr && (reinterpret_cast<uintptr_t>(d_clip) & 7u) != 0))
    return fail(ZOPT_EINVAL, f + ": a device pointer is not 16-byte aligned");
  nruns = static_cast<int64_t>(layout->nodecay.size() / 2);
  if (nruns > 0 && (d_nodecay_runs == nullptr || (reinterpret_cast<uintptr_t>(d_nodecay_runs) & 7u) != 0))
    return fail(ZOPT_EINVAL, f + ": the layout has no-decay runs but d_nodecay_runs is NULL/misaligned");
  if (grad_dtype != ZOPT_F32 && grad_dtype != ZOPT_BF16)
    return fail(ZOPT_EUNSUPPORTED, f + ": gradient dtype must be fp32 or bf16 (fp32 master)");
  const double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, eps = hp->eps, wd = hp->weight_decay;
  if (!std::isfinite(lr) || lr < 0.0) return fail(ZOPT_EINVAL, f + ": lr must be finite and >= 0");
  if (!(b1 >= 0.0 && b1 < 1.0) || !(b2 >= 0.0 && b2 < 1.0)) return fail(ZOPT_EINVAL, f + ": betas must lie in [0, 1)");
  if (!std::isfinite(eps) || eps < 0.0) return fail(ZOPT_EINVAL, f + ": eps must be finite and >= 0");
  if (!std::isfinite(wd)) return fail(ZOPT_EINVAL, f + ": weight_decay must be finite");
  hs.b1 = static_cast<float>(b1);
  hs.omb1 = static_cast<float>(1.0 - b1);
  hs.b2 = static_cast<float>(b2);
  hs.omb2 = static_cast<float>(1.0 - b2);
  hs.eps = static_cast<float>(eps);
  const double lrwd = lr * wd;
  hs.decay = static_cast<float>(1.0 - lrwd);
  hs.lr = lr;
  hs.beta1 = b1;
  hs.beta2 = b2;
  hs.skip_on_inf = hp->skip_on_inf != 0;
  return ok();
}

}  // namespace
}  // namespace zopt

extern "C" zopt_status zopt_adamw_step(const zopt_layout* layout, const int64_t* d_nodecay_runs, float* master,
                                       float* exp_avg, float* exp_avg_sq, const void* grad, zopt_dtype grad_dtype,
                                       uint16_t* out_bf16, const zopt_adamw_hparams* hp,
                                       const zopt_clip_stats* d_clip, zopt_adam_state* d_state,
                                       zopt_stream stream) {
  using namespace zopt;
  HostScalars hs;
  int64_t nruns = 0;
  zopt_status st = prepare_step("zopt_adamw_step", layout, d_nodecay_runs, master, exp_avg, exp_avg_sq, grad,
                                grad_dtype, out_bf16, hp, d_clip, d_state, hs, nruns);
  if (st != ZOPT_OK) return st;
  const int64_t n = layout->shard_len;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (grad_dtype == ZOPT_BF16) {
    return out_bf16 ? launch<__nv_bfloat16, true>(hs, master, exp_avg, exp_avg_sq, grad, out_bf16, n, d_nodecay_runs,
                                                  nruns, d_clip, d_state, s)
                    : launch<__nv_bfloat16, false>(hs, master, exp_avg, exp_avg_sq, grad, nullptr, n,
                                                   d_nodecay_runs, nruns, d_clip, d_state, s);
  }
  return out_bf16 ? launch<float, true>(hs, master, exp_avg, exp_avg_sq, grad, out_bf16, n, d_nodecay_runs, nruns,
                                        d_clip, d_state, s)
                  : launch<float, false>(hs, master, exp_avg, exp_avg_sq, grad, nullptr, n, d_nodecay_runs, nruns,
                                         d_clip, d_state, s);
}

extern "C" size_t zopt_adamw_clip_workspace(int64_t shard_len) {
  if (shard_len < 1) return 0;
  const int64_t tiles = (shard_len + zopt::adam::kTile - 1) / zopt::adam::kTile;
  const int64_t blocks = tiles < zopt::kClipMaxBlocks ? tiles : zopt::kClipMaxBlocks;
  return static_cast<size_t>(offsetof(zopt::NormWorkspace, partials) + sizeof(double) * blocks);
}

extern "C" zopt_status zopt_adamw_clip_step(const zopt_layout* layout, const int64_t* d_nodecay_runs, float* master,
                                            float* exp_avg, float* exp_avg_sq, const void* grad,
                                            zopt_dtype grad_dtype, uint16_t* out_bf16, const zopt_adamw_hparams* hp,
                                            float max_norm, void* d_ws, size_t ws_bytes, zopt_clip_stats* d_clip,
                                            zopt_adam_state* d_state, zopt_stream stream) {
  using namespace zopt;
  const char* fn = "zopt_adamw_clip_step";
  HostScalars hs;
  int64_t nruns = 0;
  zopt_status st = prepare_step(fn, layout, d_nodecay_runs, master, exp_avg, exp_avg_sq, grad, grad_dtype, out_bf16,
                                hp, d_clip, d_state, hs, nruns);
  if (st != ZOPT_OK) return st;
  if (d_clip == nullptr || d_ws == nullptr) return fail(ZOPT_EINVAL, "zopt_adamw_clip_step: NULL device pointer");
  if (!aligned16(d_ws)) return fail(ZOPT_EINVAL, "zopt_adamw_clip_step: a device pointer is not 16-byte aligned");
  if (!(max_norm >= 0.0f)) return fail(ZOPT_EINVAL, "zopt_adamw_clip_step: max_norm must be >= 0 (not NaN)");
  const int64_t n = layout->shard_len;
  if (n < 1) return fail(ZOPT_EINVAL, "zopt_adamw_clip_step: empty shard");
  if (ws_bytes < zopt_adamw_clip_workspace(n))
    return fail(ZOPT_EINVAL, "zopt_adamw_clip_step: workspace smaller than zopt_adamw_clip_workspace");
  int* err = nullptr;
  if ((st = ns::take_error_word(fn, &err)) != ZOPT_OK) return st;
  NormWorkspace* ws = static_cast<NormWorkspace*>(d_ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (grad_dtype == ZOPT_BF16) {
    return out_bf16 ? launch_clip<__nv_bfloat16, true>(hs, master, exp_avg, exp_avg_sq, grad, out_bf16, n,
                                                       d_nodecay_runs, nruns, max_norm, ws, d_clip, d_state, err, s)
                    : launch_clip<__nv_bfloat16, false>(hs, master, exp_avg, exp_avg_sq, grad, nullptr, n,
                                                        d_nodecay_runs, nruns, max_norm, ws, d_clip, d_state, err, s);
  }
  return out_bf16 ? launch_clip<float, true>(hs, master, exp_avg, exp_avg_sq, grad, out_bf16, n, d_nodecay_runs,
                                             nruns, max_norm, ws, d_clip, d_state, err, s)
                  : launch_clip<float, false>(hs, master, exp_avg, exp_avg_sq, grad, nullptr, n, d_nodecay_runs,
                                              nruns, max_norm, ws, d_clip, d_state, err, s);
}
