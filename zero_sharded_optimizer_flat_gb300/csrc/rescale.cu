// Rescale of a taken AdamW step to a new gradient scale (DeepSpeed PR #9021, adam_rescale_step
// commit): given the weights and moments after step t on g * old_scale, write those of step t
// on g * new_scale from the same starting point, in one pass over the shard.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "adam_common.cuh"
#include "internal.h"

namespace zopt {
namespace {

using namespace adam;

// Per element: m += (1-b1)(new-old)g; v = max(0, v + (1-b2)(new^2-old^2)g^2) (a NaN stays NaN);
// p += step_size*(m_old/d_old - m_new/d_new) (the decoupled decay does not depend on g).

struct RescaleHost {
  double beta1, beta2, lr, old_scale, new_scale;
  float eps;
};

// x / c, correctly rounded, for the launch's constant c = sqrt(1 - beta2^t) in (0, 1] given
// rc = RN(1 / c) (__frcp_rn): Markstein's correction (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Develop. 34(1), 1990). With rc
// correctly rounded, q = RN(x rc) is within one ulp of x / c, the residual x - q c is exact
// through an FMA, and RN(q + (x - q c) rc) = RN(x / c) as long as nothing overflows or
// underflows, which holds for every x = sqrt(v) (v >= 0: x is 0, normal, +inf or NaN). Zero
// and infinity pass through (the residual of an infinity would be NaN). Checked against
// __fdiv_rn for every v bit pattern by zopt_selftest_div_by_const.
__device__ __forceinline__ float div_by_const(float x, float c, float rc) {
  const float q = __fmul_rn(x, rc);
  const float e = __fmaf_rn(-q, c, x);
  const float r = __fmaf_rn(e, rc, q);
  return (x == 0.0f || isinf(x)) ? x : r;
}

// m / (sqrt(v) / bc2s + eps), each operation correctly rounded (bc2s: rc = RN(1 / bc2s)).
__device__ __forceinline__ float adam_dir(float m, float v, float bc2s, float rc, float eps) {
  return __fdiv_rn(m, __fadd_rn(div_by_const(__fsqrt_rn(v), bc2s, rc), eps));
}

// Tiles of kTile elements, as adamw_kernel walks them: a thread holds 2 x 4 elements of each
// array, all eight loads issued before any arithmetic, so 128 bytes per thread are in flight
// (the two update directions per element make this kernel's arithmetic twice the step's).
template <typename G, bool kOut>
__global__ void __launch_bounds__(kThreads, kBlocksPerSm) rescale_kernel(float* __restrict__ P, float* __restrict__ M,
                                                                         float* __restrict__ V, const G* __restrict__ Gr,
                                                                         uint16_t* __restrict__ out, int64_t n,
                                                                         RescaleHost hs, const zopt_clip_stats* clip,
                                                                         const zopt_adam_state* state) {
  __shared__ float s_km, s_kv, s_step, s_bc2s, s_rc;
  __shared__ int s_skip;
  if (threadIdx.x == 0) {
    const long long t = *reinterpret_cast<const volatile long long*>(&state->step);
    double nw = hs.new_scale;
    int skip = t < 1 ? 1 : 0;  // no step has been taken yet: nothing to re-target
    if (clip != nullptr) {
      nw = static_cast<double>(*reinterpret_cast<const volatile float*>(&clip->clip_coef));
      if (*reinterpret_cast<const volatile uint8_t*>(&clip->found_inf)) skip = 1;
    }
    const double od = hs.old_scale;
    s_km = __double2float_rn(__dmul_rn(__dsub_rn(1.0, hs.beta1), __dsub_rn(nw, od)));
    s_kv = __double2float_rn(__dmul_rn(__dsub_rn(1.0, hs.beta2), __dsub_rn(__dmul_rn(nw, nw), __dmul_rn(od, od))));
    const double bc1 = __dsub_rn(1.0, pow_sq_mul(hs.beta1, t));
    const double bc2 = __dsub_rn(1.0, pow_sq_mul(hs.beta2, t));
    s_step = __double2float_rn(__ddiv_rn(hs.lr, bc1));
    s_bc2s = __double2float_rn(__dsqrt_rn(bc2));
    s_rc = __frcp_rn(s_bc2s);
    s_skip = skip;
  }
  __syncthreads();
  if (s_skip) return;
  const float km = s_km, kv = s_kv, step = s_step, bc2s = s_bc2s, rc = s_rc, eps = hs.eps;
  auto one = [&](float& p, float& m, float& v, float g) {
    const float u_old = adam_dir(m, v, bc2s, rc, eps);
    m = __fadd_rn(m, __fmul_rn(km, g));
    const float vv = __fadd_rn(v, __fmul_rn(kv, __fmul_rn(g, g)));
    v = vv < 0.0f ? 0.0f : vv;
    const float u_new = adam_dir(m, v, bc2s, rc, eps);
    p = __fadd_rn(p, __fmul_rn(step, __fsub_rn(u_old, u_new)));
  };
  auto put_bf16 = [&](int64_t x, const Vec4& p) {
    *reinterpret_cast<uint2*>(out + x) =
        make_uint2(static_cast<unsigned int>(bf16_bits(p.x[0])) | (static_cast<unsigned int>(bf16_bits(p.x[1])) << 16),
                   static_cast<unsigned int>(bf16_bits(p.x[2])) | (static_cast<unsigned int>(bf16_bits(p.x[3])) << 16));
  };
  const int64_t nfull = n / kTile;  // whole tiles; the tail below
  for (int64_t tile = blockIdx.x; tile < nfull; tile += gridDim.x) {
    const int64_t x0 = tile * kTile + kGroup * threadIdx.x, x1 = x0 + kThreads * kGroup;
    Vec4 p0 = ld4(P + x0), m0 = ld4(M + x0), v0 = ld4(V + x0);
    Vec4 p1 = ld4(P + x1), m1 = ld4(M + x1), v1 = ld4(V + x1);
    const Vec4 g0 = ldg4(Gr + x0), g1 = ldg4(Gr + x1);
#pragma unroll
    for (int k = 0; k < kGroup; ++k) one(p0.x[k], m0.x[k], v0.x[k], g0.x[k]);
    st4(P + x0, p0);
    st4(M + x0, m0);
    st4(V + x0, v0);
    if (kOut) put_bf16(x0, p0);
#pragma unroll
    for (int k = 0; k < kGroup; ++k) one(p1.x[k], m1.x[k], v1.x[k], g1.x[k]);
    st4(P + x1, p1);
    st4(M + x1, m1);
    st4(V + x1, v1);
    if (kOut) put_bf16(x1, p1);
  }
  // the last partial tile, one element per thread at a time, by the block after the last whole one
  if (static_cast<int64_t>(blockIdx.x) == nfull % gridDim.x) {
    for (int64_t k = nfull * kTile + threadIdx.x; k < n; k += kThreads) {
      float p = P[k], m = M[k], v = V[k];
      one(p, m, v, ldg1(Gr + k));
      P[k] = p;
      M[k] = m;
      V[k] = v;
      if (kOut) out[k] = bf16_bits(p);
    }
  }
}

template <typename G, bool kOut>
zopt_status launch_rescale(const RescaleHost& hs, float* P, float* M, float* V, const void* g, uint16_t* out,
                           int64_t n, const zopt_clip_stats* clip, const zopt_adam_state* state, cudaStream_t s) {
  const int sms = sm_count();
  if (sms <= 0) return fail(ZOPT_ECUDA, "zopt_adamw_rescale_step: no CUDA device");
  int64_t blocks = (n + kTile - 1) / kTile;
  if (blocks > static_cast<int64_t>(sms) * kBlocksPerSm) blocks = static_cast<int64_t>(sms) * kBlocksPerSm;
  if (blocks < 1) blocks = 1;
  rescale_kernel<G, kOut><<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(P, M, V, static_cast<const G*>(g), out,
                                                                             n, hs, clip, state);
  ZOPT_CUDA_TRY(cudaGetLastError());
  return ok();
}

// div_by_const(sqrt(v), c, RN(1 / c)) against __fdiv_rn(sqrt(v), c) for every bit pattern of
// v >= 0 (and the positive NaNs): the count of results that differ (NaN matching NaN).
__global__ void __launch_bounds__(256) div_selftest_kernel(float c, unsigned long long* mismatches) {
  const float rc = __frcp_rn(c);
  unsigned long long bad = 0;
  const unsigned int stride = gridDim.x * blockDim.x;
  for (unsigned int b = blockIdx.x * blockDim.x + threadIdx.x; b < 0x80000000u; b += stride) {
    const float x = __fsqrt_rn(__uint_as_float(b));
    const float fast = div_by_const(x, c, rc), ref = __fdiv_rn(x, c);
    const bool same = __float_as_uint(fast) == __float_as_uint(ref) || (isnan(fast) && isnan(ref));
    bad += same ? 0u : 1u;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xFFFFFFFFu, bad, o);
  if ((threadIdx.x & 31) == 0 && bad != 0) atomicAdd(mismatches, bad);
}

}  // namespace
}  // namespace zopt

extern "C" zopt_status zopt_selftest_div_by_const(float c, unsigned long long* d_mismatches, zopt_stream stream) {
  using namespace zopt;
  if (d_mismatches == nullptr || (reinterpret_cast<uintptr_t>(d_mismatches) & 7u) != 0)
    return fail(ZOPT_EINVAL, "zopt_selftest_div_by_const: counter is NULL or misaligned");
  if (!(c > 0.0f && c <= 1.0f)) return fail(ZOPT_EINVAL, "zopt_selftest_div_by_const: c must lie in (0, 1]");
  const int sms = sm_count();
  if (sms <= 0) return fail(ZOPT_ECUDA, "zopt_selftest_div_by_const: no CUDA device");
  div_selftest_kernel<<<static_cast<unsigned>(sms * 8), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      c, d_mismatches);
  ZOPT_CUDA_TRY(cudaGetLastError());
  return ok();
}

extern "C" zopt_status zopt_adamw_rescale_step(const zopt_layout* layout, float* master, float* exp_avg,
                                               float* exp_avg_sq, const void* grad, zopt_dtype grad_dtype,
                                               uint16_t* out_bf16, const zopt_adamw_hparams* hp, float old_scale,
                                               float new_scale, const zopt_clip_stats* d_clip,
                                               const zopt_adam_state* d_state, zopt_stream stream) {
  using namespace zopt;
  if (layout == nullptr || hp == nullptr) return fail(ZOPT_EINVAL, "zopt_adamw_rescale_step: layout or hparams is NULL");
  if (master == nullptr || exp_avg == nullptr || exp_avg_sq == nullptr || grad == nullptr || d_state == nullptr)
    return fail(ZOPT_EINVAL, "zopt_adamw_rescale_step: NULL device pointer");
  if (!aligned16(master) || !aligned16(exp_avg) || !aligned16(exp_avg_sq) || !aligned16(grad) ||
      (out_bf16 != nullptr && !aligned16(out_bf16)) || (reinterpret_cast<uintptr_t>(d_state) & 7u) != 0 ||
      (d_clip != nullptr && (reinterpret_cast<uintptr_t>(d_clip) & 7u) != 0))
    return fail(ZOPT_EINVAL, "zopt_adamw_rescale_step: a device pointer is misaligned");
  if (grad_dtype != ZOPT_F32 && grad_dtype != ZOPT_BF16)
    return fail(ZOPT_EUNSUPPORTED, "zopt_adamw_rescale_step: gradient dtype must be fp32 or bf16");
  if (!std::isfinite(hp->lr) || hp->lr < 0.0 || !(hp->beta1 >= 0.0 && hp->beta1 < 1.0) ||
      !(hp->beta2 >= 0.0 && hp->beta2 < 1.0) || !std::isfinite(hp->eps) || hp->eps < 0.0)
    return fail(ZOPT_EINVAL, "zopt_adamw_rescale_step: hyper-parameters out of range");
  if (!std::isfinite(old_scale) || (d_clip == nullptr && !std::isfinite(new_scale)))
    return fail(ZOPT_EINVAL, "zopt_adamw_rescale_step: scales must be finite");
  RescaleHost hs{hp->beta1, hp->beta2, hp->lr, static_cast<double>(old_scale), static_cast<double>(new_scale),
                 static_cast<float>(hp->eps)};
  const int64_t n = layout->shard_len;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (grad_dtype == ZOPT_BF16)
    return out_bf16 ? launch_rescale<__nv_bfloat16, true>(hs, master, exp_avg, exp_avg_sq, grad, out_bf16, n, d_clip,
                                                          d_state, s)
                    : launch_rescale<__nv_bfloat16, false>(hs, master, exp_avg, exp_avg_sq, grad, nullptr, n, d_clip,
                                                           d_state, s);
  return out_bf16 ? launch_rescale<float, true>(hs, master, exp_avg, exp_avg_sq, grad, out_bf16, n, d_clip, d_state, s)
                  : launch_rescale<float, false>(hs, master, exp_avg, exp_avg_sq, grad, nullptr, n, d_clip, d_state,
                                                 s);
}
