// Muon's quintic Newton-Schulz orthogonalisation on whole matrices, on tcgen05 tensor cores:
// the workspace plan, the tensor maps, the entry points and the failure self-tests.
//
// bluscript_zero_ckpt.cpp, ShardedMuon design note: U = NewtonSchulz(M), the iterated matrix
// polynomial X <- aX + (bXX' + c(XX')^2)X, in which every output entry depends on the whole
// matrix (so each matrix has one owner rank); 5 steps in the trainer's config.
//
// Per step, with X m x n (m <= n; a taller input is processed as its transpose):
//   A = X X'            (symmetric: only the tiles touching the upper triangle are computed,
//                        each writes its upper part and, transposed, its mirror)
//   B' = c A A' + b A + a I
//                       (A is symmetric, so A^2 = A A': the same symmetric kernel, with the
//                        b*A term and a on the diagonal added to the accumulator)
//   X = B' X            (= aX + BX: the step's aX term rides on B's diagonal, so the largest
//                        product has no second input to read; a plain GEMM whose B-operand X
//                        is read MN-major straight from its row-major layout; the last step
//                        writes the caller's output, in the caller's orientation and dtype)
// Operands and the products A, B', X are bf16; every product accumulates in fp32 in TMEM.
// The fp32 compute mode runs the products as the pages write them on the SIMT kernel
// (ns_simt.cu).
//
// Where the work runs: ns_prep.cu normalises and orients the inputs of every job in three
// launches; below m = 1024 every product of every step runs in one persistent launch of
// ns_fused_kernel (ns_fused.cu), several shapes at once; from m = 1024 each product of a step is
// one launch of the CTA-pair GEMM for up to four shapes (in a call that has such shapes, those
// from m = 512 join them), and where an output or the coefficients rule the fused kernel out,
// one launch of the single-CTA GEMM (ns_gemm.cu). The
// tile geometry and the epilogue building blocks they share are in ns_tile.cuh. Every wait is
// bounded; a timeout sets an error word that the next call reports as ZOPT_ETIMEOUT.
// Callers inside the library (the Muon step) may hand a job's norm partials already summed, or
// its X0 already in place and unnormalised (then one small launch turns the partials into the
// scale that the first step's X X' and B'X epilogues apply), and may collect the statistics of
// the last product's output from its epilogue (orthogonalize_many).
#include <cstring>

#include "ns_tile.cuh"

namespace zopt {
namespace ns {

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

// Fill the derived fields and encode the maps of a group whose workspace is at ws (plan p).
zopt_status group_init(Group& G, const Plan& p, uint8_t* ws) {
  zopt_status st = ZOPT_OK;
  G.p = p;
  G.es = G.f32c ? 4 : 2;
  G.esz = G.io == ZOPT_F32 ? 4 : 2;
  G.osz = G.out_io == ZOPT_F32 ? 4 : 2;
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
  const long long osz = static_cast<long long>(G.osz);
  G.out_tma = !G.f32c && (reinterpret_cast<uintptr_t>(G.xo) & 15u) == 0 && (G.ld_x * osz) % 16 == 0 &&
              (G.gs == 1 || (G.bs_x * osz) % 16 == 0);
  G.g_in_place = false;
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
  // A bf16 input in X's orientation whose rows and matrices the TMA can address is read in
  // place by the first step, which also normalises it: no copy of it into X0.
  G.g_in_place = !G.x0_raw && G.io == ZOPT_BF16 && !G.transpose && (reinterpret_cast<uintptr_t>(G.g) & 15u) == 0 &&
                 (G.ld_g * 2) % 16 == 0 && (G.gs == 1 || (G.bs_g * 2) % 16 == 0);
  if (G.g_in_place) {
    const long long gb = (G.gs == 1 ? p.m * G.ld_g : G.bs_g) * 2;
    if ((st = make_map(&G.mg_p, G.g, p.n, p.m, G.ld_g, G.gs, gb, 64, BM)) != ZOPT_OK) return st;
    if ((st = make_map(&G.mg_q, G.g, p.n, p.m, G.ld_g, G.gs, gb, 64, BN)) != ZOPT_OK) return st;
    if ((st = make_map(&G.mg_mn, G.g, p.n, p.m, G.ld_g, G.gs, gb, 64, BK)) != ZOPT_OK) return st;
  }
  if (G.out_tma) {
    const long long xrows = G.transpose ? p.n : p.m, xcols = G.transpose ? p.m : p.n;  // the caller's shape
    const long long ob = (G.gs == 1 ? xrows * G.ld_x : G.bs_x) * osz;
    const bool of32 = G.out_io == ZOPT_F32;
    if ((st = make_map(&G.mo_e, G.xo, xcols, xrows, G.ld_x, G.gs, ob, 32, 32,
                       of32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, of32)) != ZOPT_OK)
      return st;
  }
  return ok();
}

// Whether every product of the group can run in the fused kernel.
bool group_fusable(const Group& G, const Coef& k) { return !G.f32c && !G.pair && G.out_tma && k.id_ok; }

// The group as one job of the fused kernel.
// Matrix 0's factor for the first step's products of a group whose X0 arrives unnormalised
// (matrix b's kScaleStride floats on): 1 / (||X0|| + eps), squared for X X'.
constexpr long long kScaleStride = static_cast<long long>(kPrepWsBytes / sizeof(float));
const float* x0_scale(const Group& G, bool squared) {
  return reinterpret_cast<const float*>(G.ws) + kScaleWord + (squared ? 1 : 0);
}

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
  if (G.g_in_place) {
    m.gp = G.mg_p;
    m.gq = G.mg_q;
    m.gmn = G.mg_mn;
  }
  job.x0_is_g = G.g_in_place ? 1 : 0;
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
  if (first_scales(G)) {  // the first step normalises: A by 1 / (||X0|| + eps)^2, B'X by 1 / (||X0|| + eps)
    pa.amat = x0_scale(G, true);
    px.amat = x0_scale(G, false);
    pa.amat_stride = px.amat_stride = kScaleStride;
  }
  job.prod[3] = px;  // the last step's, into the caller's X
  job.prod[3].d_f32 = G.out_io == ZOPT_F32 ? 1 : 0;
  job.prod[3].d_trans = G.transpose ? 1 : 0;
  job.prep = G.ws;
}

// Product `prod` of a step of a CTA-pair group as a job of a pair launch: 0 A = X X', 1 B' =
// c A A' + b A + a I (b A through the R epilogue), 2 X = B' X (into the caller's X at the last
// step). X is in buffer `cur`; `first`: the call's first step (which normalises an X0 that
// arrives unnormalised). Returns the product's epilogue.
int pair_job(const Group& G, const Coef& k, int prod, bool first, bool last, int cur, int* err, PairJob& J) {
  const int m = static_cast<int>(G.p.m), n = static_cast<int>(G.p.n);
  const long long mat_elems = G.mat_elems;
  GemmArgs& a = J.a;
  a = GemmArgs{};
  a.err = err;
  a.group = G.gs;
  a.alpha = 1.0f;
  if (first && first_scales(G) && prod != 1) {
    a.amat = x0_scale(G, prod == 0);
    a.amat_stride = kScaleStride;
  }
  if (prod == 0) {
    a.M = m; a.N = m; a.K = n; a.symmetric = 1;
    a.D = G.A; a.ldd = G.p.lda; a.d_stride = mat_elems;
    J.P = J.Q = J.R = first && G.g_in_place ? G.mg_p : G.mx_p[cur];
    J.D = G.ma_e;
    return kEpiTma;
  }
  if (prod == 1) {
    a.M = m; a.N = m; a.K = m; a.symmetric = 1;
    a.alpha = k.c; a.beta = k.b; a.diag = k.a;
    a.R = reinterpret_cast<const __nv_bfloat16*>(G.A); a.ldr = G.p.lda; a.r_stride = mat_elems;
    a.D = G.B; a.ldd = G.p.lda; a.d_stride = mat_elems;
    J.P = J.Q = G.ma_p;
    J.R = G.ma_e;
    J.D = G.mb_e;
    return kEpiTmaR;
  }
  a.M = m; a.N = n; a.K = m; a.b_mn_major = 1;
  a.D = last ? static_cast<void*>(G.xo) : static_cast<void*>(G.xb[cur ^ 1]);
  a.ldd = last ? G.ld_x : G.p.ldx;
  a.d_stride = last ? G.bs_x : mat_elems;
  a.d_f32 = last && G.out_io == ZOPT_F32 ? 1 : 0;
  a.d_trans = last && G.transpose ? 1 : 0;
  J.P = G.mb_p;
  J.Q = J.R = first && G.g_in_place ? G.mg_mn : G.mx_mn[cur];
  J.D = last ? G.mo_e : G.mx_e[cur ^ 1];
  return (!last || G.out_tma) ? kEpiTma : kEpiRegs;
}

// The smallest m that joins the CTA-pair launches of a call that has them anyway.
constexpr long long kPairRideMin = 512;

// The steps of several CTA-pair groups (bf16 compute), each product of a step one launch for
// all of them (kMaxPairJobs groups to a launch, those with the same epilogue together): the
// small groups' tiles fill the large ones' waves. Every tile is computed as in a launch of its
// own group alone, so the results are bitwise those of separate launches.
// sinks (optional, one per group): where the last product of the last step writes its output's
// statistics (a TMA epilogue only).
zopt_status pair_products(const std::vector<const Group*>& gs, const Coef& k, int steps, int* err, cudaStream_t s,
                          const std::vector<const StatsSink*>* sinks = nullptr) {
  zopt_status st = ZOPT_OK;
  int cur = 0;
  for (int it = 0; it < steps; ++it) {
    const bool last = it == steps - 1;
    for (int prod = 0; prod < 3; ++prod) {
      for (const int epi : {kEpiTma, kEpiTmaR, kEpiRegs}) {
        PairBatch B;
        std::memset(&B, 0, sizeof(B));
        for (size_t q = 0; q <= gs.size(); ++q) {
          if (B.n == kMaxPairJobs || (q == gs.size() && B.n > 0)) {
            if ((st = launch_gemm_pair_batch(B, epi, s)) != ZOPT_OK) return st;
            B.n = 0;
          }
          if (q == gs.size()) break;
          PairJob J;
          if (pair_job(*gs[q], k, prod, it == 0, last, cur, err, J) == epi) {
            const StatsSink* sk = sinks != nullptr ? (*sinks)[q] : nullptr;
            if (sk != nullptr && last && prod == 2 && epi == kEpiTma) {
              J.a.st_sum = sk->sum;
              J.a.st_max = sk->max;
              J.a.st_stride = sk->stride;
            }
            B.job[B.n++] = J;
          }
        }
      }
    }
    cur ^= 1;
  }
  return ok();
}

long long stats_slots_bound(long long rows, long long cols) {
  const long long m = rows < cols ? rows : cols, n = rows < cols ? cols : rows;
  // single-CTA tiles (128 x 256) outnumber CTA-pair tiles (256 x 256); 8 epilogue warps a tile
  return 8 * ((m + BM - 1) / BM) * ((n + BN - 1) / BN);
}

// The group's products one launch at a time (the fp32 mode, the CTA-pair kernel, single-CTA
// outputs the TMA cannot address).
zopt_status group_products(const Group& G, const Coef& k, int steps, int* err, cudaStream_t s) {
  if (G.pair && !G.f32c) return pair_products({&G}, k, steps, err, s);
  zopt_status st = ZOPT_OK;
  const int m = static_cast<int>(G.p.m), n = static_cast<int>(G.p.n), gs = G.gs;
  const long long mat_elems = G.mat_elems;
  const Plan& p = G.p;
  int cur = 0;
  for (int it = 0; it < steps; ++it) {
    const bool last = it == steps - 1;
    void* xnext = last ? static_cast<void*>(G.xo) : static_cast<void*>(G.xb[cur ^ 1]);
    const long long ldnext = last ? G.ld_x : p.ldx;
    const long long dstr_next = last ? G.bs_x : mat_elems;
    const int next_f32 = last ? (G.out_io == ZOPT_F32 ? 1 : 0) : (G.f32c ? 1 : 0);
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
      const bool norm_here = it == 0 && first_scales(G);  // this step normalises X0
      const bool from_g = it == 0 && G.g_in_place;       // and reads it from the caller's G
      ga.amat_stride = kScaleStride;
      // A = X X'
      ga.amat = norm_here ? x0_scale(G, true) : nullptr;
      ga.M = m; ga.N = m; ga.K = n;
      ga.symmetric = 1; ga.b_mn_major = 0; ga.alpha = 1.0f; ga.beta = 0.0f; ga.diag = 0.0f; ga.R = nullptr;
      ga.ldr = 0; ga.r_stride = 0; ga.D = G.A; ga.ldd = p.lda; ga.d_stride = mat_elems; ga.d_f32 = 0; ga.d_trans = 0;
      if ((st = launch_gemm(from_g ? G.mg_p : G.mx_p[cur], from_g ? G.mg_q : G.mx_q[cur], nullptr, &G.ma_e, kEpiTma, ga,
                            s)) != ZOPT_OK)
        return st;
      // B' = c A A' + b A + a I: the step's a X term joins the last product as (B + a I) X.
      // On single CTAs b A rides in the accumulator as c (h1 + h2) A (identity MMAs, h1 + h2 =
      // b / c to about 2^-18), so B' needs no second input and keeps the four-stage ring.
      ga.K = m;
      ga.amat = nullptr;
      ga.alpha = k.c; ga.beta = k.b; ga.diag = k.a;
      ga.R = reinterpret_cast<const __nv_bfloat16*>(G.A); ga.ldr = p.lda; ga.r_stride = mat_elems;
      ga.D = G.B; ga.ldd = p.lda; ga.d_stride = mat_elems;
      if (k.id_ok) {
        GemmArgs gi = ga;
        gi.beta = 0.0f; gi.R = nullptr; gi.ident = 1; gi.h1 = k.h1; gi.h2 = k.h2;
        st = launch_gemm(G.ma_p, G.ma_q, nullptr, &G.mb_e, kEpiTma, gi, s);
      } else {
        st = launch_gemm(G.ma_p, G.ma_q, &G.ma_e, &G.mb_e, kEpiTmaR, ga, s);
      }
      if (st != ZOPT_OK) return st;
      // X = B' X
      ga.amat = norm_here ? x0_scale(G, false) : nullptr;
      ga.M = m; ga.N = n; ga.K = m;
      ga.symmetric = 0; ga.b_mn_major = 1; ga.alpha = 1.0f; ga.beta = 0.0f; ga.diag = 0.0f;
      ga.R = nullptr; ga.ldr = 0; ga.r_stride = 0;
      ga.D = xnext; ga.ldd = ldnext; ga.d_stride = dstr_next; ga.d_f32 = next_f32; ga.d_trans = next_trans;
      const int x_epi = (!last || G.out_tma) ? kEpiTma : kEpiRegs;
      const CUtensorMap* xd = last ? &G.mo_e : &G.mx_e[cur ^ 1];
      if ((st = launch_gemm(G.mb_p, from_g ? G.mg_mn : G.mx_mn[cur], nullptr, xd, x_epi, ga, s)) != ZOPT_OK) return st;
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
    return fail(ZOPT_ETIMEOUT, std::string(fn) + ": a kernel of an earlier call timed out on a wait");
  }
  return ok();
}

// Whether a rows x cols matrix lies within the ZOPT_NS_MAX_DIM / ZOPT_NS_MAX_ELEMS limits.
bool shape_ok(long long rows, long long cols) {
  return rows <= ZOPT_NS_MAX_DIM && cols <= ZOPT_NS_MAX_DIM && rows * cols <= ZOPT_NS_MAX_ELEMS;
}

// The checks shared by both entry points for one shape's arguments.
zopt_status check_job(const char* fn, const void* G, const void* X, zopt_dtype io, long long rows, long long cols,
                      long long ld_g, long long ld_x, long long bs_g, long long bs_x, long long batch) {
  const std::string f(fn);
  if (G == nullptr || X == nullptr) return fail(ZOPT_EINVAL, f + ": NULL pointer");
  if (rows < 1 || cols < 1 || batch < 1) return fail(ZOPT_EINVAL, f + ": empty matrix or batch");
  if (!shape_ok(rows, cols)) return fail(ZOPT_EINVAL, f + ": a dimension above 2^30 or a matrix above 2^36 elements");
  if (ld_g < cols || ld_x < cols) return fail(ZOPT_EINVAL, f + ": leading dimension < cols");
  if (ld_g > ZOPT_NS_MAX_LD || ld_x > ZOPT_NS_MAX_LD) return fail(ZOPT_EINVAL, f + ": a leading dimension above 2^32");
  if (batch > 1 && (bs_g < rows * ld_g || bs_x < rows * ld_x))
    return fail(ZOPT_EINVAL, f + ": batch strides overlap the matrices");
  if (batch > 1 && (bs_g > ZOPT_NS_MAX_SPAN / (batch - 1) || bs_x > ZOPT_NS_MAX_SPAN / (batch - 1)))
    return fail(ZOPT_EINVAL, f + ": the batch spans more than 2^56 elements");
  if (io != ZOPT_F32 && io != ZOPT_BF16) return fail(ZOPT_EUNSUPPORTED, f + ": input/output dtype must be fp32 or bf16");
  return ok();
}

}  // namespace ns
}  // namespace zopt

extern "C" size_t zopt_ns_workspace(int64_t rows, int64_t cols, int32_t group, zopt_dtype compute_dtype) {
  if (rows < 1 || cols < 1 || group < 1 || (compute_dtype != ZOPT_BF16 && compute_dtype != ZOPT_F32)) return 0;
  if (!zopt::ns::shape_ok(rows, cols)) return 0;
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
    Gr.out_io = io_dtype;
    Gr.norm_ready = false;
    Gr.x0_raw = false;
    Gr.rows = rows; Gr.cols = cols; Gr.ld_g = ld_g; Gr.ld_x = ld_x; Gr.bs_g = batch_stride_g; Gr.bs_x = batch_stride_x;
    Gr.gs = static_cast<int>(batch - g0i < group ? batch - g0i : group);
    Gr.f32c = f32c;
    if ((st = group_init(Gr, p, static_cast<uint8_t*>(d_ws))) != ZOPT_OK) return st;
    if ((st = group_prep(&Gr, 1, eps, s)) != ZOPT_OK) return st;
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
    if (b.rows < 1 || b.cols < 1 || b.batch < 1 || b.batch > 65535 || !zopt::ns::shape_ok(b.rows, b.cols)) return 0;
    total += static_cast<size_t>(zopt::ns::round_up(
        static_cast<long long>(zopt::ns::plan(b.rows, b.cols, 2, b.batch).total), 1024));
  }
  return total;
}

namespace zopt {
namespace ns {

int norm_blocks(long long n) {
  const long long bpm = (n + kSumsqElems - 1) / kSumsqElems;
  return static_cast<int>(bpm < 1 ? 1 : (bpm > kPrepBlocks ? kPrepBlocks : bpm));
}

void many_norm_partials(const zopt_ns_job* jobs, int32_t n_jobs, void* d_ws, double** base, long long* stride_doubles) {
  size_t at = 0;
  for (int32_t j = 0; j < n_jobs; ++j) {
    const zopt_ns_job& b = jobs[j];
    // a group's prep scratch opens its workspace slice: matrix b's NormWorkspace at b * kPrepWsBytes
    base[j] = reinterpret_cast<double*>(static_cast<uint8_t*>(d_ws) + at + offsetof(NormWorkspace, partials));
    stride_doubles[j] = static_cast<long long>(kPrepWsBytes / sizeof(double));
    at += static_cast<size_t>(round_up(static_cast<long long>(plan(b.rows, b.cols, 2, b.batch).total), 1024));
  }
}

bool x0_raw_ok(long long rows, long long cols, zopt_dtype io) {
  // bf16 compute in the input's orientation, X0's rows packed (its pitch is cols rounded to 8)
  return io == ZOPT_BF16 && rows <= cols && cols % 8 == 0;
}

void many_x0(const zopt_ns_job* jobs, int32_t n_jobs, void* d_ws, uint16_t** base, long long* stride, bool* ok) {
  size_t at = 0;
  for (int32_t j = 0; j < n_jobs; ++j) {
    const zopt_ns_job& b = jobs[j];
    const Plan p = plan(b.rows, b.cols, 2, b.batch);
    // matrix 0's region opens after the header, X0 first; matrix b's per_mat bytes on
    base[j] = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(d_ws) + at + p.header);
    stride[j] = static_cast<long long>(p.per_mat / 2);
    ok[j] = x0_raw_ok(b.rows, b.cols, static_cast<zopt_dtype>(b.io_dtype));
    at += static_cast<size_t>(round_up(static_cast<long long>(p.total), 1024));
  }
}

zopt_status orthogonalize_many(const char* fn, const zopt_ns_job* jobs, int32_t n_jobs, int32_t steps,
                               const float* abc, float eps, void* d_ws, size_t ws_bytes, cudaStream_t s,
                               const zopt_dtype* out_io, const bool* norm_ready, const StatsSink* sinks,
                               int* slots_out, const bool* x0_raw) {
  const std::string f(fn);
  if (jobs == nullptr || d_ws == nullptr || abc == nullptr) return fail(ZOPT_EINVAL, f + ": NULL pointer");
  if (n_jobs < 1) return fail(ZOPT_EINVAL, f + ": no jobs");
  if (steps < 1) return fail(ZOPT_EINVAL, f + ": steps < 1");
  if (!std::isfinite(abc[0]) || !std::isfinite(abc[1]) || !std::isfinite(abc[2]) || !std::isfinite(eps) || eps < 0)
    return fail(ZOPT_EINVAL, f + ": coefficients and eps must be finite (eps >= 0)");
  if (!aligned16(d_ws)) return fail(ZOPT_EINVAL, f + ": workspace is not 16-byte aligned");
  zopt_status st = ZOPT_OK;
  for (int32_t j = 0; j < n_jobs; ++j) {
    const zopt_ns_job& b = jobs[j];
    if ((st = check_job(fn, b.G, b.X, static_cast<zopt_dtype>(b.io_dtype), b.rows, b.cols, b.ld_g, b.ld_x,
                        b.batch_stride_g, b.batch_stride_x, b.batch)) != ZOPT_OK)
      return st;
    if (b.batch > 65535) return fail(ZOPT_EINVAL, f + ": a job's batch exceeds 65535");
    if (out_io != nullptr && out_io[j] != ZOPT_F32 && out_io[j] != ZOPT_BF16)
      return fail(ZOPT_EUNSUPPORTED, f + ": output dtype must be fp32 or bf16");
    if (x0_raw != nullptr && x0_raw[j] &&
        (norm_ready == nullptr || !norm_ready[j] || !x0_raw_ok(b.rows, b.cols, static_cast<zopt_dtype>(b.io_dtype))))
      return fail(ZOPT_EINVAL, f + ": internal: an unnormalised X0 for a job that cannot take one");
  }
  const size_t need = zopt_ns_workspace_many(jobs, n_jobs);
  if (need == 0 || ws_bytes < need) return fail(ZOPT_EINVAL, f + ": workspace smaller than zopt_ns_workspace_many");
  if (slots_out != nullptr)
    for (int32_t j = 0; j < n_jobs; ++j) slots_out[j] = 0;
  int* err_dev = nullptr;
  if ((st = take_error_word(fn, &err_dev)) != ZOPT_OK) return st;
  const int sms = sm_count();
  if (sms <= 0) return fail(ZOPT_ECUDA, f + ": no CUDA device");
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
    Gr.out_io = out_io != nullptr ? out_io[j] : Gr.io;
    Gr.norm_ready = norm_ready != nullptr && norm_ready[j];
    Gr.x0_raw = x0_raw != nullptr && x0_raw[j];
    Gr.rows = b.rows; Gr.cols = b.cols; Gr.ld_g = b.ld_g; Gr.ld_x = b.ld_x;
    Gr.bs_g = b.batch_stride_g; Gr.bs_x = b.batch_stride_x;
    Gr.gs = b.batch;
    Gr.f32c = false;
    const Plan p = plan(b.rows, b.cols, 2, b.batch);
    if ((st = group_init(Gr, p, static_cast<uint8_t*>(d_ws) + at)) != ZOPT_OK) return st;
    at += static_cast<size_t>(round_up(static_cast<long long>(p.total), 1024));
  }
  // When the call has CTA-pair jobs, jobs with kPairRideMin <= m < 1024 ride their launches: one
  // launch per product of a step then covers them too, their tiles filling the large jobs' last
  // waves, instead of a fused launch of their own that would run alone after (or before) them.
  bool any_pair = false;
  for (const Group& Gr : groups) any_pair = any_pair || (Gr.pair && !Gr.f32c);
  if (any_pair)
    for (Group& Gr : groups)
      if (!Gr.f32c && Gr.p.m >= kPairRideMin) Gr.pair = true;
  if ((st = group_prep(groups.data(), n_jobs, eps, s)) != ZOPT_OK) return st;
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
      FusedJob& fj = fa.job[fa.n_jobs];
      group_job(Gr, k, err_dev, fj, fm.job[fa.n_jobs]);
      if (sinks != nullptr) {  // the last step's B'X writes its output's statistics
        GemmArgs t3 = fj.prod[3];
        if (tiles_1cta(t3) && 8LL * t3.tiles_per_mat <= sinks[j].cap) {
          fj.prod[3].st_sum = sinks[j].sum;
          fj.prod[3].st_max = sinks[j].max;
          fj.prod[3].st_stride = sinks[j].stride;
          slots_out[j] = 8 * t3.tiles_per_mat;
        }
      }
      ++fa.n_jobs;
    }
  }
  // the CTA-pair jobs: each product of a step in one launch for all of them
  std::vector<const Group*> pairs;
  std::vector<const StatsSink*> pair_sinks;
  for (int32_t j = 0; j < n_jobs; ++j) {
    const Group& Gr = groups[static_cast<size_t>(j)];
    if (!group_fusable(Gr, k) && Gr.pair) {
      pairs.push_back(&Gr);
      const StatsSink* sk = nullptr;
      if (sinks != nullptr && Gr.out_tma) {  // the last B'X's epilogue is a TMA one
        const long long slots = 8 * ((Gr.p.m + BM2 - 1) / BM2) * ((Gr.p.n + BN - 1) / BN);
        if (slots <= sinks[j].cap) {
          sk = &sinks[j];
          slots_out[j] = static_cast<int>(slots);
        }
      }
      pair_sinks.push_back(sk);
    }
  }
  if (!pairs.empty() && (st = pair_products(pairs, k, steps, err_dev, s, &pair_sinks)) != ZOPT_OK) return st;
  for (int32_t j = 0; j < n_jobs; ++j) {
    const Group& Gr = groups[static_cast<size_t>(j)];
    if (!group_fusable(Gr, k) && !Gr.pair && (st = group_products(Gr, k, steps, err_dev, s)) != ZOPT_OK) return st;
  }
  return ok();
}

}  // namespace ns
}  // namespace zopt

extern "C" zopt_status zopt_ns_orthogonalize_many(const zopt_ns_job* jobs, int32_t n_jobs, int32_t steps,
                                                  const float* abc, float eps, void* d_ws, size_t ws_bytes,
                                                  zopt_stream stream) {
  return zopt::ns::orthogonalize_many("zopt_ns_orthogonalize_many", jobs, n_jobs, steps, abc, eps, d_ws, ws_bytes,
                                      reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr);
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

// A completion counter that nothing advances.
__device__ uint32_t g_never_counted;

// One thread waits, with the given limit, for that counter to reach 1: the bounded wait of the
// fused kernel's dependencies between products, run on purpose.
__global__ void count_selftest_kernel(int* err, unsigned long long limit_ns) {
  if (threadIdx.x == 0) wait_count(&g_never_counted, 1u, err, limit_ns);
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

extern "C" zopt_status zopt_selftest_count_timeout(int64_t limit_ns, zopt_stream stream) {
  using namespace zopt;
  if (limit_ns < 1 || limit_ns > 2000000000LL)
    return fail(ZOPT_EINVAL, "zopt_selftest_count_timeout: limit must lie in (0, 2 s]");
  int* h = nullptr;
  int* d = nullptr;
  zopt_status st = ns::error_word(&h, &d);
  if (st != ZOPT_OK) return st;
  ns::count_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
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
