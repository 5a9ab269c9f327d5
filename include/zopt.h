/*
 * zopt.h — C ABI of libzopt, the rank-local optimizer step of a ZeRO-sharded trainer on one
 * GB300 (sm_103a).
 *
 * Five parts, each a few calls:
 *   1. the flat bucketed shard layout            (zopt_shard_layout and accessors, host only)
 *   2. the gradient norm / clip / found_inf stats (zopt_grad_norm_clip, zopt_clip_finalize,
 *      zopt_grad_accumulate / zopt_grad_accumulate2 for micro-step sums with the stats fused;
 *      device values)
 *   3. the fused AdamW update of the fp32 shard   (zopt_adamw_step, zopt_adamw_clip_step,
 *                                                 zopt_adamw_rescale_step)
 *   4. Muon's quintic Newton-Schulz               (zopt_ns_orthogonalize, _many)
 *   5. Muon's update around Newton-Schulz         (zopt_muon_step, _many)
 *
 * Conventions shared by every call:
 *   - Pointers named d_* and every tensor argument are DEVICE pointers owned by the caller,
 *     except where a call says otherwise (zopt_grad_accumulate also reads page-locked host
 *     memory). The library allocates no device memory; scratch space is a caller-provided
 *     workspace whose size a *_workspace() query returns.
 *   - Every device call is asynchronous on the given stream (a cudaStream_t; NULL is the
 *     legacy default stream) and never synchronises the host. Every per-step quantity (clip
 *     coefficient, found_inf, the AdamW step counter, the Newton-Schulz norms, the Muon
 *     guard) stays on the device, so a whole step can be captured in a CUDA graph and
 *     replayed; make each entry point's first call outside the capture (one-time setup:
 *     kernel attributes, occupancy queries, the mapped error word).
 *   - Arguments are validated before any launch. On failure a call returns a non-zero
 *     zopt_status, launches nothing, and zopt_last_error() describes the problem.
 *   - Device arrays must start on a 16-byte boundary (128-bit vector access).
 *   - All device values that a call writes are plain little-endian structs declared below.
 */
#ifndef ZOPT_H
#define ZOPT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ZOPT_API __attribute__((visibility("default")))
#else
#define ZOPT_API
#endif

typedef struct CUstream_st* zopt_stream; /* a cudaStream_t */

typedef enum zopt_status {
  ZOPT_OK = 0,
  ZOPT_EINVAL = 1,       /* an argument is out of range, misaligned or inconsistent */
  ZOPT_EUNSUPPORTED = 2, /* a dtype combination or shape class without a kernel */
  ZOPT_ECUDA = 3,        /* the CUDA runtime reported an error (message in zopt_last_error) */
  ZOPT_ETIMEOUT = 4      /* a bounded device-side wait gave up (see zopt_ns_orthogonalize) */
} zopt_status;

typedef enum zopt_dtype { ZOPT_F32 = 0, ZOPT_BF16 = 1 } zopt_dtype;

/* Message of the last failing call on this host thread (never NULL; "" if none). */
ZOPT_API const char* zopt_last_error(void);
/* Library version string. */
ZOPT_API const char* zopt_version(void);

/* ======================================================================================
 * 1. Flat bucketed shard layout  (host only, pure)
 *
 * deg/zero.py, ZeroMaster (class docstring and __init__): the trainable parameters are laid
 * end to end in a flat vector of N elements, cut into buckets of `bucket` elements after
 * rounding the bucket down to a multiple of `world` (never below `world`); every bucket
 * [s, e) is padded to L = ceil((e-s)/world)*world elements; rank r owns the r-th of world
 * equal pieces (L/world elements) of every bucket, and its shard is those pieces
 * concatenated in bucket order. Padding slots hold zeros.
 * ====================================================================================== */
typedef struct zopt_layout zopt_layout; /* opaque, host memory, owned by the library */

/* Build rank `rank`'s layout. numel[n_params] are the parameter sizes in flat order;
 * decay[n_params] (may be NULL = every parameter decays) is 1 where AdamW's decoupled
 * weight decay applies (bluscript_zero_ckpt.cpp, ZeroConfig: 1-D parameters excluded).
 * Errors: EINVAL for n_params < 1 (ZeroMaster "needs trainable parameters"), a negative
 * size, a total of 0 or >= 2^62 elements, bucket < 1, world < 1, rank outside [0, world).
 * On success *out must later be released with zopt_layout_free. */
ZOPT_API zopt_status zopt_shard_layout(const int64_t* numel, const uint8_t* decay, int32_t n_params,
                              int64_t bucket, int32_t world, int32_t rank, zopt_layout** out);
ZOPT_API void zopt_layout_free(zopt_layout* layout);

ZOPT_API int64_t zopt_layout_numel(const zopt_layout* layout);       /* N, the unpadded flat length */
ZOPT_API int64_t zopt_layout_shard_len(const zopt_layout* layout);   /* S = sum over buckets of L/world */
/* Device bytes of this rank's optimizer state under the layout: the fp32 master, the two fp32
 * AdamW moments and the shard gradient, per shard slot 12 B + 4 (fp32 gradient) or + 2 (bf16).
 * With an fp32 gradient this is the per-rank 16/W share of deg/zero.py's memory plan
 * (sharded_static_bytes: fp32 master + moments + gradient per shard), counted exactly, with the
 * padding of every bucket's pieces. -1 for a NULL layout or another dtype. */
ZOPT_API int64_t zopt_layout_state_bytes(const zopt_layout* layout, zopt_dtype grad_dtype);
ZOPT_API int32_t zopt_layout_world(const zopt_layout* layout);
ZOPT_API int32_t zopt_layout_rank(const zopt_layout* layout);
ZOPT_API int32_t zopt_layout_num_buckets(const zopt_layout* layout);
/* Bucket b: flat [start, end), padded length, and the shard offset of this rank's piece. */
ZOPT_API zopt_status zopt_layout_bucket(const zopt_layout* layout, int32_t b, int64_t* start, int64_t* end,
                               int64_t* padded, int64_t* shard_offset);
/* Segments (ZeroMaster._segments over each of this rank's pieces): maximal runs
 * (param index, offset inside the param, shard offset, length) in shard order.
 * The four output arrays (any may be NULL) must hold zopt_layout_num_segments() entries. */
ZOPT_API int64_t zopt_layout_num_segments(const zopt_layout* layout);
ZOPT_API zopt_status zopt_layout_segments(const zopt_layout* layout, int32_t* param, int64_t* param_offset,
                                 int64_t* shard_offset, int64_t* length);
/* The shard's no-decay runs: sorted, disjoint, non-adjacent half-open ranges
 * [begin_k, end_k) of shard slots that take NO weight decay (excluded parameters and
 * padding). Written to runs[2k] = begin_k, runs[2k+1] = end_k; `runs` is host memory of
 * 2*zopt_layout_num_nodecay_runs() int64 values. The caller copies this table to the device
 * once and passes it to zopt_adamw_step. */
ZOPT_API int64_t zopt_layout_num_nodecay_runs(const zopt_layout* layout);
ZOPT_API zopt_status zopt_layout_nodecay_runs(const zopt_layout* layout, int64_t* runs);

/* ======================================================================================
 * 2. Gradient norm, clip coefficient, found_inf  (device values, no host sync)
 *
 * deg/zero.py, grad_sq_norm: the squared L2 norm of the shard's fp32 gradient (a simulated
 * rank has no all-reduce, so it is the local shard's). bluscript_zero_ckpt.cpp, global clip
 * block: coef = min(1, max_norm / (norm + 1e-6)), with a non-finite norm kept away from min.
 * dmuon PR #16, sync-free clip stats: total_norm / clip_coef / clipped / found_inf are 0-dim
 * device values; finiteness is judged on the norm; an inf norm gives coef 0,
 * found_inf = 1, clipped = 0.
 * ====================================================================================== */
typedef struct zopt_clip_stats {
  double sumsq;      /* sum of g^2 over the shard, accumulated in fp64 */
  float norm;        /* fp32(sqrt(sumsq)) */
  float clip_coef;   /* min(1, max_norm / (norm + 1e-6f)) in fp32; 0 when found_inf */
  uint8_t clipped;   /* clip_coef < 1 and !found_inf */
  uint8_t found_inf; /* norm is inf or NaN */
  uint8_t reserved[6];
} zopt_clip_stats; /* 24 bytes, device resident */

/* Workspace bytes zopt_grad_norm_clip needs for n elements (a block-partials array and an
 * arrival counter). */
ZOPT_API size_t zopt_grad_norm_workspace(int64_t n);
/* Reduce grad[n] (fp32 or bf16, bf16 promoted exactly) into *d_stats on `stream`.
 * d_ws: at least zopt_grad_norm_workspace(n) bytes; it MUST be zero-filled before its first
 * use, and every call leaves it zero-filled again. Calls sharing a workspace or a stats
 * struct must be ordered (same stream). The result is deterministic for a given n and GPU.
 * Errors: EINVAL for n < 1, NULL pointers, misalignment, a short workspace, max_norm
 * negative or NaN. */
ZOPT_API zopt_status zopt_grad_norm_clip(const void* grad, zopt_dtype dtype, int64_t n, float max_norm, void* d_ws,
                                size_t ws_bytes, zopt_clip_stats* d_stats, zopt_stream stream);
/* Recompute norm / clip_coef / clipped / found_inf from d_stats->sumsq (one thread). This is
 * where a multi-rank job would all-reduce sumsq between zopt_grad_norm_clip and the step. */
ZOPT_API zopt_status zopt_clip_finalize(zopt_clip_stats* d_stats, float max_norm, zopt_stream stream);

/* zopt_grad_norm_clip without a workspace, for callers that cannot allocate device memory:
 * a plain-C host or plugin that only receives device pointers from its framework, a training
 * loop that forbids allocation after start-up, or a process whose device memory another
 * runtime has already reserved. The source pages have no counterpart to this call; it exists
 * for those callers only. Same arguments and results as zopt_grad_norm_clip, minus d_ws.
 * The scratch (an arrival counter and up to 1024 fp64 block partials, 8,448 bytes) is a
 * file-scope __device__ array that every GPU loading the library holds until the process
 * exits. The first call on each device looks up that array's device address (once, with the
 * device current); make that first call before any stream capture. Each call clears the
 * counter itself. All calls share the one array, so calls that overlap on the GPU (other
 * streams, unordered host threads) race and give wrong results; order them on one stream.
 * A launch takes zopt_grad_norm_clip's grid (one wave of resident blocks) capped at 1024
 * blocks; below the cap (always on a 152-SM GB300) the stats are bit for bit those of
 * zopt_grad_norm_clip. The looked-up address is cached per device index: after a
 * cudaDeviceReset of a device it used, a process must not call this entry point again.
 * Errors: those of zopt_grad_norm_clip. */
ZOPT_API zopt_status zopt_grad_norm_clip_noalloc(const void* grad, zopt_dtype dtype, int64_t n, float max_norm,
                                                 zopt_clip_stats* d_stats, zopt_stream stream);

/* Micro-step gradient accumulation into the fp32 shard gradient (deg/zero.py, ZeroMaster
 * collect / reduce_scatter: the parts of a step are summed in fp32 into the shard gradient,
 * which grad_sq_norm then reads). acc[n] (fp32) = micro_grad on the micro-step flagged
 * ZOPT_ACC_FIRST (acc is not read), else acc = acc + micro_grad (fp32, each addition rounded,
 * in call order). On the micro-step flagged ZOPT_ACC_LAST the same pass also reduces the
 * finished sum exactly as zopt_grad_norm_clip does and writes *d_stats (d_ws and d_stats are
 * only used then; d_ws follows zopt_grad_norm_clip's rules). Both flags together: one part.
 * micro_grad may be device memory or page-locked host memory (cudaHostAlloc / cudaHostRegister,
 * e.g. a pinned torch tensor): the pass then reads it through the memory's device mapping over
 * the CPU-GPU link, so the host-to-device transfer and the addition are one pass with no staging
 * buffer in HBM. The caller keeps that host memory unchanged until the call has run on the stream.
 * Errors: EINVAL for n < 1, NULL/misaligned pointers, pageable host memory or memory of another
 * device as micro_grad, unknown flags, a missing workspace or stats on the last micro-step;
 * EUNSUPPORTED for a dtype other than fp32/bf16. */
#define ZOPT_ACC_FIRST 1
#define ZOPT_ACC_LAST 2
ZOPT_API zopt_status zopt_grad_accumulate(float* acc, const void* micro_grad, zopt_dtype dtype, int64_t n,
                                          int32_t flags, float max_norm, void* d_ws, size_t ws_bytes,
                                          zopt_clip_stats* d_stats, zopt_stream stream);
/* Two micro-steps in one pass: the result (acc, and the stats on ZOPT_ACC_LAST) is bit for bit
 * that of zopt_grad_accumulate(micro_grad_a) followed by zopt_grad_accumulate(micro_grad_b) with
 * the same flags split between them (ZOPT_ACC_FIRST applies to a, ZOPT_ACC_LAST to b): acc =
 * fp32(a) + fp32(b) on the first micro-steps, else (acc + a) + b, each addition rounded. It saves
 * one read and one write of the fp32 sum: 8 B per element instead of 16 for the first two
 * micro-steps, 12 instead of 20 for two later ones (bf16 parts). Both parts share the dtype and
 * the rules for micro_grad, and either may be page-locked host memory. Errors: those of
 * zopt_grad_accumulate, and EINVAL for a NULL micro_grad_b. */
ZOPT_API zopt_status zopt_grad_accumulate2(float* acc, const void* micro_grad_a, const void* micro_grad_b,
                                           zopt_dtype dtype, int64_t n, int32_t flags, float max_norm, void* d_ws,
                                           size_t ws_bytes, zopt_clip_stats* d_stats, zopt_stream stream);

/* ======================================================================================
 * 3. Fused AdamW over the flat fp32 shard
 *
 * dmuon PR #16, foreach AdamW: decoupled weight decay -> moments -> bias-corrected addcdiv;
 * bias corrections are per-step scalars. DeepSpeed PR #9021: the gradient is multiplied by
 * the scale (here the clip coefficient) as it is loaded, after the bf16 -> fp32 promotion;
 * a bf16 gradient of fp32 masters is read as bf16. bluscript_zero_ckpt.cpp: fp32 master and
 * fp32 moments (a bf16 master would round the (1 - lr*wd) decay away). deg/zero.py,
 * gather_params: the updated shard rounded to bf16 compute weights.
 *
 * Per element, each operation rounded to fp32 in this order (no fused multiply-add):
 *   g = g_in * coef;  if decay: p = p * fp32(1 - lr*wd);
 *   m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*(g*g);
 *   d = sqrt(v) / fp32(sqrt(1 - beta2^t)) + eps;  p = p - fp32(lr / (1 - beta1^t)) * (m / d);
 *   out = bf16_rne(p)
 * with t = d_state->step + 1, beta^t an fp64 power by right-to-left square-and-multiply,
 * and every scalar formed in fp64 from the fp64 hyper-parameters then rounded once to fp32.
 * ====================================================================================== */
typedef struct zopt_adamw_hparams {
  double lr;
  double beta1;
  double beta2;
  double eps;
  double weight_decay;
  int32_t skip_on_inf; /* 1: a step whose clip stats report found_inf changes nothing */
  int32_t reserved;
} zopt_adamw_hparams;

typedef struct zopt_adam_state {
  int64_t step;     /* AdamW steps taken; advanced on the device by every step not skipped */
  uint32_t arrive;  /* internal arrival counter; 0 between calls */
  int32_t reserved;
} zopt_adam_state; /* 16 bytes, device resident; all-zero = a fresh optimizer */

/* One AdamW step of this rank's shard, in place, on `stream`.
 *   master, exp_avg, exp_avg_sq: fp32 [S] device arrays (S = zopt_layout_shard_len);
 *   grad: [S] of grad_dtype (ZOPT_F32 or ZOPT_BF16), the shard of the summed gradient;
 *   out_bf16: [S] bf16 bit patterns of the updated master, or NULL to skip the round-out;
 *   d_nodecay_runs: the device copy of zopt_layout_nodecay_runs (may be NULL only when the
 *     layout has no such runs);
 *   d_clip: clip stats from zopt_grad_norm_clip (NULL = coef 1, never skip);
 *   d_state: the step counter (required).
 * Padding slots (zero master, zero gradient) stay exactly zero.
 * Errors: EINVAL for NULL/misaligned pointers, non-finite or out-of-range hyper-parameters
 * (lr < 0, beta outside [0, 1), eps < 0); EUNSUPPORTED for another gradient dtype. */
ZOPT_API zopt_status zopt_adamw_step(const zopt_layout* layout, const int64_t* d_nodecay_runs, float* master,
                            float* exp_avg, float* exp_avg_sq, const void* grad, zopt_dtype grad_dtype,
                            uint16_t* out_bf16, const zopt_adamw_hparams* hparams,
                            const zopt_clip_stats* d_clip, zopt_adam_state* d_state, zopt_stream stream);

/* Workspace bytes zopt_adamw_clip_step needs for a shard of shard_len elements (a 256-byte
 * header of counters and one fp64 partial sum per block; 0 for shard_len < 1). */
ZOPT_API size_t zopt_adamw_clip_workspace(int64_t shard_len);
/* zopt_grad_norm_clip over grad[S] followed by zopt_adamw_step with those stats, in one launch
 * (for a gradient that arrives whole, with no accumulation pass to carry the sum of squares).
 * The norm is this shard's own: right for one rank, or a simulated rank; a multi-rank job,
 * whose clip needs the all-reduced sum of squares, keeps zopt_grad_norm_clip, the all-reduce
 * and zopt_clip_finalize before zopt_adamw_step. bluscript_zero_ckpt.cpp, global clip block,
 * and dmuon PR #16, sync-free clip stats: the same arithmetic as the two calls. One
 * cooperative wave of blocks: each block sums the squares of the run of the shard it then
 * updates, all blocks meet at a grid-wide barrier (bounded: a block whose wait gives up
 * updates nothing, so the step is left incomplete, and the next call of a kernel with bounded
 * waits returns ETIMEOUT), and every block adds the blocks' sums in the same fixed order, so
 * the stats are deterministic for a given S and GPU. The sum of squares is the same sum as
 * zopt_grad_norm_clip's but added in another order, so it can differ from it in its last bits.
 * d_clip receives the stats (required); d_ws: at least zopt_adamw_clip_workspace(S) bytes,
 * 16-byte aligned, zero-filled before its first use; every call leaves its counters (the first
 * 256 bytes) at zero again (after an ETIMEOUT it must be zero-filled again). Calls sharing a
 * workspace must be ordered (same stream). Other arguments and errors as zopt_adamw_step, plus
 * EINVAL for a NULL d_clip or d_ws, a short workspace, max_norm negative or NaN; ECUDA if the
 * device cannot hold the wave (cooperative launch). */
ZOPT_API zopt_status zopt_adamw_clip_step(const zopt_layout* layout, const int64_t* d_nodecay_runs, float* master,
                                         float* exp_avg, float* exp_avg_sq, const void* grad,
                                         zopt_dtype grad_dtype, uint16_t* out_bf16,
                                         const zopt_adamw_hparams* hparams, float max_norm, void* d_ws,
                                         size_t ws_bytes, zopt_clip_stats* d_clip, zopt_adam_state* d_state,
                                         zopt_stream stream);

/* Re-target the last step (t = d_state->step, not advanced) from g*old_scale to g*new_scale,
 * in one pass (DeepSpeed PR #9021, adam_rescale_step commit: a step taken speculatively on
 * an unclipped gradient becomes the step on the final clip coefficient without an undo and a
 * redo). Per element, each operation an fp32 rounding: d(m, v) = m / (sqrt(v)/fp32(sqrt(1 -
 * beta2^t)) + eps); u_old = d(m, v); m += fp32((1-b1)(new-old))*g;
 * v = max(0, v + fp32((1-b2)(new^2-old^2))*(g*g)) (a NaN stays NaN); p += fp32(lr/(1 -
 * beta1^t))*(u_old - d(m, v)); out = bf16_rne(p). The decoupled decay cancels. With d_clip
 * non-NULL new_scale is d_clip->clip_coef, and a found_inf there leaves everything unchanged;
 * with no step taken yet (step 0) the call changes nothing. Same buffers and errors as
 * zopt_adamw_step (the no-decay table is not needed). */
ZOPT_API zopt_status zopt_adamw_rescale_step(const zopt_layout* layout, float* master, float* exp_avg,
                                             float* exp_avg_sq, const void* grad, zopt_dtype grad_dtype,
                                             uint16_t* out_bf16, const zopt_adamw_hparams* hparams, float old_scale,
                                             float new_scale, const zopt_clip_stats* d_clip,
                                             const zopt_adam_state* d_state, zopt_stream stream);

/* ======================================================================================
 * 4. Muon's quintic Newton-Schulz on whole matrices
 *
 * bluscript_zero_ckpt.cpp, ShardedMuon design note: U = NewtonSchulz(M), the iterated matrix
 * polynomial X <- aX + (bXX' + c(XX')^2)X over the WHOLE matrix (a flat slice would cut it
 * mid-row, so each matrix has one owner rank); the trainer runs 5 steps.
 *
 * X0 = G / (||G||_F + eps); a matrix with more rows than columns is processed as its
 * transpose (m = min(rows, cols) <= n) and transposed back on output. Per step:
 * A = X X' (m x m), B = b A + c A A', X = a X + B X. With compute_dtype ZOPT_BF16 the
 * operands and the products A, B, X are bf16 (round-to-nearest-even) with fp32 accumulation
 * on the tensor cores, and the last two are formed as B' = B + a I and X = B' X (the same
 * map; B' is rounded to bf16 once). A bf16 G in X's orientation (rows <= cols) with 16-byte
 * aligned rows and matrices is read in place by the first step, whose X X' and B'X apply
 * 1/(||G||+eps) (squared for X X') to their fp32 accumulators: X0 is then not rounded to bf16
 * on its own. ZOPT_F32 computes the products as written. (a, b, c) = abc[0..2] (the pages print
 * no triple; the usual quintic Muon choice is 3.4445, -4.7750, 2.0315).
 * ====================================================================================== */

/* Size limits of one Newton-Schulz (or Muon) matrix, under which every tile coordinate and
 * count the kernels form fits in 32 bits and every element offset in 64. */
#define ZOPT_NS_MAX_DIM (1LL << 30)    /* rows and cols */
#define ZOPT_NS_MAX_ELEMS (1LL << 36)  /* rows * cols */
#define ZOPT_NS_MAX_LD (1LL << 32)     /* leading dimensions (elements) */
#define ZOPT_NS_MAX_SPAN (1LL << 56)   /* (batch - 1) * batch stride (elements) */

/* Workspace bytes to process `group` rows x cols matrices together (0 for an unsupported
 * compute dtype, group < 1, or a shape beyond the limits above). A call processes its batch in
 * groups of as many matrices as its workspace holds: every product of a step is one launch
 * over the whole group, so a larger group means fewer launches and better use of the SMs. */
ZOPT_API size_t zopt_ns_workspace(int64_t rows, int64_t cols, int32_t group, zopt_dtype compute_dtype);
/* Orthogonalise `batch` matrices G[b] (rows x cols, row-major, leading dimension ld_g,
 * matrix b at G + b*batch_stride_g elements) into X[b] (same shape, ld_x, batch_stride_x).
 *   io_dtype: dtype of G and X (ZOPT_BF16 or ZOPT_F32);
 *   compute_dtype: ZOPT_BF16 (tcgen05 tensor cores) or ZOPT_F32 (fp32 FMA, for callers that
 *     need agreement with fp64 to about 1e-4);
 *   steps >= 1; abc: 3 host floats; eps >= 0 (1e-7 is the usual choice);
 *   d_ws: at least zopt_ns_workspace(rows, cols, 1, compute_dtype) bytes, 16-byte aligned.
 * G and X must not overlap. Errors: EINVAL for NULL pointers, empty shapes, shapes, leading
 * dimensions or batch spans beyond the ZOPT_NS_MAX_* limits, leading dimensions < cols,
 * overlapping batch strides, steps < 1, non-finite
 * coefficients, a short workspace; EUNSUPPORTED for other dtypes; ETIMEOUT when a kernel of
 * an earlier call gave up on a bounded wait (its results are not valid). */
ZOPT_API zopt_status zopt_ns_orthogonalize(const void* G, void* X, zopt_dtype io_dtype, int64_t rows, int64_t cols,
                                           int64_t ld_g, int64_t ld_x, int64_t batch_stride_g,
                                           int64_t batch_stride_x, int32_t batch, zopt_dtype compute_dtype,
                                           int32_t steps, const float* abc, float eps, void* d_ws, size_t ws_bytes,
                                           zopt_stream stream);

/* One shape's matrices for zopt_ns_orthogonalize_many: `batch` matrices G[b] -> X[b], rows x
 * cols, with the meaning zopt_ns_orthogonalize gives its arguments (io_dtype a zopt_dtype;
 * batch at most 65535). 72 bytes. */
typedef struct zopt_ns_job {
  const void* G;
  void* X;
  int64_t rows, cols;
  int64_t ld_g, ld_x;
  int64_t batch_stride_g, batch_stride_x;
  int32_t batch;
  int32_t io_dtype;
} zopt_ns_job;

/* Workspace bytes for zopt_ns_orthogonalize_many over these jobs (0 if a job is empty or has
 * more than 65535 matrices): each job's zopt_ns_workspace(rows, cols, batch, ZOPT_BF16),
 * rounded up to 1 KiB, summed. */
ZOPT_API size_t zopt_ns_workspace_many(const zopt_ns_job* jobs, int32_t n_jobs);
/* Orthogonalise every matrix of every job: `steps` quintic steps with coefficients abc and
 * eps as for zopt_ns_orthogonalize, bf16 compute. Jobs whose shorter side m is 1024 and above
 * run each product of a step in one launch of the CTA-pair kernel for up to four jobs (their
 * tiles filling each other's waves); when the call has such jobs, jobs with 512 <= m < 1024
 * join those launches too (their tiles fill the large jobs' last waves instead of running in a
 * launch of their own). The other jobs whose output rows are 16-byte aligned run in one
 * persistent launch per six jobs, the products of each step interleaved across jobs (one job's
 * waits for its previous product are filled by the other jobs' tiles); any other job runs
 * product by product. The inputs of all jobs are normalised in three launches before any
 * product. A tile is computed the same way in any launch of its kind, so each result is
 * bitwise the one zopt_ns_orthogonalize gives with a workspace that holds the job's whole
 * batch, except for a job with 512 <= m < 1024 in a call with CTA-pair jobs: that result is
 * bitwise the same in every such call (and within the bf16 tolerance of the single call's).
 * jobs is read during the call only; d_ws (16-byte aligned) is owned by the call until the
 * stream passes it. Same errors as zopt_ns_orthogonalize. */
ZOPT_API zopt_status zopt_ns_orthogonalize_many(const zopt_ns_job* jobs, int32_t n_jobs, int32_t steps,
                                                const float* abc, float eps, void* d_ws, size_t ws_bytes,
                                                zopt_stream stream);

/* Device-side failure reporting. Every wait of the tensor-core kernels and of
 * zopt_adamw_clip_step's grid barrier is bounded (4 s); one that runs out records an error
 * word in mapped host memory, drains the kernel's copies and MMAs, frees its TMEM and returns,
 * so the context stays usable; the next zopt_ns_orthogonalize / zopt_muon_step /
 * zopt_adamw_clip_step then returns ZOPT_ETIMEOUT.
 * zopt_take_device_error returns the error word (0 = none, -1 if it cannot be set up) and
 * clears it, without synchronising (read it after the work it covers has completed).
 * zopt_selftest_wait_timeout launches one thread that waits, limited to limit_ns (at most
 * 2 s), on an mbarrier phase that nothing completes: the same bounded-wait code, run out on
 * purpose, so a test can check the reporting path. zopt_selftest_count_timeout does the same
 * with the wait of the fused Newton-Schulz kernel on a per-matrix completion counter (in
 * global memory) that nothing advances. */
ZOPT_API int32_t zopt_take_device_error(void);
ZOPT_API zopt_status zopt_selftest_wait_timeout(int64_t limit_ns, zopt_stream stream);
ZOPT_API zopt_status zopt_selftest_count_timeout(int64_t limit_ns, zopt_stream stream);
/* The rescale kernel divides sqrt(v) by the launch's constant c = sqrt(1 - beta2^t) through a
 * reciprocal and one FMA correction (Markstein, IBM J. Res. Develop. 34(1), 1990) instead of an
 * IEEE division. zopt_selftest_div_by_const compares the two for every bit pattern of v >= 0
 * at the given c in (0, 1] and adds the number of differing results to *d_mismatches (device
 * uint64, 8-byte aligned; NaN matches NaN). EINVAL for a bad counter or c. */
ZOPT_API zopt_status zopt_selftest_div_by_const(float c, unsigned long long* d_mismatches, zopt_stream stream);

/* ======================================================================================
 * 5. Muon's update around Newton-Schulz (matrices owned whole by this rank)
 *
 * bluscript_zero_ckpt.cpp, ShardedMuon: the owner rank keeps each matrix's fp32 master and
 * momentum; momentum 0.95 with Nesterov; decoupled weight decay; U = NewtonSchulz(u);
 * adjust_lr "match_rms_adamw" lifts the update RMS to 0.2 (scale 0.2*sqrt(max(rows, cols))),
 * "original" uses sqrt(max(1, rows/cols)); nsratio = ||U||_F / sqrt(min(rows, cols)) and a
 * divergence guard on the largest |U| element.
 *
 * Per matrix, each operation rounded to fp32 as written:
 *   buf = mu*buf + g;  u = g + mu*buf (nesterov) or buf;  U = NewtonSchulz(bf16(u)) (bf16
 *   compute, normalised by the norm of bf16(u), which the momentum pass sums itself; for a
 *   matrix no taller than wide with a width that is a multiple of 8 the pass writes bf16(u)
 *   into Newton-Schulz's own input buffer and the first step's products apply the
 *   normalisation; U the method's bf16 result);
 *   unless max|U| > guard (or not finite): p = p*fp32(1 - lr*wd) - fp32(lr*scale)*U;
 *   out = bf16_rne(p).  A rejected matrix keeps its master; its momentum is still updated.
 * ====================================================================================== */
#define ZOPT_MUON_MATCH_RMS_ADAMW 0
#define ZOPT_MUON_ORIGINAL 1

typedef struct zopt_muon_hparams {
  double lr;
  double momentum;
  double weight_decay;
  int32_t nesterov;  /* 1: u = g + mu*buf */
  int32_t adjust;    /* ZOPT_MUON_MATCH_RMS_ADAMW or ZOPT_MUON_ORIGINAL */
  int32_t ns_steps;  /* Newton-Schulz steps (5) */
  float abc[3];      /* quintic coefficients */
  float eps;         /* Newton-Schulz normalisation eps (1e-7) */
  float guard;       /* reject an update with an element of magnitude above this (1000) */
} zopt_muon_hparams;

typedef struct zopt_muon_stats {
  float update_fro; /* ||U||_F */
  float ns_ratio;   /* ||U||_F / sqrt(min(rows, cols)), healthy ~1 */
  float max_abs;    /* largest |U| element */
  uint32_t rejected;
} zopt_muon_stats; /* 16 bytes per matrix, device resident */

/* Workspace bytes to step `group` rows x cols matrices together (the Newton-Schulz workspace
 * plus, per group member, u and U in bf16 and U's statistics slots: 12 bytes for each
 * 128 x 256 tile's eight 32-row parts, at least 512 of them; 0 for a shape beyond the
 * ZOPT_NS_MAX_* limits). A call steps its batch in groups of as many matrices as the workspace
 * holds. */
ZOPT_API size_t zopt_muon_workspace(int64_t rows, int64_t cols, int32_t group);
/* One Muon step of `batch` rows x cols matrices stored back to back (matrix b at offset
 * b*rows*cols of master, momentum, grad and out_bf16). master, momentum: fp32; grad: fp32 or
 * bf16; out_bf16: may be NULL; d_stats: `batch` structs. U's sum of squares and largest
 * magnitude come from the epilogue of Newton-Schulz's last product where that writes U through
 * the TMA, else from a pass over U; either way they are summed in a fixed order, so a call
 * repeated on the same inputs gives the same stats. Errors: EINVAL for NULL or
 * misaligned pointers (16 bytes; a batch needs rows*cols to be a multiple of 4), an empty
 * shape or one beyond the ZOPT_NS_MAX_* limits, a batch of more than 2^46 elements,
 * out-of-range hyper-parameters (lr < 0, momentum outside [0, 1), steps < 1, guard <=
 * 0), a short workspace; EUNSUPPORTED for another gradient dtype; and the errors of
 * zopt_ns_orthogonalize. */
ZOPT_API zopt_status zopt_muon_step(float* master, float* momentum, const void* grad, zopt_dtype grad_dtype,
                                    uint16_t* out_bf16, int64_t rows, int64_t cols, int32_t batch,
                                    const zopt_muon_hparams* hparams, zopt_muon_stats* d_stats, void* d_ws,
                                    size_t ws_bytes, zopt_stream stream);

/* One shape's matrices for zopt_muon_step_many: the arguments of zopt_muon_step (grad_dtype a
 * zopt_dtype; batch at most 65535). 64 bytes. */
typedef struct zopt_muon_job {
  float* master;
  float* momentum;
  const void* grad;
  uint16_t* out_bf16;
  zopt_muon_stats* d_stats;
  int64_t rows, cols;
  int32_t batch;
  int32_t grad_dtype;
} zopt_muon_job;

/* Workspace bytes for zopt_muon_step_many over these jobs (0 if a job is empty or has more than
 * 65535 matrices). */
ZOPT_API size_t zopt_muon_workspace_many(const zopt_muon_job* jobs, int32_t n_jobs);
/* One Muon step for every matrix of every job with the same hyper-parameters: the Newton-Schulz
 * part of all jobs is one zopt_ns_orthogonalize_many call, so each job's results (master,
 * momentum, bf16 weights, stats) are bitwise what zopt_muon_step gives with a workspace that
 * holds the job's whole batch, with that call's one exception (a job with 512 <= min(rows, cols)
 * < 1024 beside a job with both sides 1024 and above: the momentum is still bitwise, the
 * update rides the CTA-pair launches). jobs is read during the call only. Same errors as
 * zopt_muon_step. */
ZOPT_API zopt_status zopt_muon_step_many(const zopt_muon_job* jobs, int32_t n_jobs, const zopt_muon_hparams* hparams,
                                         void* d_ws, size_t ws_bytes, zopt_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* ZOPT_H */
