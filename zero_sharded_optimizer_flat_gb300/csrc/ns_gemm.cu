// The Newton-Schulz products on tcgen05 tensor cores, one launch per product: the single-CTA
// persistent GEMM and its CTA-pair form (whose launch may cover the same product of up to four
// shapes), and their host launchers.
//
// Single CTA: one CTA per SM (persistent), 192 threads. Warp 0 streams 128x64 and 256x64 bf16
// tiles into a shared-memory ring with TMA (128-byte swizzle); one thread of warp 1 issues
// tcgen05.mma (M=128, N=256, K=16) into one of two TMEM accumulators (2 x 256 fp32 columns),
// committing stage-release and accumulator-ready events to mbarriers; warps 2-5 drain the other
// accumulator (tcgen05.ld), apply alpha*acc (+ beta*R, + the diagonal term) and store it while
// the next tile is being multiplied: through registers and plain stores (kEpiRegs) or as
// 32 x 32 bf16 boxes handed to the TMA (kEpiTma, kEpiTmaR).
#include <cstring>

#include "ns_tile.cuh"

namespace zopt {
namespace ns {

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
      if (lane == 0) ok = tc::mbar_wait_idle(tfull + b, tph, a.err) ? 1 : 0;
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
      if (lane == 0) ok = tc::mbar_wait_idle(tfull + b, tph, a.err) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc::fence_after_sync();
      int mb, ti, tj;
      tile_coords(a, t, mb, ti, tj);
      GemmArgs am = a;  // this matrix's R, D and alpha
      am.alpha = a.alpha * amat_of(a, mb);
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
// A launch covers the jobs of a PairBatch (one or more products of the same kind): the pairs
// walk the launch's tile index, and each tile takes its job's maps and arguments.
template <int kEpi>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_pair_kernel(const __grid_constant__ PairBatch B) {
  constexpr int S2 = stages2_of(kEpi);
  constexpr bool kTma = kEpi != kEpiRegs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S2 * kHalf;
  uint8_t* sEpi = sB + S2 * kHalf;  // the TMA epilogue's boxes
  uint64_t* full = reinterpret_cast<uint64_t*>(sEpi + epi_bytes2(kEpi));
  uint64_t* empty = full + S2;
  uint64_t* tfull = empty + S2;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 5);
  float* stage_base = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_rank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int total = B.start[B.n];
  int* err = B.job[0].a.err;
  if (threadIdx.x == 0) {
    for (int q = 0; q < S2; ++q) {
      tc::mbar_init(full + q, 1);
      tc::mbar_init(empty + q, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(tfull + b, 1);
      tc::mbar_init(tempty + b, 8);  // the epilogue warps of both CTAs, one arrival each (used in the leader)
    }
    tc::mbar_init(drain, 1);
    tc::fence_mbar_init();
    for (int j = 0; j < B.n; ++j) {
      tc::prefetch_tmap(&B.job[j].P);
      tc::prefetch_tmap(&B.job[j].Q);
      if (kTma) tc::prefetch_tmap(&B.job[j].D);
    }
  }
  if (warp == 1) {
    tc::tmem_alloc_pair(tslot, kTmemCols);
    tc::tmem_relinquish_pair();
  }
  tc::fence_before_sync();
  tc::cluster_sync();  // the peer's barriers exist before anyone arrives on them
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
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
      for (int t = pair; ok && t < total; t += npairs) {
        const int j = pair_job_of(B, t);
        const PairJob& J = B.job[j];
        int mb, tp, tj;
        tile_coords2(J.a, t - B.start[j], mb, tp, tj);
        const int nk = (J.a.K + BK - 1) / BK;
        const int row0 = tp * BM2 + static_cast<int>(rank) * 128;  // this CTA's A rows
        const int col0 = tj * BN + static_cast<int>(rank) * 128;    // this CTA's B columns
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(empty + s, ph ^ 1u, err)) {
            ok = false;
            break;
          }
          if (leader) tc::mbar_arrive_expect_tx(full + s, 4 * kHalf);  // both CTAs' A and B halves
          armed[s] = static_cast<int>(ph);
          const uint32_t bar = tc::map_to_rank(tc::smem_u32(full + s), 0);
          tc::tma_load_3d_pair(sA + s * kHalf, &J.P, bar, kb * BK, row0, mb);
          if (!J.a.b_mn_major) {
            tc::tma_load_3d_pair(sB + s * kHalf, &J.Q, bar, kb * BK, col0, mb);
          } else {
            tc::tma_load_3d_pair(sB + s * kHalf, &J.Q, bar, col0, kb * BK, mb);
            tc::tma_load_3d_pair(sB + s * kHalf + kBoxMN, &J.Q, bar, col0 + 64, kb * BK, mb);
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
      int s = 0, it = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = pair; ok && t < total; t += npairs, ++it) {
        const GemmArgs& a = B.job[pair_job_of(B, t)].a;
        const int nk = (a.K + BK - 1) / BK;
        const uint32_t idesc = tc::idesc_bf16_f32(BM2, BN, false, a.b_mn_major != 0);
        const int b = it & 1;
        const uint32_t tph = static_cast<uint32_t>(it >> 1) & 1u;
        if (!tc::mbar_wait(tempty + b, tph ^ 1u, err)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + static_cast<uint32_t>(b * BN);
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(full + s, ph, err)) {
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
    uint8_t* mine = sEpi + quad * (epi_bytes2(kEpi) / 4);
    const uint32_t tempty_leader[2] = {tc::map_to_rank(tc::smem_u32(tempty), 0),
                                       tc::map_to_rank(tc::smem_u32(tempty + 1), 0)};
    const int rows0 = static_cast<int>(rank) * 128 + 32 * quad;  // this warp's rows within a tile
    auto has_r = [](const GemmArgs& a) { return kEpi == kEpiTmaR && a.beta != 0.0f; };
    // kEpiTmaR: R's piece for the first block the warp writes in tile t, loaded from L2 into
    // registers before the tile's accumulator is ready (while its MMAs still run)
    uint4 r0[4];
    auto first_r = [&](int t) {
      if constexpr (kEpi == kEpiTmaR) {
        const int j = pair_job_of(B, t);
        const GemmArgs& a = B.job[j].a;
        if (!has_r(a)) return;
        int mb, tp, tj;
        tile_coords2(a, t - B.start[j], mb, tp, tj);
        prefetch_r_first(a, mb, tp * BM2 + rows0, tj, lane, r0);
      }
    };
    int last_par = -1;
    int t = pair;
    if (t < total) first_r(t);
    for (int it = 0; t < total; t += npairs, ++it) {
      const int b = it & 1;
      const uint32_t tph = static_cast<uint32_t>(it >> 1) & 1u;
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait_idle(tfull + b, tph, err) ? 1 : 0;
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
      tc::fence_after_sync();
      const int j = pair_job_of(B, t);
      const GemmArgs& a = B.job[j].a;
      int mb, tp, tj;
      tile_coords2(a, t - B.start[j], mb, tp, tj);
      // statistics slot (when wanted): the tile's index within its matrix, then 8 per tile
      const int st_slot = a.st_sum != nullptr
                              ? ((t - B.start[j]) - mb * a.tiles_per_mat) * 8 + static_cast<int>(rank) * 4 + quad
                              : -1;
      epi_tile_tma<false, 2, kEpi == kEpiTmaR, true>(
          a, &B.job[j].D, mine, tmem + (static_cast<uint32_t>(32 * quad) << 16) + static_cast<uint32_t>(b * BN),
          tp * BM2 + rows0, tj, mb, has_r(a), lane, last_par, 0, BN / 32, r0, st_slot);
      tc::fence_before_sync();
      __syncwarp();  // every lane's TMEM reads are done: one arrival releases the warp's part
      if (lane == 0) tc::mbar_arrive_cluster(tempty_leader[b]);  // the leader's MMA thread may reuse this accumulator
      if (t + npairs < total) first_r(t + npairs);
    }
    if (lane == 0) tc::bulk_wait_all();  // every store has reached global memory
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2..5)
    const int quad = warp & 3;
    const int row = 32 * quad + lane;
    const uint32_t tempty_leader[2] = {tc::map_to_rank(tc::smem_u32(tempty), 0),
                                       tc::map_to_rank(tc::smem_u32(tempty + 1), 0)};
    int it = 0;
    for (int t = pair; t < total; t += npairs, ++it) {
      const int b = it & 1;
      const uint32_t tph = static_cast<uint32_t>(it >> 1) & 1u;
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait_idle(tfull + b, tph, err) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc::fence_after_sync();
      const int j = pair_job_of(B, t);
      const GemmArgs& a = B.job[j].a;
      int mb, tp, tj;
      tile_coords2(a, t - B.start[j], mb, tp, tj);
      GemmArgs am = a;
      am.alpha = a.alpha * amat_of(a, mb);
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
          __syncwarp();
          if (lane == 0) tc::mbar_arrive_cluster(tempty_leader[b]);
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

// ---------------------------------------------------------------------- launchers

// The CTA-pair kernel over the jobs of B with epilogue `epi`: P is read with 128-row boxes, Q
// with 128-row (K-major) or 64 x 64 (MN-major) boxes; kEpiTmaR reads R, the TMA epilogues store
// D through each job's maps.
zopt_status launch_gemm_pair_batch(PairBatch& B, int epi, cudaStream_t stream) {
  ZOPT_CUDA_TRY(once([] {
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_pair_kernel<kEpiRegs>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes2(kEpiRegs));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_bf16_pair_kernel<kEpiTmaR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes2(kEpiTmaR));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_bf16_pair_kernel<kEpiTma>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes2(kEpiTma));
    return e;
  }));
  if (B.n < 1 || B.n > kMaxPairJobs) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: internal: bad pair batch");
  long long total = 0;
  for (int j = 0; j < B.n; ++j) {
    GemmArgs& a = B.job[j].a;
    a.tiles_m = static_cast<int>((a.M + BM2 - 1) / BM2);
    a.tiles_n = static_cast<int>((a.N + BN - 1) / BN);
    long long per = 0;
    if (a.symmetric) {
      for (int r = 0; r < a.tiles_m; ++r) per += a.tiles_n - r;
    } else {
      per = static_cast<long long>(a.tiles_m) * a.tiles_n;
    }
    const long long tiles = per * a.group;
    if (tiles < 1 || total + tiles > 0x7FFFFFFFLL) return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: too many tiles");
    a.tiles_per_mat = static_cast<int>(per);
    a.num_tiles = static_cast<int>(tiles);
    B.start[j] = static_cast<int>(total);
    total += tiles;
    if (epi != kEpiRegs) {
      if ((epi == kEpiTmaR && (a.d_f32 || a.d_trans)) || (epi == kEpiTma && a.beta != 0.0f) ||
          (a.symmetric && (a.d_f32 || a.d_trans)))
        return fail(ZOPT_EINVAL, "zopt_ns_orthogonalize: internal: TMA epilogue without its maps");
    }
  }
  B.start[B.n] = static_cast<int>(total);
  const int sms = sm_count();
  if (sms < 2) return fail(ZOPT_ECUDA, "zopt_ns_orthogonalize: no CUDA device");
  const long long pairs = total < sms / 2 ? total : sms / 2;
  const dim3 grid(static_cast<unsigned>(2 * pairs));
  if (epi == kEpiRegs)
    return launch_pdl(gemm_bf16_pair_kernel<kEpiRegs>, grid, dim3(kGemmThreads), static_cast<size_t>(smem_bytes2(kEpiRegs)),
                      stream, B);
  if (epi == kEpiTmaR)
    return launch_pdl(gemm_bf16_pair_kernel<kEpiTmaR>, grid, dim3(kGemmThreads), static_cast<size_t>(smem_bytes2(kEpiTmaR)),
                      stream, B);
  return launch_pdl(gemm_bf16_pair_kernel<kEpiTma>, grid, dim3(kGemmThreads), static_cast<size_t>(smem_bytes2(kEpiTma)),
                    stream, B);
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
  ZOPT_CUDA_TRY(once([] {
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel<kEpiRegs>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes(kEpiRegs));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_bf16_kernel<kEpiTmaR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes(kEpiTmaR));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_bf16_kernel<kEpiTma>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes(kEpiTma));
    return e;
  }));
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


}  // namespace ns
}  // namespace zopt
