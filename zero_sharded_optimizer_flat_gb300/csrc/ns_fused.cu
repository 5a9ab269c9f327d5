// The fused Newton-Schulz call: every product of every step of up to six jobs in one persistent
// launch (the work list and its counters are described with their definitions in ns_tile.cuh).
#include "ns_tile.cuh"

namespace zopt {
namespace ns {

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
      if (f.job[j].x0_is_g) {
        tc::prefetch_tmap(&m.gp);
        tc::prefetch_tmap(&m.gq);
        tc::prefetch_tmap(&m.gmn);
      }
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
        const bool from_g = it.s == 0 && f.job[it.j].x0_is_g;  // the first step reads the caller's G
        const CUtensorMap* P = it.p == 0 ? (from_g ? &m.gp : &m.xp[cur]) : (it.p == 1 ? &m.ap : &m.bp);
        const CUtensorMap* Q =
            it.p == 0 ? (from_g ? &m.gq : &m.xq[cur]) : (it.p == 1 ? &m.aq : (from_g ? &m.gmn : &m.xmn[cur]));
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
      if (lane == 0) ok = tc::mbar_wait_idle(tfull + b, tph, f.err) ? 1 : 0;
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
      tc::fence_after_sync();
      const int cur = it.s & 1;
      const FusedJobMaps& m = mp.job[it.j];
      const CUtensorMap* D = it.p == 0 ? &m.ae : (it.p == 1 ? &m.be : (it.s == f.steps - 1 ? &m.oe : &m.xe[cur ^ 1]));
      // statistics slot (when wanted): the tile's index within its matrix, then 8 per tile
      const int st_slot = a.st_sum != nullptr ? (it.ti + it.tj * a.tiles_m) * 8 + (warp - 2) : -1;
      epi_tile_tma<false, 1>(a, D, mine, tmem + (static_cast<uint32_t>(32 * quad) << 16) + static_cast<uint32_t>(b * BN),
                             it.ti * BM + 32 * quad, it.tj, it.mb, false, lane, last_par, 4 * half, 4 * half + 4,
                             nullptr, st_slot, it.s == 0);
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

// ---------------------------------------------------------------------- launcher

// One launch of the fused kernel for every step of f.n_jobs groups (see ns_fused_kernel): each
// job's prod[0..3] hold X X', B', B'X and the last step's B'X with everything but their tile
// counts.
zopt_status launch_fused(const FusedMaps& maps, FusedArgs f, cudaStream_t stream) {
  ZOPT_CUDA_TRY(once([] {
    return cudaFuncSetAttribute(ns_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes(kEpiTma));
  }));
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

}  // namespace ns
}  // namespace zopt
