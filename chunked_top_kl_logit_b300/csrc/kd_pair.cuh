// CTA-pair contraction pipeline (tcgen05.mma.cta_group::2), kept separate
// from kd_gemm_kernel: C = A B^T with K-major bf16 operands and an fp32 tile
// store, used by the diagnostic entry kd_gemm_bf16_diag_pair.
//
// A cluster of two CTAs computes each 256 x BN tile with one MMA per 16-deep
// k-slice: CTA rank r loads rows [128 r, 128 r + 128) of the A tile and rows
// [r BN/2, (r + 1) BN/2) of the B tile into its own shared memory, and holds
// rows [128 r, 128 r + 128) of the fp32 accumulator in its own tensor memory.
// The even CTA (the leader) arms one barrier per stage with both CTAs' bytes,
// issues the MMAs and commits them to the barriers of both CTAs; each epilogue
// warp returns its accumulator to the leader with a cluster-scoped arrive.
// Every wait is bounded like the single-CTA kernel's; barrier set-up and
// tear-down are cluster-synchronised so that no cross-CTA access outlives
// either CTA.  (Under the 1.1 kW power cap this schedule made the loss step
// slower, so the loss runs one CTA per tile.)
#pragma once

#include "kd_kernels.cuh"

namespace kd {

__device__ __forceinline__ void pair_producer(const GemmParams& p, const CUtensorMap* tmA,
                                              const CUtensorMap* tmB, uint8_t* smem,
                                              uint64_t* full, uint64_t* empty,
                                              volatile int* abort_flag, uint32_t rank, int first,
                                              int stride) {
  tma_prefetch_desc(tmA);
  tma_prefetch_desc(tmB);
  const Sched sc{p.m_tiles, p.n_tiles, p.num_tiles, p.k_steps, p.ks_per_split, 1, p.M, p.N};
  int stage = 0;
  uint32_t phase = 0;
  int issued = 0;
  bool ok = true;
  for (int t = first; t < p.num_tiles && ok; t += stride) {
    TileCoord c = decode_tile(p, sc, t);
    c.m = 2 * c.m + static_cast<int>(rank);
    for (int ks = 0; ks < p.k_steps; ++ks) {
      if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
      uint8_t* sa = smem + static_cast<size_t>(stage) * p.stage_bytes;
      uint8_t* sb = sa + p.a_bytes;
      // both CTAs' bytes complete on the leader's barrier, which the leader arms
      if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2u * p.stage_bytes);
      const uint32_t fbar = mapa_shared(smem_u32(&full[stage]), 0);
      tma_load_2d_pair(sa, tmA, fbar, ks * BK, c.m * BM);
      tma_load_2d_pair(sb, tmB, fbar, ks * BK, c.n * p.BN + static_cast<int>(rank) * (p.BN / 2));
      ++issued;
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
  }
  if (!ok) {
    if (rank == 0) {
      for (int i = max(0, issued - p.stages); i < issued; ++i)
        mbar_wait_drain(&full[i % p.stages], static_cast<uint32_t>((i / p.stages) & 1));
    } else {
      __nanosleep(200000);  // the leader's barrier counts these loads
    }
    return;
  }
  // every stage's last fill has been released by the leader's commits (arrivals
  // into this CTA's barriers) before the pair tears down
  for (int i = 0; i < p.stages; ++i) {
    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) break;
    if (++stage == p.stages) { stage = 0; phase ^= 1u; }
  }
}

__device__ __forceinline__ void pair_mma(const GemmParams& p, uint8_t* smem, uint64_t* full,
                                         uint64_t* tfull, uint64_t* empty, uint64_t* tempty,
                                         uint64_t* drain, uint32_t tmem_base,
                                         volatile int* abort_flag, int first, int stride) {
  const uint32_t smem0 = smem_u32(smem);
  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  int lt = 0;
  for (int t = first; t < p.num_tiles; t += stride, ++lt) {
    const int acc = lt & 1;
    const uint32_t use = static_cast<uint32_t>(lt >> 1);
    if (!mbar_wait(&tempty[acc], (use & 1u) ^ 1u, abort_flag, p.status)) { ok = false; break; }
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 256);
    for (int ks = 0; ks < p.k_steps; ++ks) {
      if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sa = smem0 + static_cast<uint32_t>(stage) * p.stage_bytes;
      const uint32_t sb = sa + p.a_bytes;
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk)
        umma_bf16_pair(d_tmem, make_sdesc(sa + kk * 32u, 16u, 1024u),
                       make_sdesc(sb + kk * 32u, 16u, 1024u), p.idesc,
                       (ks > 0 || kk > 0) ? 1u : 0u);
      umma_commit_pair_both(&empty[stage]);
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
    if (!ok) break;
    umma_commit_pair_both(&tfull[acc]);
  }
  if (!ok) {
    umma_commit_pair_both(drain);
    mbar_wait_drain(drain, 0);
  }
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    kd_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(p.stages) * p.stage_bytes);
  uint64_t* empty = full + MAX_STAGES;
  uint64_t* tfull = empty + MAX_STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int first = static_cast<int>(blockIdx.x >> 1);
  const int stride = static_cast<int>(gridDim.x >> 1);
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);  // one lane per epilogue warp, two CTAs
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  cluster_sync();  // both CTAs' barriers exist before either touches the other's
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) pair_producer(p, &tmA, &tmB, smem, full, empty, abort_flag, rank, first, stride);
  } else if (warp == 1) {
    if (lane == 0 && rank == 0)
      pair_mma(p, smem, full, tfull, empty, tempty, drain, tmem_base, abort_flag, first, stride);
  } else {
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const uint32_t tmem_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const Sched sc{p.m_tiles, p.n_tiles, p.num_tiles, p.k_steps, p.ks_per_split, 1, p.M, p.N};
    const uint32_t leader_tempty0 = mapa_shared(smem_u32(&tempty[0]), 0);
    int lt = 0;
    for (int t = first; t < p.num_tiles; t += stride, ++lt) {
      TileCoord c = decode_tile(p, sc, t);
      c.m = 2 * c.m + static_cast<int>(rank);
      const int acc = lt & 1;
      const uint32_t use = static_cast<uint32_t>(lt >> 1);
      const int row = c.m * BM + q * 32 + lane;
      const bool w = mbar_wait(&tfull[acc], use & 1u, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, w)) break;
      tc_fence_after();
      float* orow = p.out + static_cast<int64_t>(row) * p.ld_out;
#pragma unroll 1
      for (int cc = 0; cc < p.BN / 32; ++cc) {
        const int cb = c.n * p.BN + cc * 32;
        if (cb >= p.N) break;
        uint32_t r[32];
        tmem_ld32(tmem_row + static_cast<uint32_t>(acc * 256 + cc * 32), r);
        tmem_ld_wait(r);
        if (row < p.M) {
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const int col = cb + 4 * q4;
            if (col < p.N)
              *reinterpret_cast<float4*>(orow + col) =
                  make_float4(__uint_as_float(r[4 * q4 + 0]), __uint_as_float(r[4 * q4 + 1]),
                              __uint_as_float(r[4 * q4 + 2]), __uint_as_float(r[4 * q4 + 3]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(leader_tempty0 + static_cast<uint32_t>(acc * 8));
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no cross-CTA access is left in flight
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace kd
