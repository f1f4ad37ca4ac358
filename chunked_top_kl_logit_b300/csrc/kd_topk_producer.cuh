// Teacher-side top-K cache producer: the SIMT steps after the contraction
// (aipuls.nl summary of "Making Knowledge Distillation Cheap Enough to Run at
// Scale", section "Summary": the teacher's top-100 logits per position are
// cached offline).
//
// Every logit z_tv gets the unique 64-bit key (order(z), ~v): larger logit
// first, then the lower vocabulary index.  The contraction (EPI_TMAX) records
// each vocabulary tile's largest key and stores the chunk's fp32 logits.  The
// K-th largest of those tile maxima, theta, is a lower bound of the row's K-th
// largest key (the K tiles with the largest maxima hold K distinct keys >=
// theta), and only the fewer than K tiles whose maximum exceeds theta, plus
// theta itself, can hold keys >= theta: at most (K - 1) * 256 + 1 candidates.
// The scan kernel collects them from the stored logits; the finalize kernel
// selects the K largest candidate keys exactly and writes them in descending
// order.
#pragma once

#include <math_constants.h>
#include <stdint.h>

#include "kd_ptx.cuh"

namespace kd {

// k-th largest (k >= 1) of n >= k unique 64-bit keys, one warp, MSB-first
// radix select with 8-bit digits; hist = 256 words of this warp's shared memory.
__device__ __forceinline__ uint64_t warp_kth_largest(const uint64_t* keys, int n, int k,
                                                     uint32_t* hist) {
  const int lane = threadIdx.x & 31;
  uint64_t prefix = 0ull, mask = 0ull;
  uint32_t need = static_cast<uint32_t>(k);
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = lane; i < 256; i += 32) hist[i] = 0u;
    __syncwarp();
    for (int i = lane; i < n; i += 32) {
      const uint64_t key = keys[i];
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncwarp();
    // lane l owns digits 255 - 8l .. 248 - 8l; counts from the top digit down
    uint32_t own = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) own += hist[255 - 8 * lane - j];
    uint32_t incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t excl = incl - own;
    const bool mine = excl < need && incl >= need;
    uint32_t dg = 0u, rem = 0u;
    if (mine) {
      uint32_t cum = excl;
      for (int j = 0; j < 8; ++j) {
        const int dd = 255 - 8 * lane - j;
        if (cum + hist[dd] >= need) {
          dg = static_cast<uint32_t>(dd);
          rem = need - cum;
          break;
        }
        cum += hist[dd];
      }
    }
    const unsigned owner = __ballot_sync(0xffffffffu, mine);
    const int src = owner ? __ffs(owner) - 1 : 0;
    dg = __shfl_sync(0xffffffffu, dg, src);
    rem = __shfl_sync(0xffffffffu, rem, src);
    prefix |= static_cast<uint64_t>(dg) << shift;
    mask |= 0xFFull << shift;
    need = rem;
    __syncwarp();
  }
  return prefix;
}

constexpr int TOPK_WARPS = 8;  // rows per block of the SIMT kernels

// One warp per row of the chunk: the threshold key (theta = 0, i.e. every
// logit a candidate, when the row has fewer than K tiles), its logit value,
// and the row's full-vocabulary lse of z / tau from the tile partials.  A NaN
// or +inf logit makes its tile's partial NaN (and a tile of -inf logits gives
// one too), so a row whose lse is not finite is flagged: theta_val = NaN,
// which no logit passes in the scan, and KD_ERR_NONFINITE.
__global__ void kd_topk_threshold_kernel(const uint64_t* __restrict__ tkeys,
                                         const float* __restrict__ part, int64_t part_ld,
                                         int rows, int n_tiles, int K,
                                         uint64_t* __restrict__ theta,
                                         float* __restrict__ theta_val,
                                         float* __restrict__ full_lse, int* status) {
  __shared__ uint32_t hist[TOPK_WARPS][256];
  const int wid = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * TOPK_WARPS + wid;
  if (row >= rows) return;  // whole warp
  uint64_t th = 0ull;
  if (K <= n_tiles) th = warp_kth_largest(tkeys + static_cast<int64_t>(row) * n_tiles, n_tiles, K,
                                          hist[wid]);
  // lse: lane-strided online logsumexp, then a fixed-order butterfly
  float m = -CUDART_INF_F, s = 0.f;
  for (int j = lane; j < n_tiles; j += 32) {
    const float x = part[static_cast<int64_t>(j) * part_ld + row];
    if (x > m) {
      s = s * expf(m - x) + 1.f;
      m = x;
    } else {
      s += expf(x - m);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float mn = fmaxf(m, m2);
    s = (mn == -CUDART_INF_F) ? 0.f : s * expf(m - mn) + s2 * expf(m2 - mn);
    m = mn;
  }
  if (lane == 0) {
    const float lse = m + logf(s);
    const bool finite = isfinite(lse);
    theta[row] = th;
    theta_val[row] = !finite ? CUDART_NAN_F
                   : th     ? float_from_order_key(static_cast<uint32_t>(th >> 32))
                            : -CUDART_INF_F;
    if (full_lse) full_lse[row] = finite ? lse : CUDART_NAN_F;
    if (!finite) set_status(status, KD_ERR_NONFINITE);
  }
}

constexpr int SCAN_THREADS = 256;  // one block per row of the chunk

// One block per row: every stored logit whose key is at least the row's
// threshold becomes a candidate (appended in no particular order; the
// finalize kernel sorts).  z holds the row's V logits (V a multiple of 8, rows
// 32-byte aligned); the value test discards almost every logit before a key is
// formed.
__global__ void __launch_bounds__(SCAN_THREADS)
    kd_topk_scan_kernel(const float* __restrict__ z, int64_t ldz, int V,
                        const uint64_t* __restrict__ theta, const float* __restrict__ theta_val,
                        uint64_t* __restrict__ cand, int* __restrict__ cand_cnt, int cand_cap,
                        int* status) {
  const int row = blockIdx.x;
  const uint64_t th = theta[row];
  const float tv = theta_val[row];
  const float4* z4 = reinterpret_cast<const float4*>(z + static_cast<int64_t>(row) * ldz);
  const int n4 = V >> 2;
  constexpr int U = 4;  // independent 16-byte loads in flight per thread
  for (int base = threadIdx.x; base < n4; base += U * SCAN_THREADS) {
    float4 q[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * SCAN_THREADS;
      q[u] = i < n4 ? __ldcs(z4 + i) : make_float4(-CUDART_INF_F, -CUDART_INF_F,
                                                   -CUDART_INF_F, -CUDART_INF_F);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * SCAN_THREADS;
      const float xs[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (i < n4 && xs[e] >= tv) {  // rare: only near the row's top-K
          const uint64_t key = logit_key(xs[e], 4 * i + e);
          if (key >= th) {
            const int pos = atomicAdd(cand_cnt + row, 1);
            if (pos < cand_cap)
              cand[static_cast<int64_t>(row) * cand_cap + pos] = key;
            else
              set_status(status, KD_ERR_INTERNAL);
          }
        }
      }
    }
  }
}

// One warp per row: the K largest candidate keys, in descending order.  A row
// flagged non-finite (theta_val NaN), or one with fewer than K candidates
// (which the threshold bound rules out for finite rows: KD_ERR_INTERNAL), is
// written as index -1 and value NaN; no candidate slot past the row's count
// is ever read.
__global__ void kd_topk_finalize_kernel(uint64_t* __restrict__ cand,
                                        const int* __restrict__ cand_cnt, int cand_cap,
                                        const float* __restrict__ theta_val, int rows, int K,
                                        int32_t* __restrict__ out_idx,
                                        float* __restrict__ out_val, int* status) {
  __shared__ uint32_t hist[TOPK_WARPS][256];
  const int wid = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * TOPK_WARPS + wid;
  if (row >= rows) return;
  uint64_t* c = cand + static_cast<int64_t>(row) * cand_cap;
  const int n = min(cand_cnt[row], cand_cap);
  int32_t* oi = out_idx + static_cast<int64_t>(row) * K;
  float* ov = out_val + static_cast<int64_t>(row) * K;
  const bool flagged = isnan(theta_val[row]);
  if (flagged || n < K) {  // warp-uniform
    if (!flagged && lane == 0) set_status(status, KD_ERR_INTERNAL);
    for (int i = lane; i < K; i += 32) {
      oi[i] = -1;
      ov[i] = CUDART_NAN_F;
    }
    return;
  }
  const uint64_t kth = warp_kth_largest(c, n, K, hist[wid]);
  // move the K keys >= kth to the front (reads of a 32-key block precede its
  // writes, and writes never pass the block being read)
  int w = 0;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    const uint64_t key = i < n ? c[i] : 0ull;
    const bool sel = i < n && key >= kth;
    const unsigned b = __ballot_sync(0xffffffffu, sel);
    __syncwarp();
    if (sel) c[w + __popc(b & ((1u << lane) - 1u))] = key;
    w += __popc(b);
    __syncwarp();
  }
  // rank by pairwise comparison among the K and write in descending order
  for (int i = lane; i < K; i += 32) {
    const uint64_t key = c[i];
    int r = 0;
    for (int j = 0; j < K; ++j) r += c[j] > key;
    oi[r] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
    ov[r] = float_from_order_key(static_cast<uint32_t>(key >> 32));
  }
}

}  // namespace kd
