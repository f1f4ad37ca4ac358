// Teacher-entropy token filter: the mask producer in front of the loss.
//
// asibiont.com rewrite, "Distillation Token Filtering": score each token by
// the entropy of the teacher's distribution and, per batch, keep a fixed
// percentage of the tokens with the highest entropy.  Here the distribution is
// the renormalised top-K softmax at temperature tau (the one the loss uses),
// H_t = -sum_k p_tk log p_tk; among rows with valid_in != 0 the
// n_keep = ceil(N_in * keep_num / keep_den) rows of largest H are kept, equal
// entropies ordered by row index (lower first).  The selection is exact and
// deterministic: an MSB-first radix select over order-preserving 32-bit keys
// of H, then an ordered scan that admits the threshold's ties by row.
#pragma once

#include <math_constants.h>
#include <stdint.h>

#include "kd_ptx.cuh"

namespace kd {

// One warp per row: H_t and its key; rows that are not candidates
// (valid_in == 0) get key 0, which no finite entropy maps to.
__global__ void kd_entropy_kernel(const float* __restrict__ tl, const uint8_t* __restrict__ valid_in,
                                  int T, int K, float inv_tau, float* __restrict__ entropy,
                                  uint32_t* __restrict__ keys) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= T) return;
  const float* tr = tl + static_cast<int64_t>(row) * K;
  float m = -CUDART_INF_F;
  for (int k = lane; k < K; k += 32) m = fmaxf(m, tr[k] * inv_tau);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float S = 0.f;
  for (int k = lane; k < K; k += 32) S += expf(tr[k] * inv_tau - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
  const float logS = logf(S);
  float H = 0.f;
  for (int k = lane; k < K; k += 32) {
    const float lp = tr[k] * inv_tau - m - logS;
    const float pk = expf(lp);
    if (pk > 0.f) H -= pk * lp;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) H += __shfl_xor_sync(0xffffffffu, H, o);
  if (lane == 0) {
    if (entropy) entropy[row] = H;
    keys[row] = valid_in[row] ? float_order_key(H) : 0u;
  }
}

constexpr int FILTER_THREADS = 1024;

// Histogram of the digit (k >> shift) & 255 over candidate keys (k != 0) whose
// bits under `mask` equal `prefix`.  Keys are read four at a time; `keys` has
// room for T rounded up to a multiple of 4 (the tail is read as key 0).
__device__ __forceinline__ void filter_histogram(const uint32_t* __restrict__ keys, int T,
                                                 uint32_t mask, uint32_t prefix, int shift,
                                                 uint32_t* hist) {
  const int n4 = (T + 3) >> 2;
  const uint4* k4 = reinterpret_cast<const uint4*>(keys);
#pragma unroll 4
  for (int i = threadIdx.x; i < n4; i += FILTER_THREADS) {
    const uint4 v = k4[i];
    const int t = i << 2;
    const uint32_t kk[4] = {v.x, t + 1 < T ? v.y : 0u, t + 2 < T ? v.z : 0u, t + 3 < T ? v.w : 0u};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (kk[j] != 0u && (kk[j] & mask) == prefix) atomicAdd(&hist[(kk[j] >> shift) & 255u], 1u);
  }
}

// Single block: count the candidates, radix-select the n_keep-th largest key
// among them, then write the mask (ties at the threshold by row order).
__global__ void __launch_bounds__(FILTER_THREADS, 1)
    kd_entropy_select_kernel(const uint32_t* __restrict__ keys, int T, int keep_num,
                             int keep_den, uint8_t* __restrict__ valid_out) {
  __shared__ uint32_t hist[256];
  __shared__ int warp_sum[FILTER_THREADS / 32];
  __shared__ uint32_t s_prefix, s_remaining, s_eq_total;
  __shared__ int s_base;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int wid = tid >> 5;

  // N_in
  int cnt = 0;
  for (int t = tid; t < T; t += FILTER_THREADS) cnt += keys[t] != 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if (lane == 0) warp_sum[wid] = cnt;
  __syncthreads();
  if (tid == 0) {
    long long n_in = 0;
    for (int w = 0; w < FILTER_THREADS / 32; ++w) n_in += warp_sum[w];
    const long long n_keep = (n_in * keep_num + keep_den - 1) / keep_den;
    s_remaining = static_cast<uint32_t>(n_keep);
    s_prefix = 0u;
    s_eq_total = 0u;
  }
  __syncthreads();
  const uint32_t n_keep = s_remaining;

  // radix select, 8 bits per pass from the top: afterwards s_prefix is the key
  // of the n_keep-th largest candidate, s_remaining the number of rows with
  // exactly that key that are kept and s_eq_total the number of candidates
  // with that key
  uint32_t mask = 0u;
  if (n_keep > 0) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += FILTER_THREADS) hist[i] = 0u;
      __syncthreads();
      const uint32_t prefix = s_prefix;
      filter_histogram(keys, T, mask, prefix, shift, hist);
      __syncthreads();
      if (wid == 0) {
        // lane l owns digits 255 - 8l .. 248 - 8l (descending); suffix counts
        // from the top are an inclusive scan over lanes
        uint32_t own = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) own += hist[255 - 8 * lane - j];
        uint32_t incl = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t need = s_remaining;
        const uint32_t excl = incl - own;
        if (excl < need && incl >= need) {  // exactly one lane holds the digit
          uint32_t cum = excl;
          for (int j = 0; j < 8; ++j) {
            const int dg = 255 - 8 * lane - j;
            if (cum + hist[dg] >= need) {
              s_prefix = prefix | (static_cast<uint32_t>(dg) << shift);
              s_remaining = need - cum;
              s_eq_total = hist[dg];
              break;
            }
            cum += hist[dg];
          }
        }
      }
      mask |= 255u << shift;
      __syncthreads();
    }
  }
  const uint32_t theta = s_prefix;
  const uint32_t k_eq = s_remaining;

  // mask: keys above the threshold, and the first k_eq rows (in row order)
  // whose key equals it; when every row with the threshold key is kept the
  // order does not matter and no scan is needed
  if (n_keep == 0 || s_eq_total == k_eq) {
    for (int t = tid; t < T; t += FILTER_THREADS) {
      const uint32_t k = keys[t];
      valid_out[t] = (n_keep > 0 && k != 0u && k >= theta) ? 1 : 0;
    }
    return;
  }
  if (tid == 0) s_base = 0;
  __syncthreads();
  for (int t0 = 0; t0 < T; t0 += FILTER_THREADS) {
    const int t = t0 + tid;
    const uint32_t k = t < T ? keys[t] : 0u;
    const int eq = (k != 0u && k == theta) ? 1 : 0;
    int x = eq;  // inclusive scan of eq over the block, in row order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sum[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int v = warp_sum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      warp_sum[lane] = v;
    }
    __syncthreads();
    const int before = s_base + (wid > 0 ? warp_sum[wid - 1] : 0) + x - eq;
    if (t < T) {
      const bool keep = k != 0u && (k > theta || (eq && before < static_cast<int>(k_eq)));
      valid_out[t] = keep ? 1 : 0;
    }
    __syncthreads();
    if (tid == 0) s_base += warp_sum[FILTER_THREADS / 32 - 1];
    __syncthreads();
  }
}

}  // namespace kd
