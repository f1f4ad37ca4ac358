// Device kernels of the fused top-K KL loss.
//
// The contraction kernel is one persistent, warp-specialised tcgen05 GEMM
// (tile 128 x BN x 64, bf16 in, fp32 accumulate in TMEM) shared by the
// contractions of the method and of the teacher-side cache producer:
//
//   forward   z = h W^T tile by tile       -> EPI_FWD: online log-sum-exp partial
//                                             per (row, vocab tile) and the gather
//                                             of z at the row's cached indices
//   backward  z = h_c W^T again (chunk c)  -> EPI_DZ: G = s (q - scatter p) / tau
//                                             as bf16 into the chunk buffer
//             dh_c^T = W^T G_c^T           -> EPI_DH: transposed store through the
//                                             valid-row map (split over V on demand)
//             dW^T  += h_c^T G_c           -> EPI_DW: TMA store / reduce-add of
//                                             staged 32 x 32 pieces
//   teacher   z = h_t W_t^T                -> EPI_TMAX: tile maxima, lse partials and
//                                             the fp32 logits of the chunk (TMA store
//                                             of staged 32 x 32 pieces)
//   (diagnostic C = A B^T                  -> EPI_STORE)
//
// Warp roles (192 threads): warp 0 issues TMA loads into a ring of shared
// memory stages, warp 1 owns TMEM and issues tcgen05.mma from one thread,
// warps 2..5 drain the two TMEM accumulators (one TMEM lane = one tile row
// per thread) while the next tile accumulates into the other one.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "kd_ptx.cuh"

namespace kd {

constexpr int BM = 128;            // tile rows = TMEM lanes
constexpr int BK = 64;             // contraction elements per stage (128 B of bf16)
constexpr int ZBN = 256;           // logit tile width over the vocabulary
constexpr int TMEM_COLS = 512;     // two accumulators of up to 256 fp32 columns
constexpr int NUM_THREADS = 192;   // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int MAX_STAGES = 8;
constexpr int DW_PIECE_FLOATS = 32 * 32;  // one 4 KB epilogue staging buffer (EPI_DZ, EPI_DW)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// EPI_STORE: plain fp32 tile store (diagnostic GEMM).  EPI_DH / EPI_DW: the
// two gradient contractions, computed transposed (output rows = hidden units,
// so the stores run along d and coalesce) and written through the row map /
// accumulated; they differ only in schedule, and are separate instantiations
// so that profiles tell them apart.
// EPI_TMAX: the contraction of the teacher-side top-K producer.
// EPI_FWD_RESID: the forward of the residual-mass variant, whose lse partials
// cover only the columns outside the row's cache.  EPI_FWDZ: the forward of
// the single-sweep training step on one chunk of rows (valid rows first),
// which also stores the valid rows' logits as bf16 exp((z - o) / tau) for the
// gradient contractions.  EPI_FWDZ_RESID: the same for the residual-mass
// variant (lse partials over the columns outside the cache).
enum EpiMode {
  EPI_FWD = 0,
  EPI_DZ = 1,
  EPI_STORE = 2,
  EPI_DH = 3,
  EPI_DW = 4,
  EPI_TMAX = 5,
  EPI_FWD_RESID = 6,
  EPI_FWDZ = 7,
  EPI_FWDZ_RESID = 8
};

struct GemmParams {
  // schedule: tile t -> (split s, m tile, n tile)
  int m_tiles, n_tiles, splits, num_tiles;
  int k_steps;        // contraction length in steps of BK
  int ks_per_split;   // steps per split (the last split may be shorter, never empty)
  int group_m;        // n_fast == 0: m tiles per raster group (n-major inside a group)
  int n_fast;         // 1: n is the fastest index inside a split
  // operands
  int a_mn, b_mn;     // 0: K-major tile, 1: MN-major tile
  int BN;             // tile width (MMA N)
  int stages;
  uint32_t epi_smem;  // shared-memory bytes of the epilogue's staging buffers
  uint32_t a_bytes, b_bytes, stage_bytes;
  uint32_t idesc;
  // epilogue, all modes
  int M, N;           // valid output rows / columns of this launch
  int* status;
  // EPI_STORE: split 0 writes `out`, split s >= 1 writes `out2 + (s-1)*split_stride`
  float* out;
  float* out2;
  int64_t ld_out;
  int64_t split_stride;
  int accumulate;     // add into the existing values of `out`
  // EPI_FWD / EPI_DZ (per-row tables are indexed by the global row row0 + local row)
  int row0;
  int K;
  const int* sidx;        // [T][K] teacher indices, ascending per row
  const float* sp;        // [T][K] teacher probabilities in the same order
  const int16_t* sslot;   // [T][K] original slot of each sorted entry
  float inv_tau;          // 1 / tau
  float c_log2;           // log2(e) / tau
  int64_t part_ld;        // row stride (= T) of the partial table
  float* part;            // [n_tiles][T] natural-log lse of each vocabulary tile
  float* zg;              // [T][K] z / tau gathered at the sorted entries
  int* gidx;              // [T][K] (slot order) vocabulary column read, or null
  const float* lse;       // [T]
  const float* resid;     // [T] teacher mass outside the cached entries, or null (main loss)
  const float* outside_mass; // [T] student mass outside the cached entries (with resid)
  const uint8_t* valid;   // [T]
  const int* nvalid;      // device scalar
  float grad_loss;
  __nv_bfloat16* dz;      // [rows][dz_ld] chunk buffer
  int64_t dz_ld;
  // Row counts known only on the device (the backward works on the valid rows
  // only): rows = clamp(*dyn_count - dyn_base, 0, dyn_cap).  dyn_kind 0: static
  // shape; 1: rows are the M dimension; 2: rows are the contraction (splits == 1);
  // 3: rows are the N dimension.
  const int* dyn_count;
  int dyn_base, dyn_cap, dyn_kind;
  // Compact row -> original row, rowmap[rowmap_base + local row]; null = identity.
  const int* rowmap;
  int rowmap_base;
  // Split count chosen on the device (dyn_kind 3 with splits > 1): at most
  // `splits`, limited so that (S - 1) partial blocks of n_tiles*BN rows fit in
  // part_rows rows, scored for policy_sms CTAs.  CTA 0 publishes
  // {S, n_tiles*BN} in split_info for the reduction that follows.
  int part_rows, policy_sms;
  int* split_info;
  // Teacher top-K producer (per row of the launch): the key of each vocabulary
  // tile's largest logit goes to tkeys[row * n_tiles + tile]; the logits
  // themselves leave through the output tensor map (rows x vocabulary, fp32).
  uint64_t* tkeys;
  // EPI_FWDZ (single sweep): the offset o of each local row (a raw logit) that
  // the stored values exp((z - o) / tau) are relative to, and the chunk's
  // flag, set when a stored value would leave the range that the later steps
  // can take (the chunk's G is then recomputed from the known lse).
  const float* roff;
  int* ovf;
  // EPI_DH: per-column (local chunk row) factor applied to the stored tile, or
  // null.  EPI_DW: device scalar factor applied to the stored tile, or null.
  const float* cscale;
  const float* oscale;
  // Launch gate: with gate != null the whole launch returns at once unless
  // *gate != 0 (set on the device by an earlier kernel of the stream).
  const int* gate;
};

// Largest c (zc - o) (log2 units) that a stored value may reach before the
// chunk is flagged for recompute: 2^64 keeps the values, the sums of the dh
// contraction and the scales exp(o / tau - lse) inside fp32 / bf16 range.
constexpr float YREL_MAX_LOG2 = 64.f;
// Smallest |1 - R/Q| the residual variant's single sweep carries as a row
// factor (its cached columns are stored divided by it).
constexpr float YREL_MIN_FACTOR = 1.f / 65536.f;

// Per-launch schedule, resolved on the device at kernel start.
struct Sched {
  int m_tiles, n_tiles, num_tiles, k_steps, ks_per_split, splits, M, N;
};

// Longest contraction slab of a split dh (in BK steps): 51200 vocabulary columns.
constexpr int DH_SLAB_STEPS = 800;

// Split count for `tiles` output tiles over `k_steps` contraction steps: the
// fewest splits whose (tile, split) units fill the policy's CTA count to 95%,
// else the best fill; each split keeps at least 32 steps.
__host__ __device__ inline int pick_splits(int tiles, int k_steps, int max_splits, int sms) {
  if (tiles <= 0 || sms <= 0) return 1;
  int best = 1;
  double best_eff = 0.0;
  for (int s = 1; s <= max_splits; ++s) {
    if (s > 1 && k_steps / s < 32) break;
    const long long units = static_cast<long long>(tiles) * s;
    const long long waves = (units + sms - 1) / sms;
    const double eff = static_cast<double>(units) / static_cast<double>(waves * sms);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = s;
    }
    if (eff >= 0.95) break;
  }
  return best;
}

__device__ __forceinline__ Sched make_sched(const GemmParams& p) {
  Sched s{p.m_tiles, p.n_tiles, p.num_tiles, p.k_steps, p.ks_per_split, p.splits, p.M, p.N};
  if (p.dyn_kind != 0) {
    const int rows = max(0, min(*p.dyn_count - p.dyn_base, p.dyn_cap));
    if (p.dyn_kind == 1) {
      s.M = rows;
      s.m_tiles = (rows + BM - 1) / BM;
      s.num_tiles = s.m_tiles * s.n_tiles * s.splits;
    } else if (p.dyn_kind == 2) {
      s.k_steps = (rows + BK - 1) / BK;
      s.ks_per_split = s.k_steps;
    } else {
      s.N = rows;
      s.n_tiles = (rows + p.BN - 1) / p.BN;
      if (p.splits > 1) {
        const int pad = s.n_tiles * p.BN;
        int smax = p.splits;
        if (pad > 0) smax = min(smax, 1 + p.part_rows / pad);
        s.splits = pick_splits(s.m_tiles * s.n_tiles, s.k_steps, smax, p.policy_sms);
        // a long contraction is also cut into slabs of at most DH_SLAB_STEPS steps:
        // the split-major tile order then keeps the co-running CTAs on one slab of
        // the operands, which stays in L2 (dh's DRAM re-reads fall)
        s.splits = max(s.splits, min(smax, (s.k_steps + DH_SLAB_STEPS - 1) / DH_SLAB_STEPS));
        s.ks_per_split = (s.k_steps + s.splits - 1) / s.splits;
        if (p.split_info && blockIdx.x == 0 && threadIdx.x == 0) {
          p.split_info[0] = s.splits;
          p.split_info[1] = pad;
        }
      }
      s.num_tiles = s.m_tiles * s.n_tiles * s.splits;
    }
  }
  return s;
}

struct TileCoord {
  int m, n, s;
};

__device__ __forceinline__ TileCoord decode_tile(const GemmParams& p, const Sched& sc, int t) {
  const int per_split = sc.m_tiles * sc.n_tiles;
  TileCoord c;
  c.s = t / per_split;
  const int r = t - c.s * per_split;
  if (p.n_fast) {
    c.m = r / sc.n_tiles;
    c.n = r - c.m * sc.n_tiles;
  } else {
    const int gsz = p.group_m * sc.n_tiles;
    const int g = r / gsz;
    const int m0 = g * p.group_m;
    const int gm = min(p.group_m, sc.m_tiles - m0);
    const int j = r - g * gsz;
    c.n = j / gm;
    c.m = m0 + (j - c.n * gm);
  }
  return c;
}

// First position in the ascending row `s[0..K)` whose value is >= key.
__device__ __forceinline__ int lower_bound_row(const int* __restrict__ s, int K, int key) {
  int lo = 0, hi = K;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(s + mid) < key) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// ------------------------------------------------------------------ roles

__device__ __forceinline__ void producer_role(const GemmParams& p, const Sched& sc,
                                              const CUtensorMap* tmA,
                                              const CUtensorMap* tmB, uint8_t* smem,
                                              uint64_t* full, uint64_t* empty,
                                              volatile int* abort_flag) {
  tma_prefetch_desc(tmA);
  tma_prefetch_desc(tmB);
  int stage = 0;
  uint32_t phase = 0;
  int issued = 0;
  bool ok = true;
  for (int t = blockIdx.x; t < sc.num_tiles && ok; t += gridDim.x) {
    const TileCoord c = decode_tile(p, sc, t);
    const int kb = c.s * sc.ks_per_split;
    const int ke = min(sc.k_steps, kb + sc.ks_per_split);
    for (int ks = kb; ks < ke; ++ks) {
      if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
      uint8_t* sa = smem + static_cast<size_t>(stage) * p.stage_bytes;
      uint8_t* sb = sa + p.a_bytes;
      mbar_arrive_expect_tx(&full[stage], p.stage_bytes);
      const int k0 = ks * BK;
      if (!p.a_mn) {
        tma_load_2d(sa, tmA, &full[stage], k0, c.m * BM);
      } else {
        tma_load_2d(sa, tmA, &full[stage], c.m * BM, k0);
        tma_load_2d(sa + 8192, tmA, &full[stage], c.m * BM + 64, k0);
      }
      if (!p.b_mn) {
        tma_load_2d(sb, tmB, &full[stage], k0, c.n * p.BN);
      } else {
        for (int j = 0; j < p.BN / 64; ++j)
          tma_load_2d(sb + j * 8192, tmB, &full[stage], c.n * p.BN + 64 * j, k0);
      }
      ++issued;
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
  }
  if (!ok) {
    // let the loads this thread started land before the CTA leaves
    for (int i = max(0, issued - p.stages); i < issued; ++i)
      mbar_wait_drain(&full[i % p.stages], static_cast<uint32_t>((i / p.stages) & 1));
  }
}

__device__ __forceinline__ void mma_role(const GemmParams& p, const Sched& sc, uint8_t* smem,
                                         uint64_t* full,
                                         uint64_t* empty, uint64_t* tfull, uint64_t* tempty,
                                         uint64_t* drain, uint32_t tmem_base,
                                         volatile int* abort_flag) {
  const uint32_t a_lbo = p.a_mn ? 8192u : 16u;
  const uint32_t b_lbo = p.b_mn ? 8192u : 16u;
  const uint32_t a_adv = p.a_mn ? 2048u : 32u;  // bytes per 16-element K step
  const uint32_t b_adv = p.b_mn ? 2048u : 32u;
  const uint32_t smem0 = smem_u32(smem);
  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  int lt = 0;
  for (int t = blockIdx.x; t < sc.num_tiles; t += gridDim.x, ++lt) {
    const TileCoord c = decode_tile(p, sc, t);
    const int kb = c.s * sc.ks_per_split;
    const int ke = min(sc.k_steps, kb + sc.ks_per_split);
    const int acc = lt & 1;
    const uint32_t use = static_cast<uint32_t>(lt >> 1);
    if (!mbar_wait(&tempty[acc], (use & 1u) ^ 1u, abort_flag, p.status)) { ok = false; break; }
    tc_fence_after();
    if (kb >= ke) {          // empty contraction: the epilogue writes zeros, no MMA
      mbar_arrive(&tfull[acc]);
      continue;
    }
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 256);
    for (int ks = kb; ks < ke; ++ks) {
      if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sa = smem0 + static_cast<uint32_t>(stage) * p.stage_bytes;
      const uint32_t sb = sa + p.a_bytes;
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        const uint64_t ad = make_sdesc(sa + kk * a_adv, a_lbo, 1024u);
        const uint64_t bd = make_sdesc(sb + kk * b_adv, b_lbo, 1024u);
        umma_bf16(d_tmem, ad, bd, p.idesc, (ks > kb || kk > 0) ? 1u : 0u);
      }
      umma_commit(&empty[stage]);  // frees the stage once these MMAs have read it
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
    if (!ok) break;
    umma_commit(&tfull[acc]);      // accumulator ready for the epilogue
  }
  if (!ok) {
    umma_commit(drain);
    mbar_wait_drain(drain, 0);
  }
}

// ------------------------------------------------------------------ epilogues

// Gather z/tau at the row's cached entries that fall in the 32 columns from
// cb (the sorted walk: pos / nxt are the row's next entry and its column) and
// return the mask of those columns.  Warp-uniform loop, one entry per lane
// per iteration, the register picked by a 32-way select.
__device__ __forceinline__ uint32_t gather_chunk(const GemmParams& p, const uint32_t (&r)[32],
                                                 int cb, int64_t grow, const int* srow, int& pos,
                                                 int& nxt) {
  uint32_t hit = 0u;
  const int ce = cb + 32;
  while (__any_sync(0xffffffffu, nxt < ce)) {
    if (nxt < ce) {
      const int j = nxt - cb;
      uint32_t bits = 0;
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) bits = (jj == j) ? r[jj] : bits;
      p.zg[grow * p.K + pos] = __uint_as_float(bits) * p.inv_tau;
      if (p.gidx) p.gidx[grow * p.K + p.sslot[grow * p.K + pos]] = nxt;
      hit |= 1u << j;
      ++pos;
      nxt = pos < p.K ? __ldg(srow + pos) : INT_MAX;
    }
  }
  return hit;
}

// Forward: per (row, vocab tile) natural-log lse partial of z/tau and the
// gather of z/tau at the row's cached indices that fall inside the tile.
// EXCL (residual-mass variant): the partial leaves out the cached columns, so
// that the mass outside the cache is a sum of its own terms, never 1 minus
// the cached mass (the chunk's reference zc still includes them; a chunk with
// only cached columns adds 0 to the sum).
// STOREZ (single sweep): the launch covers rows rowmap[rowmap_base + local row]
// of one chunk, valid rows first; the partial goes to part[tile][local row].
// Warps holding valid rows also store, for the contractions that follow, each
// valid row's logits as bf16 values exp((z - o) / tau) relative to the row's
// offset o (roff[local row], a logit of the row, so that the largest value is
// at least about 1); other rows of those warps store 0.  Formed as y times
// 2^(c zc - c o) from the chunk-relative y of the lse sum, so one exponential
// per element serves both.  G of the row is then rscale times these values
// once the cached columns are corrected: the dh contraction applies the scale
// to its output columns and the dW contraction takes it inside h_c^T.  A row
// whose largest logit lies more than YREL_MAX_LOG2 / c above o flags the chunk
// (ovf), whose G is then recomputed from the lse.  The values of two 32-column
// chunks (32 rows x 64 columns, 128 bytes a row) are staged in the 128-byte
// swizzle and the TMA stores the piece into the chunk's G buffer.  The lse
// arithmetic is the plain forward's, so lse, row_kl and the loss equal it bit
// for bit.
template <bool EXCL, bool STOREZ>
__device__ __forceinline__ void epi_fwd(const GemmParams& p, const Sched& sc_, const TileCoord& c,
                                        int acc,
                                        uint32_t tmem_row, int r_in_tile, uint64_t* tfull,
                                        uint64_t* tempty, uint32_t use, volatile int* abort_flag,
                                        bool& ok, const CUtensorMap* tmC, float* stage_buf,
                                        uint32_t& piece) {
  const int lane = threadIdx.x & 31;
  const int lrow = c.m * BM + r_in_tile;
  const bool row_ok = lrow < sc_.M;
  int64_t grow = static_cast<int64_t>(p.row0) + lrow;
  bool zstore = false;
  bool yrow = false;  // STOREZ: a valid row, whose values are stored
  float uo = 0.f;     // STOREZ: c o, the row's offset in log2 units
  if (STOREZ) {
    grow = row_ok ? p.rowmap[p.rowmap_base + lrow] : 0;
    const int nvc = min(max(*p.nvalid - p.rowmap_base, 0), sc_.M);
    zstore = lrow - lane < nvc;  // warp-uniform: the warp's first row is valid
    yrow = lrow < nvc;
    if (yrow) uo = __fmul_rn(p.roff[lrow], p.c_log2);
  }
  const int v0 = c.n * ZBN;
  const int* srow = p.sidx + grow * p.K;
  int pos = p.K;
  int nxt = INT_MAX;
  if (row_ok) {  // start of this row's entries inside the tile (overlaps the MMA)
    pos = lower_bound_row(srow, p.K, v0);
    nxt = pos < p.K ? __ldg(srow + pos) : INT_MAX;
  }
  bool w = mbar_wait(&tfull[acc], use & 1u, abort_flag, p.status);
  ok = __all_sync(0xffffffffu, w);
  if (!ok) return;
  tc_fence_after();
  float m = -CUDART_INF_F;
  float s = 0.f;
#pragma unroll 1
  for (int cc = 0; cc < ZBN / 32; ++cc) {
    const int cb = v0 + cc * 32;
    if (cb >= p.N) break;  // uniform: depends on the tile only
    uint32_t r[32];
    tmem_ld32(tmem_row + static_cast<uint32_t>(acc * 256 + cc * 32), r);
    tmem_ld_wait(r);
    // EXCL: the gather first, so that the sum below can leave out the columns it hit
    const uint32_t hit = EXCL ? gather_chunk(p, r, cb, grow, srow, pos, nxt) : 0u;
    // The chunk's largest raw logit zc inside the vocabulary (c > 0, so c zc is
    // the largest scaled one), then y_j = 2^(c z_j - c zc) in (0, 1]: one FFMA
    // and one ex2 per element give the lse term and, in the single sweep, the
    // stored value.  The rounding is pinned (explicit _rn operations),
    // so that the sweep's lse equals the plain forward's bit for bit.
    const bool full = cb + 32 <= p.N;  // uniform: all 32 columns inside the vocabulary
    float zc = -CUDART_INF_F;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      zc = (full || cb + j < p.N) ? fmaxf(zc, __uint_as_float(r[j])) : zc;
    const float uzc = __fmul_rn(zc, p.c_log2);
    float f = 0.f;  // STOREZ: 2^(c zc - c o), from y to the stored value (0: a row not stored)
    if (STOREZ && yrow) {
      const float e = uzc - uo;
      if (e > YREL_MAX_LOG2) *p.ovf = 1;  // the chunk's G is recomputed instead
      f = ex2f(e);
    }
    float cs = 0.f;
    uint32_t hy[16];  // STOREZ: the 32 stored values as 16 pairs of bf16
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float y0 =
          (full || cb + 2 * j < p.N) ? ex2f(fmaf(__uint_as_float(r[2 * j]), p.c_log2, -uzc)) : 0.f;
      const float y1 = (full || cb + 2 * j + 1 < p.N)
                           ? ex2f(fmaf(__uint_as_float(r[2 * j + 1]), p.c_log2, -uzc))
                           : 0.f;
      if (EXCL)  // the columns outside the row's cache only
        cs = __fadd_rn(__fadd_rn(cs, ((hit >> (2 * j)) & 1u) ? 0.f : y0),
                       ((hit >> (2 * j + 1)) & 1u) ? 0.f : y1);
      else
        cs = __fadd_rn(__fadd_rn(cs, y0), y1);
      if (STOREZ) {
        const __nv_bfloat162 hb = __floats2bfloat162_rn(__fmul_rn(y0, f), __fmul_rn(y1, f));
        hy[j] = *reinterpret_cast<const uint32_t*>(&hb);
      }
    }
    const float mn = fmaxf(m, uzc);
    s = __fadd_rn(__fmul_rn(s, ex2f(m - mn)), __fmul_rn(cs, ex2f(uzc - mn)));
    m = mn;
    if (STOREZ && zstore) {  // warp-uniform
      const int hf = cc & 1;
      uint4* b4 = reinterpret_cast<uint4*>(stage_buf + (piece & 1u) * DW_PIECE_FLOATS);
      if (hf == 0) {  // a new 64-column piece: wait until its buffer is free
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)  // row `lane`, 16-byte chunk hf*4 + q, 128-byte swizzle
        b4[lane * 8 + ((hf * 4 + q) ^ (lane & 7))] =
            make_uint4(hy[4 * q + 0], hy[4 * q + 1], hy[4 * q + 2], hy[4 * q + 3]);
      if (hf == 1 || cb + 32 >= p.N) {  // piece complete (or the vocabulary ends)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(tmC, b4, cb - hf * 32, lrow - lane);
          bulk_commit_group();
        }
        ++piece;
      }
    }
    if (!EXCL) gather_chunk(p, r, cb, grow, srow, pos, nxt);
  }
  tc_fence_before();
  mbar_arrive(&tempty[acc]);
  if (row_ok)
    p.part[static_cast<int64_t>(c.n) * p.part_ld + (STOREZ ? lrow : grow)] = (m + lg2f(s)) * LN2;
}

// Backward: G = s_t (exp(z/tau - lse) - scatter p) / tau as bf16 into the chunk buffer.
__device__ __forceinline__ void epi_dz(const GemmParams& p, const Sched& sc_, const TileCoord& c,
                                       int acc,
                                       uint32_t tmem_row, int r_in_tile, uint64_t* tfull,
                                       uint64_t* tempty, uint32_t use, volatile int* abort_flag,
                                       bool& ok, const CUtensorMap* tmC, float* stage_buf,
                                       uint32_t& piece) {
  const int lrow = c.m * BM + r_in_tile;
  const bool active = lrow < sc_.M;    // a real row of this chunk (others store zeros)
  int64_t grow = 0;
  if (active) grow = p.rowmap ? p.rowmap[p.rowmap_base + lrow] : static_cast<int64_t>(p.row0) + lrow;
  const int v0 = c.n * ZBN;
  const int* srow = p.sidx + grow * p.K;
  float sc = 0.f;   // g * valid / N_valid / tau
  float lb = 0.f;   // lse in base 2
  float rq = 0.f;   // residual variant: R / Q (0 for the main loss)
  int pos = p.K;
  int nxt = INT_MAX;
  if (active) {
    const int nv = *p.nvalid;
    if (p.valid[grow] && nv > 0) {
      sc = p.grad_loss / static_cast<float>(nv) * p.inv_tau;
      lb = p.lse[grow] * LOG2E;
      if (p.resid) {
        const float R = p.resid[grow];
        if (R > 0.f) rq = R / p.outside_mass[grow];
      }
      pos = lower_bound_row(srow, p.K, v0);
      nxt = pos < p.K ? __ldg(srow + pos) : INT_MAX;
    }
  }
  // every column gets a q (1 - R/Q); each cached slot adds (R/Q) q - P.  The
  // residual variant forms a cached column's value directly as s (q - P) at its
  // first slot: with Q small (the student's mass on the cache near 1) R/Q is
  // large, and s (1 - R/Q) q + s (R/Q) q would cancel away the digits of s q.
  const float a_row = sc * (1.f - rq);
  bool w = mbar_wait(&tfull[acc], use & 1u, abort_flag, p.status);
  ok = __all_sync(0xffffffffu, w);
  if (!ok) return;
  tc_fence_after();
  // G leaves through the TMA: each warp stages its 32 rows x 64 columns (two
  // 32-column chunks, 128 bytes of bf16 per row) in the 128-byte swizzle
  // (chunk j of row r at j ^ (r % 8)) and one lane stores the piece; the TMA
  // clips rows past the chunk buffer and columns past V.
  const int lane = threadIdx.x & 31;
  const int wrow = lrow - lane;  // first row of this warp
  uint4* b4 = nullptr;
#pragma unroll 1
  for (int cc = 0; cc < ZBN / 32; ++cc) {
    const int cb = v0 + cc * 32;
    if (cb >= p.N) break;
    uint32_t r[32];
    tmem_ld32(tmem_row + static_cast<uint32_t>(acc * 256 + cc * 32), r);
    tmem_ld_wait(r);
    float g[32];
    if (sc != 0.f) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        g[j] = __fmul_rn(a_row, ex2f(fmaf(__uint_as_float(r[j]), p.c_log2, -lb)));
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) g[j] = 0.f;
    }
    const int ce = cb + 32;
    while (__any_sync(0xffffffffu, nxt < ce)) {
      if (nxt < ce) {
        const int j = nxt - cb;
        const float add = -__fmul_rn(sc, __ldg(p.sp + grow * p.K + pos));
        if (rq != 0.f) {
          uint32_t bits = 0;
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) bits = (jj == j) ? r[jj] : bits;
          const float sq = __fmul_rn(sc, ex2f(fmaf(__uint_as_float(bits), p.c_log2, -lb)));
          const bool first = pos == 0 || __ldg(srow + pos - 1) != nxt;
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            g[jj] = (jj == j) ? (first ? __fadd_rn(sq, add) : g[jj] + (rq * sq + add)) : g[jj];
        } else {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) g[jj] = (jj == j) ? __fadd_rn(g[jj], add) : g[jj];
        }
        ++pos;
        nxt = pos < p.K ? __ldg(srow + pos) : INT_MAX;
      }
    }
    const int half = cc & 1;
    if (half == 0) {  // a new 64-column piece: wait until its buffer is free
      b4 = reinterpret_cast<uint4*>(stage_buf + (piece & 1u) * DW_PIECE_FLOATS);
      if (lane == 0) bulk_wait_group_read<1>();
      __syncwarp();
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 pk;
      __nv_bfloat162 b0 = __floats2bfloat162_rn(g[8 * q + 0], g[8 * q + 1]);
      __nv_bfloat162 b1 = __floats2bfloat162_rn(g[8 * q + 2], g[8 * q + 3]);
      __nv_bfloat162 b2 = __floats2bfloat162_rn(g[8 * q + 4], g[8 * q + 5]);
      __nv_bfloat162 b3 = __floats2bfloat162_rn(g[8 * q + 6], g[8 * q + 7]);
      pk.x = *reinterpret_cast<uint32_t*>(&b0);
      pk.y = *reinterpret_cast<uint32_t*>(&b1);
      pk.z = *reinterpret_cast<uint32_t*>(&b2);
      pk.w = *reinterpret_cast<uint32_t*>(&b3);
      b4[lane * 8 + ((half * 4 + q) ^ (lane & 7))] = pk;
    }
    if (half == 1 || cb + 32 >= p.N) {  // piece complete (or the vocabulary ends)
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tmC, b4, cb - half * 32, wrow);
        bulk_commit_group();
      }
      ++piece;
    }
  }
  tc_fence_before();
  mbar_arrive(&tempty[acc]);
}

// fp32 tile store, optionally accumulating into the existing output.
__device__ __forceinline__ void epi_store(const GemmParams& p, const Sched& sc_, const TileCoord& c,
                                          int acc,
                                          uint32_t tmem_row, int r_in_tile, uint64_t* tfull,
                                          uint64_t* tempty, uint32_t use,
                                          volatile int* abort_flag, bool& ok) {
  const int row = c.m * BM + r_in_tile;
  const bool row_ok = row < sc_.M;
  const int n0 = c.n * p.BN;
  int64_t orow_idx = row;
  if (row_ok && p.rowmap && c.s == 0) orow_idx = p.rowmap[p.rowmap_base + row];
  float* orow = (c.s == 0 ? p.out : p.out2 + static_cast<int64_t>(c.s - 1) * p.split_stride) +
                orow_idx * p.ld_out;
  const bool accum = p.accumulate && c.s == 0;
  const int kb = c.s * sc_.ks_per_split;
  const bool kempty = kb >= min(sc_.k_steps, kb + sc_.ks_per_split);
  bool w = mbar_wait(&tfull[acc], use & 1u, abort_flag, p.status);
  ok = __all_sync(0xffffffffu, w);
  if (!ok) return;
  tc_fence_after();
#pragma unroll 1
  for (int cc = 0; cc < p.BN / 32; ++cc) {
    const int cb = n0 + cc * 32;
    if (cb >= p.N) break;
    uint32_t r[32];
    if (kempty) {            // nothing accumulated: the tile is zero
      if (accum) break;
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = 0u;
    } else {
      tmem_ld32(tmem_row + static_cast<uint32_t>(acc * 256 + cc * 32), r);
      tmem_ld_wait(r);
    }
    if (row_ok) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int col = cb + 4 * q;
        if (col < p.N) {
          float4 v = make_float4(__uint_as_float(r[4 * q + 0]), __uint_as_float(r[4 * q + 1]),
                                 __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
          float4* dst = reinterpret_cast<float4*>(orow + col);
          if (accum) {
            const float4 o = *dst;
            v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
          }
          *dst = v;
        }
      }
    }
  }
  tc_fence_before();
  mbar_arrive(&tempty[acc]);
}

// Transposed fp32 tile store for the gradient contractions.  The tile's rows
// are hidden units (TMEM lane = one output column index m in [0, d)), its
// columns are output rows n: element (m, n) goes to out[orow(n) * ld_out + m],
// so for a fixed column the 32 lanes of a warp write 32 consecutive floats.
//   EPI_DH: n is a compacted row of the chunk; split 0 writes dh at the
//           original row rowmap[rowmap_base + n], split s >= 1 writes its
//           partial block out2 + (s-1) * (n_tiles*BN) * ld_out at row n.
//   EPI_DW: n is a vocabulary row; accumulate adds into the existing dW.
// cscale != null: column n of the tile is multiplied by cscale[n] first.
__device__ __forceinline__ void epi_store_t(const GemmParams& p, const Sched& sc_,
                                            const TileCoord& c, int acc, uint32_t tmem_row,
                                            int r_in_tile, uint64_t* tfull, uint64_t* tempty,
                                            uint32_t use, volatile int* abort_flag, bool& ok) {
  const int m = c.m * BM + r_in_tile;
  const bool m_ok = m < sc_.M;
  const int n0 = c.n * p.BN;
  const bool mapped = p.rowmap && c.s == 0;
  float* base = c.s == 0 ? p.out
                         : p.out2 + static_cast<int64_t>(c.s - 1) * sc_.n_tiles * p.BN * p.ld_out;
  const bool accum = p.accumulate && c.s == 0;
  const int kb = c.s * sc_.ks_per_split;
  const bool kempty = kb >= min(sc_.k_steps, kb + sc_.ks_per_split);
  const int lane = threadIdx.x & 31;
  bool w = mbar_wait(&tfull[acc], use & 1u, abort_flag, p.status);
  ok = __all_sync(0xffffffffu, w);
  if (!ok) return;
  tc_fence_after();
#pragma unroll 1
  for (int cc = 0; cc < p.BN / 32; ++cc) {
    const int cb = n0 + cc * 32;
    if (cb >= sc_.N) break;  // uniform: depends on the tile only
    uint32_t r[32];
    if (kempty) {            // nothing accumulated: the tile is zero
      if (accum) break;
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = 0u;
    } else {
      tmem_ld32(tmem_row + static_cast<uint32_t>(acc * 256 + cc * 32), r);
      tmem_ld_wait(r);
    }
    // output row of column cb + lane, shared across the warp by shuffles
    // (every lane takes part; m_ok is warp-uniform because d % 64 == 0)
    int my_row = cb + lane;
    if (mapped && cb + lane < sc_.N) my_row = p.rowmap[p.rowmap_base + cb + lane];
    int orow[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) orow[j] = __shfl_sync(0xffffffffu, my_row, j);
    if (p.cscale) {  // uniform: the column's factor (a chunk row's G scale)
      const float my_sc = cb + lane < sc_.N ? p.cscale[cb + lane] : 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        r[j] = __float_as_uint(__uint_as_float(r[j]) * __shfl_sync(0xffffffffu, my_sc, j));
    }
    const int ncols = min(32, sc_.N - cb);
    if (m_ok) {
      float o[32];
#pragma unroll
      for (int j = 0; j < 32; ++j)
        o[j] = (accum && j < ncols) ? base[static_cast<int64_t>(orow[j]) * p.ld_out + m] : 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < ncols) base[static_cast<int64_t>(orow[j]) * p.ld_out + m] = __uint_as_float(r[j]) + o[j];
    }
  }
  tc_fence_before();
  mbar_arrive(&tempty[acc]);
}

// dW epilogue (EPI_DW): dW tile = G_c^T h_c, rows = vocabulary rows (TMEM
// lanes), columns = hidden units.  Each epilogue warp owns 32 vocabulary rows
// and moves its part of the tile 32 hidden units at a time through its own two
// 4 KB staging buffers, laid out as the TMA's 128-byte swizzle expects (the
// 16-byte chunk j of row r sits at chunk j ^ (r % 8), so the row-per-lane
// stores do not collide in shared-memory banks); one lane then hands the piece
// to the TMA: a tensor store for the first chunk, a tensor reduce-add (the L2
// adds it to dW) for later chunks.  A tile width that is an odd multiple of 16
// ends with a 16-column piece, staged unswizzled for its own tensor map (tmD).
// Each output element has exactly one owner per launch, so the sum is
// deterministic.  No barrier spans warps, so a warp that leaves early on an
// abort cannot leave another waiting.  oscale != null: the tile is multiplied
// by *oscale first.
__device__ __forceinline__ void epi_dw(const GemmParams& p, const Sched& sc_, const TileCoord& c,
                                       int acc, uint32_t tmem_row, int q, uint64_t* tfull,
                                       uint64_t* tempty, uint32_t use, volatile int* abort_flag,
                                       bool& ok, const CUtensorMap* tmC, const CUtensorMap* tmD,
                                       float* stage_buf, uint32_t& piece) {
  const int lane = threadIdx.x & 31;
  const int vw = c.m * BM + q * 32;       // first vocabulary row of this warp
  const bool warp_ok = vw < sc_.M;        // rows past V are clipped by the TMA
  const int n0 = c.n * p.BN;
  const bool accum = p.accumulate != 0;
  const bool kempty = sc_.k_steps == 0;   // no valid row in this chunk
  const float osc = p.oscale ? *p.oscale : 1.f;
  bool w = mbar_wait(&tfull[acc], use & 1u, abort_flag, p.status);
  ok = __all_sync(0xffffffffu, w);
  if (!ok) return;
  tc_fence_after();
  const int pieces = (p.BN + 31) / 32;
#pragma unroll 1
  for (int cc = 0; cc < pieces; ++cc) {
    const int cb = n0 + cc * 32;
    if (!warp_ok || (kempty && accum)) break;  // warp-uniform
    const bool half = p.BN - cc * 32 == 16;    // the tile's last 16 columns
    uint32_t r[32];
    if (kempty) {
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = 0u;
    } else {
      tmem_ld32(tmem_row + static_cast<uint32_t>(acc * 256 + cc * 32), r);
      tmem_ld_wait(r);
      if (p.oscale) {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * osc);
      }
    }
    float* buf = stage_buf + (piece & 1u) * DW_PIECE_FLOATS;
    if (lane == 0) bulk_wait_group_read<1>();  // the copy from this buffer two pieces ago is done
    __syncwarp();
    float4* b4 = reinterpret_cast<float4*>(buf);
    if (!half) {
#pragma unroll
      for (int j = 0; j < 8; ++j)  // row `lane`, 16-byte chunk j, 128-byte swizzle
        b4[lane * 8 + (j ^ (lane & 7))] =
            make_float4(__uint_as_float(r[4 * j + 0]), __uint_as_float(r[4 * j + 1]),
                        __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)  // rows of 64 bytes, no swizzle
        b4[lane * 4 + j] =
            make_float4(__uint_as_float(r[4 * j + 0]), __uint_as_float(r[4 * j + 1]),
                        __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      const CUtensorMap* map = half ? tmD : tmC;
      if (accum)
        tma_reduce_add_2d(map, buf, cb, vw);
      else
        tma_store_2d(map, buf, cb, vw);
      bulk_commit_group();
    }
    ++piece;
  }
  tc_fence_before();
  mbar_arrive(&tempty[acc]);
}

// Teacher top-K producer (EPI_TMAX): per (row, vocabulary tile) the key of
// the tile's largest logit (the lowest index among equal maxima) and the
// natural-log lse partial of z / tau (for the teacher's full-vocabulary
// normaliser); the tile's fp32 logits go out through the TMA (32 x 32 pieces
// staged in the 128-byte swizzle, columns past the vocabulary clipped) for the
// candidate scan that follows.
__device__ __forceinline__ void epi_tmax(const GemmParams& p, const Sched& sc_, const TileCoord& c,
                                         int acc, uint32_t tmem_row, int r_in_tile,
                                         uint64_t* tfull, uint64_t* tempty, uint32_t use,
                                         volatile int* abort_flag, bool& ok,
                                         const CUtensorMap* tmC, float* stage_buf,
                                         uint32_t& piece) {
  const int lane = threadIdx.x & 31;
  const int lrow = c.m * BM + r_in_tile;
  const bool row_ok = lrow < sc_.M;
  const int wrow = lrow - lane;           // first row of this warp
  const bool warp_ok = wrow < sc_.M;      // rows past the chunk are clipped by the TMA
  const int v0 = c.n * ZBN;
  bool w = mbar_wait(&tfull[acc], use & 1u, abort_flag, p.status);
  ok = __all_sync(0xffffffffu, w);
  if (!ok) return;
  tc_fence_after();
  float m = -CUDART_INF_F;
  float s = 0.f;
  float best = -CUDART_INF_F;
  int bidx = v0;
#pragma unroll 1
  for (int cc = 0; cc < ZBN / 32; ++cc) {
    const int cb = v0 + cc * 32;
    if (cb >= p.N) break;
    uint32_t r[32];
    tmem_ld32(tmem_row + static_cast<uint32_t>(acc * 256 + cc * 32), r);
    tmem_ld_wait(r);
    if (warp_ok) {  // warp-uniform
      float* buf = stage_buf + (piece & 1u) * DW_PIECE_FLOATS;
      if (lane == 0) bulk_wait_group_read<1>();  // the copy from this buffer two pieces ago is done
      __syncwarp();
      float4* b4 = reinterpret_cast<float4*>(buf);
#pragma unroll
      for (int j = 0; j < 8; ++j)  // row `lane`, 16-byte chunk j, 128-byte swizzle
        b4[lane * 8 + (j ^ (lane & 7))] =
            make_float4(__uint_as_float(r[4 * j + 0]), __uint_as_float(r[4 * j + 1]),
                        __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tmC, buf, cb, wrow);
        bulk_commit_group();
      }
      ++piece;
    }
    float u[32];
    float cm = -CUDART_INF_F;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float x = __uint_as_float(r[j]);
      const bool in = cb + j < p.N;
      if (in && x > best) {  // ascending j: the first of equal maxima stays
        best = x;
        bidx = cb + j;
      }
      u[j] = in ? x * p.c_log2 : -CUDART_INF_F;
      cm = fmaxf(cm, u[j]);
    }
    const float mn = fmaxf(m, cm);
    float cs = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) cs += ex2f(u[j] - mn);
    s = s * ex2f(m - mn) + cs;
    m = mn;
  }
  tc_fence_before();
  mbar_arrive(&tempty[acc]);
  if (row_ok) {
    p.part[static_cast<int64_t>(c.n) * p.part_ld + lrow] = (m + lg2f(s)) * LN2;
    p.tkeys[static_cast<int64_t>(lrow) * sc_.n_tiles + c.n] = logit_key(best, bidx);
  }
}

// ------------------------------------------------------------------ kernel

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    kd_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmD, const GemmParams p) {
  if (p.gate != nullptr && *p.gate == 0) return;  // uniform: nothing to do in this launch
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  // [pipeline stages][epilogue staging (EPI_DW, EPI_DZ, EPI_TMAX, EPI_FWDZ*)][barriers, TMEM slot,
  // abort flag]
  float* epi_stage = reinterpret_cast<float*>(smem + static_cast<size_t>(p.stages) * p.stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(p.stages) * p.stage_bytes +
                                               p.epi_smem);
  uint64_t* empty = full + MAX_STAGES;
  uint64_t* tfull = empty + MAX_STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const Sched sc = make_sched(p);
  if (warp == 0) {
    if (lane == 0) producer_role(p, sc, &tmA, &tmB, smem, full, empty, abort_flag);
  } else if (warp == 1) {
    if (lane == 0) mma_role(p, sc, smem, full, empty, tfull, tempty, drain, tmem_base, abort_flag);
  } else {
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r_in_tile = q * 32 + lane;
    const uint32_t tmem_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    bool ok = true;
    int lt = 0;
    uint32_t piece = 0;
    float* my_stage = epi_stage + q * 2 * DW_PIECE_FLOATS;
    if (MODE == EPI_DW && lane == 0) {
      tma_prefetch_desc(&tmC);
      tma_prefetch_desc(&tmD);
    }
    for (int t = blockIdx.x; t < sc.num_tiles; t += gridDim.x, ++lt) {
      const TileCoord c = decode_tile(p, sc, t);
      const int acc = lt & 1;
      const uint32_t use = static_cast<uint32_t>(lt >> 1);
      if (MODE == EPI_DW)
        epi_dw(p, sc, c, acc, tmem_row, q, tfull, tempty, use, abort_flag, ok, &tmC, &tmD,
               my_stage, piece);
      else if (MODE == EPI_FWD || MODE == EPI_FWD_RESID || MODE == EPI_FWDZ ||
               MODE == EPI_FWDZ_RESID)
        epi_fwd<MODE == EPI_FWD_RESID || MODE == EPI_FWDZ_RESID,
                MODE == EPI_FWDZ || MODE == EPI_FWDZ_RESID>(p, sc, c, acc, tmem_row, r_in_tile,
                                                            tfull, tempty, use, abort_flag, ok,
                                                            &tmC, my_stage, piece);
      else if (MODE == EPI_DZ)
        epi_dz(p, sc, c, acc, tmem_row, r_in_tile, tfull, tempty, use, abort_flag, ok, &tmC,
               my_stage, piece);
      else if (MODE == EPI_STORE)
        epi_store(p, sc, c, acc, tmem_row, r_in_tile, tfull, tempty, use, abort_flag, ok);
      else if (MODE == EPI_TMAX)
        epi_tmax(p, sc, c, acc, tmem_row, r_in_tile, tfull, tempty, use, abort_flag, ok, &tmC,
                 my_stage, piece);
      else
        epi_store_t(p, sc, c, acc, tmem_row, r_in_tile, tfull, tempty, use, abort_flag, ok);
      if (!ok) break;
    }
    // the TMA copies this warp issued finish before the CTA leaves
    if ((MODE == EPI_DW || MODE == EPI_DZ || MODE == EPI_TMAX || MODE == EPI_FWDZ ||
         MODE == EPI_FWDZ_RESID) && lane == 0)
      bulk_wait_group_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ SIMT kernels

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Teacher side of each row, one warp per row: range check of the cached
// indices, the teacher probabilities of the K entries, the teacher term
// sum_k p log p, and the entries sorted by vocabulary index (ties keep slot
// order) so that the contraction epilogues can walk them tile by tile.
// teacher_lse == null: p = softmax(teacher_logits / tau) over the K entries
// (renormalised).  Otherwise p = exp(teacher_logits / tau - teacher_lse) under
// the teacher's full-vocabulary normaliser and resid = max(0, 1 - sum_k p),
// the mass outside the cache (formed without cancellation).
__global__ void kd_prep_kernel(const int* __restrict__ idx, const float* __restrict__ tl,
                               const float* __restrict__ teacher_lse,
                               const uint8_t* __restrict__ valid, int T, int K, int V,
                               float inv_tau, int* __restrict__ sidx, float* __restrict__ sp,
                               int16_t* __restrict__ sslot, float* __restrict__ tterm,
                               float* __restrict__ resid, int* __restrict__ nvalid, int* status) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= T) return;
  const int* ir = idx + static_cast<int64_t>(row) * K;
  const float* tr = tl + static_cast<int64_t>(row) * K;
  float m = -CUDART_INF_F;
  int bad = 0;
  for (int k = lane; k < K; k += 32) {
    m = fmaxf(m, tr[k] * inv_tau);
    const int v = ir[k];
    bad |= (v < 0 || v >= V);
  }
  m = warp_max(m);
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, KD_ERR_INDEX_RANGE);
  float L = 0.f;     // full-vocabulary normaliser (teacher_lse given)
  float S = 0.f;
  for (int k = lane; k < K; k += 32) S += expf(tr[k] * inv_tau - m);
  S = warp_sum(S);
  const float logS = logf(S);  // log sum_k exp(a_k - m): the cached entries' normaliser
  if (teacher_lse) L = teacher_lse[row];
  float tt = 0.f;
  int* so = sidx + static_cast<int64_t>(row) * K;
  float* po = sp + static_cast<int64_t>(row) * K;
  int16_t* lo = sslot + static_cast<int64_t>(row) * K;
  for (int k = lane; k < K; k += 32) {
    const float lp = teacher_lse ? tr[k] * inv_tau - L : tr[k] * inv_tau - m - logS;
    const float pk = expf(lp);
    if (pk > 0.f) tt += pk * lp;
    const int v = ir[k];
    int rank = 0;
    for (int j = 0; j < K; ++j) {
      const int u = ir[j];
      rank += (u < v) || (u == v && j < k);
    }
    so[rank] = v;
    po[rank] = pk;
    lo[rank] = static_cast<int16_t>(k);
  }
  tt = warp_sum(tt);
  if (lane == 0) {
    tterm[row] = tt;
    // 1 - sum_k p = 1 - exp(lseK - L) with lseK = m + log S, formed by expm1 so
    // that a teacher with nearly all its mass in the cache keeps R's digits
    if (resid) resid[row] = teacher_lse ? fmaxf(0.f, -expm1f(m + logS - L)) : 0.f;
    if (valid[row]) atomicAdd(nvalid, 1);
  }
}

// lse from the per-tile partials, row_kl, and a per-block (double) partial sum
// of row_kl for the deterministic loss reduction.  Block (32, COMBINE_SPLIT):
// thread (x, y) takes row 32 b + x and every COMBINE_SPLIT-th tile (and
// cached entry) from y, so a warp reads 32 consecutive rows of one tile's
// partials (coalesced); the COMBINE_SPLIT partial results of a row are merged
// in the fixed order y = 0, 1, ...
// resid != null (residual variant): the partials cover only the columns
// outside the row's cache (lse_out = Lu over those); the cached columns, each
// distinct index once (sidx is ascending), complete the normaliser, lse =
// log(exp(Lu) + sum exp(zg)).  The student mass outside the cache is then
// Q = exp(Lu - lse), less the mass of repeated slots (each slot is its own
// outcome), with no 1 - sum cancellation; it goes to outside_mass_out (if
// given) and row_kl gains R (log R - log Q) for R > 0.
// rowmap != null (single sweep): the launch covers the T rows
// rowmap[rowmap_base + i] of one chunk, whose partials sit at part[tile][i]
// (part_ld = the chunk's row capacity); losspart may then be null.
constexpr int COMBINE_SPLIT = 8;

__device__ __forceinline__ void online_lse_add(float v, float& m, float& s) {
  if (v == -CUDART_INF_F) return;  // exp(-inf) adds nothing
  if (v > m) {
    s = s * expf(m - v) + 1.f;
    m = v;
  } else {
    s += expf(v - m);
  }
}

// Fixed-order merge of the COMBINE_SPLIT (max, sum) pairs of column x.
__device__ __forceinline__ float merge_lse(const float (&sm)[COMBINE_SPLIT][32],
                                           const float (&ss)[COMBINE_SPLIT][32], int x) {
  float M = sm[0][x], S = ss[0][x];
  for (int i = 1; i < COMBINE_SPLIT; ++i) {
    const float mi = sm[i][x], si = ss[i][x];
    const float mn = fmaxf(M, mi);
    if (mn != -CUDART_INF_F) S = S * expf(M - mn) + si * expf(mi - mn);
    M = mn;
  }
  return M + logf(S);
}

// The single sweep's scales of the chunk's stored values, formed with the lse
// (rscale == null everywhere else).  For local row i below the chunk's valid
// count: escale[i] = exp(o_i / tau - lse) g_i and rscale[i] = s escale[i], with
// s = grad_loss / N_valid / tau and g_i = 1 - R/Q for the residual-mass variant
// (1 for the main loss), so that G = rscale times the stored values away from
// the cached columns; *oscale = s.  Rows past the valid count get 0.  A row
// with |g| below YREL_MIN_FACTOR (R close to Q) flags the chunk (ovf), whose
// G is then recomputed whole; the cached-column pass then sets the scales to
// 1.  valid_only: the logit GEMM covered the chunk's valid rows only, so the
// other rows get lse = NaN (and Q = NaN) and row_kl = 0 without reading
// partials.
struct SweepScales {
  const float* roff;
  int* ovf;
  const int* nvalid;
  float grad_loss, inv_tau;
  float* rscale;
  float* escale;
  float* oscale;
  int valid_only;
};

__global__ void __launch_bounds__(32 * COMBINE_SPLIT)
    kd_combine_kernel(const float* __restrict__ part, int64_t part_ld, int n_tiles, int T, int K,
                      const int* __restrict__ rowmap, int rowmap_base,
                      const int* __restrict__ sidx, const float* __restrict__ sp,
                      const float* __restrict__ zg, const float* __restrict__ tterm,
                      const float* __restrict__ resid, const uint8_t* __restrict__ valid,
                      float* __restrict__ lse_out, float* __restrict__ row_kl_out,
                      float* __restrict__ outside_mass_out, double* __restrict__ losspart,
                      const SweepScales sw) {
  __shared__ float sm[COMBINE_SPLIT][32], ss[COMBINE_SPLIT][32];
  __shared__ float s_lse[32], s_lu[32];
  __shared__ float sa[COMBINE_SPLIT][32], smass[COMBINE_SPLIT][32];
  __shared__ double red[32];
  const int x = threadIdx.x, y = threadIdx.y;
  const int li = blockIdx.x * 32 + x;  // row of this launch
  const bool in = li < T;
  const int row = (in && rowmap) ? rowmap[rowmap_base + li] : li;
  const int64_t rk0 = static_cast<int64_t>(row) * K;
  // a row whose logits were formed (all rows unless valid_only)
  const bool live = in && !(sw.valid_only && li >= *sw.nvalid - rowmap_base);
  // online logsumexp over this thread's tiles
  float m = -CUDART_INF_F;
  float s = 0.f;
  if (live)
    for (int j = y; j < n_tiles; j += COMBINE_SPLIT)
      online_lse_add(part[static_cast<int64_t>(j) * part_ld + li], m, s);
  sm[y][x] = m;
  ss[y][x] = s;
  __syncthreads();
  if (y == 0) {
    const float L = merge_lse(sm, ss, x);
    s_lse[x] = L;
    if (in && lse_out && !resid) lse_out[row] = live ? L : CUDART_NAN_F;
  }
  __syncthreads();
  if (resid) {  // uniform: the cached columns complete the normaliser
    m = -CUDART_INF_F;
    s = 0.f;
    if (live)
      for (int k = y; k < K; k += COMBINE_SPLIT)
        if (k == 0 || sidx[rk0 + k] != sidx[rk0 + k - 1]) online_lse_add(zg[rk0 + k], m, s);
    sm[y][x] = m;
    ss[y][x] = s;
    __syncthreads();
    if (y == 0) {
      const float Lu = s_lse[x];
      const float Lc = merge_lse(sm, ss, x);
      const float L = fmaxf(Lu, Lc) + log1pf(expf(-fabsf(Lu - Lc)));  // Lc is finite
      s_lu[x] = Lu;
      s_lse[x] = L;
      if (in && lse_out) lse_out[row] = live ? L : CUDART_NAN_F;
    }
    __syncthreads();
  }
  const float lse = s_lse[x];
  // this thread's share of sum_k p_k (lse - zg_k) and of the repeated slots' mass
  float acc = 0.f, mass = 0.f;
  if (live) {
    for (int k = y; k < K; k += COMBINE_SPLIT) {
      const float zk = zg[rk0 + k];
      acc += sp[rk0 + k] * (lse - zk);
      if (resid && k > 0 && sidx[rk0 + k] == sidx[rk0 + k - 1]) mass += expf(zk - lse);
    }
  }
  sa[y][x] = acc;
  smass[y][x] = mass;
  __syncthreads();
  if (y == 0) {
    double kl = 0.0;
    if (in) {
      float a = 0.f, dup = 0.f;
      for (int i = 0; i < COMBINE_SPLIT; ++i) {
        a += sa[i][x];
        dup += smass[i][x];
      }
      float Q = 0.f, logQ = 0.f;
      if (resid) {
        const float lu = s_lu[x] - lse;
        Q = expf(lu) - dup;
        logQ = dup == 0.f ? lu : logf(Q);
        if (outside_mass_out) outside_mass_out[row] = live ? Q : CUDART_NAN_F;
      }
      float rk = 0.f;
      if (live && valid[row]) {
        rk = tterm[row] + a;
        if (resid) {
          const float R = resid[row];
          if (R > 0.f) rk += R * (logf(R) - logQ);
        }
      }
      if (row_kl_out) row_kl_out[row] = rk;
      kl = rk;
      if (sw.rscale) {  // uniform: the single sweep's scales of this row's stored values
        const int nv = *sw.nvalid;
        float e = 0.f, c = 0.f;
        if (li < nv - rowmap_base) {  // a valid row of the chunk
          float g = 1.f;
          if (resid) {
            const float R = resid[row];
            if (R > 0.f) g = 1.f - R / Q;
          }
          if (!(fabsf(g) >= YREL_MIN_FACTOR)) *sw.ovf = 1;  // (also a NaN factor)
          const float sg = sw.grad_loss / static_cast<float>(nv) * sw.inv_tau;
          e = expf(sw.roff[li] * sw.inv_tau - lse) * g;
          c = sg * e;
        }
        sw.escale[li] = e;
        sw.rscale[li] = c;
      }
    }
    red[x] = kl;
    if (sw.rscale && blockIdx.x == 0 && x == 0) {
      const int nv = *sw.nvalid;
      *sw.oscale = nv > 0 ? sw.grad_loss / static_cast<float>(nv) * sw.inv_tau : 0.f;
    }
  }
  __syncthreads();
  if (y == 0 && x == 0 && losspart) {
    double t = 0.0;
    for (int i = 0; i < 32; ++i) t += red[i];
    losspart[blockIdx.x] = t;
  }
}

// Per block of 32 consecutive rows, the double sum of row_kl in row order:
// the partials the combine forms when it runs over all rows in order (the
// single sweep's combine runs chunk by chunk in another row order), so that
// kd_loss_final_kernel gives the same loss bit for bit.
__global__ void kd_loss_blocks_kernel(const float* __restrict__ row_kl, int T,
                                      double* __restrict__ losspart) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b * 32 >= T) return;
  double t = 0.0;
  for (int i = 0; i < 32; ++i) {
    const int r = b * 32 + i;
    t += r < T ? static_cast<double>(row_kl[r]) : 0.0;
  }
  losspart[b] = t;
}

// Single block: fixed-order sum of the per-block partials, divided by N_valid.
__global__ void kd_loss_final_kernel(const double* __restrict__ losspart, int nb,
                                     const int* __restrict__ nvalid, float* __restrict__ loss) {
  __shared__ double red[256];
  double s = 0.0;
  for (int i = threadIdx.x; i < nb; i += blockDim.x) s += losspart[i];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int o = blockDim.x >> 1; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int n = *nvalid;
    *loss = n > 0 ? static_cast<float>(red[0] / n) : 0.f;
  }
}

// Valid rows in ascending order: rowmap[i] = the i-th row with valid != 0.
// nvalid != null (the valid-row count): the invalid rows follow, also in
// ascending order, rowmap[*nvalid + j] = the j-th row with valid == 0.
// One block; fixed order, so the compaction is deterministic.
__global__ void kd_compact_rows_kernel(const uint8_t* __restrict__ valid, int T,
                                       const int* __restrict__ nvalid, int* __restrict__ rowmap) {
  __shared__ int warp_incl[32];
  __shared__ int base;
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  if (threadIdx.x == 0) base = 0;
  __syncthreads();
  for (int t0 = 0; t0 < T; t0 += blockDim.x) {
    const int t = t0 + threadIdx.x;
    const int f = (t < T && valid[t]) ? 1 : 0;
    int x = f;  // inclusive scan inside the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_incl[w] = x;
    __syncthreads();
    if (w == 0) {
      int v = lane < nw ? warp_incl[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      if (lane < nw) warp_incl[lane] = v;
    }
    __syncthreads();
    const int excl = base + (w > 0 ? warp_incl[w - 1] : 0) + x - f;  // valid rows before t
    if (f)
      rowmap[excl] = t;
    else if (nvalid && t < T)
      rowmap[*nvalid + (t - excl)] = t;
    __syncthreads();
    if (threadIdx.x == 0) base += warp_incl[nw - 1];
    __syncthreads();
  }
}

// Chunk of compacted rows: hc[i] = h[rowmap[c0 + i]] for i < rows and 0 for
// rows <= i < cap, with rows = clamp(*nvalid - c0, 0, cap), or rows = cap when
// nvalid is null.  d8 = d / 8.
__global__ void kd_gather_rows_kernel(const uint4* __restrict__ h, const int* __restrict__ rowmap,
                                      const int* __restrict__ nvalid, int c0, int cap, int d8,
                                      uint4* __restrict__ hc) {
  const int rows = nvalid ? max(0, min(*nvalid - c0, cap)) : cap;
  const int64_t n = static_cast<int64_t>(cap) * d8;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / d8);
    const int j = static_cast<int>(i - static_cast<int64_t>(r) * d8);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows) v = h[static_cast<int64_t>(rowmap[c0 + r]) * d8 + j];
    hc[i] = v;
  }
}

// The chunk's valid rows of h, transposed: hcT[j * ld + i] = h[rowmap[c0 + i]][j]
// for i < rows and 0 for rows <= i < cap, rows = clamp(*nvalid - c0, 0, cap).
// escale != null (single sweep): row i is multiplied by escale[i] and rounded
// to bf16.  32 x 32 tiles through shared memory; block (32, 8).
__global__ void kd_gather_rows_t_kernel(const __nv_bfloat16* __restrict__ h,
                                        const int* __restrict__ rowmap,
                                        const int* __restrict__ nvalid, int c0, int cap, int ld,
                                        int d, const float* __restrict__ escale,
                                        __nv_bfloat16* __restrict__ hcT) {
  __shared__ __nv_bfloat16 tile[32][33];
  const int rows = max(0, min(*nvalid - c0, cap));
  const int j0 = blockIdx.x * 32;
  const int i0 = blockIdx.y * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = i0 + ty + 8 * r;
    const int j = j0 + tx;
    __nv_bfloat16 v = __float2bfloat16_rn(0.f);
    if (i < rows && j < d) {
      v = h[static_cast<int64_t>(rowmap[c0 + i]) * d + j];
      if (escale) v = __float2bfloat16_rn(__bfloat162float(v) * escale[i]);
    }
    tile[ty + 8 * r][tx] = v;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int j = j0 + ty + 8 * r;
    const int i = i0 + tx;
    if (j < d && i < cap) hcT[static_cast<int64_t>(j) * ld + i] = tile[tx][ty + 8 * r];
  }
}

// Single sweep, before the chunk's logit GEMM: one warp per local row i < cap
// copies hc[i] = h[rowmap[c0 + i]] and, for the chunk's valid rows (i below
// clamp(*nvalid - c0, 0, cap)), forms the row's offset roff[i] = h_t . W[v],
// the student's logit at the teacher's highest cached entry v (the first
// slot among equal teacher logits).  It is a logit of the row, so the
// largest stored value exp((z - o) / tau) is at least about 1 and none of the
// row's significant values underflows.  d8 = d / 8 (uint4 = 8 bf16).
__global__ void kd_gather_rows_offset_kernel(const uint4* __restrict__ h,
                                             const uint4* __restrict__ W,
                                             const int* __restrict__ rowmap,
                                             const int* __restrict__ nvalid,
                                             const int* __restrict__ tidx,
                                             const float* __restrict__ tlog, int K, int V, int c0,
                                             int cap, int d8, uint4* __restrict__ hc,
                                             float* __restrict__ roff) {
  const int lane = threadIdx.x & 31;
  const int i = static_cast<int>((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  if (i >= cap) return;  // whole warp
  const int rows = max(0, min(*nvalid - c0, cap));
  const int64_t t = rowmap[c0 + i];
  const uint4* hr = h + t * d8;
  uint4* out = hc + static_cast<int64_t>(i) * d8;
  if (i >= rows) {
    for (int j = lane; j < d8; j += 32) out[j] = hr[j];
    return;
  }
  float best = -CUDART_INF_F;
  int bk = K;
  for (int k = lane; k < K; k += 32) {
    const float x = tlog[t * K + k];
    if (x > best) {  // ascending k: the first of equal logits stays
      best = x;
      bk = k;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int ok = __shfl_xor_sync(0xffffffffu, bk, o);
    if (ob > best || (ob == best && ok < bk)) {
      best = ob;
      bk = ok;
    }
  }
  const int v = min(max(tidx[t * K + (bk < K ? bk : 0)], 0), V - 1);  // in range even for bad input
  const uint4* wr = W + static_cast<int64_t>(v) * d8;
  float acc = 0.f;
  for (int j = lane; j < d8; j += 32) {
    const uint4 a = hr[j];
    out[j] = a;
    const uint4 b = __ldg(wr + j);
    const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aa[q]));
      const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bb[q]));
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) roff[i] = acc;
}

// Single sweep, after the combine and the gated recompute: completes the
// chunk's stored values so that G = rscale times them.  At each distinct cached
// column v of a valid local row i (original row t) the value becomes
//   (exp((z_v - o)/tau) a_v - P exp(lse - o/tau)) / g,
// P the teacher probability summed over the c_v slots naming v, from the fp32
// z_v / tau of the gather (one rounding to bf16, as for G itself).  Main loss:
// a_v = g = 1.  Residual-mass variant (resid != null): rq = R/Q (0 when
// R = 0), g = 1 - rq, a_v = 1 + (c_v - 1) rq, so that rscale times the value
// is s (q_v a_v - P) with no cancellation between the two parts of a_v.  Rows
// from the valid count up to the next multiple of 64 (within c_cap) are set to
// 0: the dW contraction reads whole 64-row steps of the buffer against zero
// rows of h_c^T, and what an earlier chunk left there must not add NaN.  A
// chunk flagged (ovf) by the logit GEMM or the combine has had its G
// recomputed whole: then this kernel only writes the zero rows and sets the
// valid rows' scales (and the dW factor) to 1.  One warp per row, the lanes
// over the row's sorted slots (a repeated index is handled by the first slot
// of its run, so no two lanes write one column).
constexpr int FIX_WARPS = 8;

__global__ void __launch_bounds__(32 * FIX_WARPS)
    kd_fix_cached_kernel(__nv_bfloat16* __restrict__ gbuf, int V, int c0, int c_cap,
                         const int* __restrict__ rowmap, const int* __restrict__ nvalid,
                         const int* __restrict__ sidx, const float* __restrict__ sp,
                         const float* __restrict__ zg, int K, const float* __restrict__ lse,
                         const float* __restrict__ roff, float inv_tau,
                         const float* __restrict__ resid, const float* __restrict__ outside_mass,
                         const int* __restrict__ ovf, float* __restrict__ rscale,
                         float* __restrict__ escale, float* __restrict__ oscale) {
  const int rows = max(0, min(*nvalid - c0, c_cap));
  const int tail_end = min(c_cap, (rows + 63) & ~63);
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t n16 = static_cast<int64_t>(tail_end - rows) * (V / 8);  // V % 8 == 0
  uint4* tail = reinterpret_cast<uint4*>(gbuf + static_cast<int64_t>(rows) * V);
  for (int64_t e = tid; e < n16; e += nthreads) tail[e] = make_uint4(0u, 0u, 0u, 0u);
  if (*ovf) {  // G was recomputed: it needs no scale
    for (int64_t i = tid; i < rows; i += nthreads) {
      rscale[i] = 1.f;
      escale[i] = 1.f;
    }
    if (tid == 0) *oscale = 1.f;
    return;
  }
  const int lane = threadIdx.x & 31;
  for (int64_t i = tid >> 5; i < rows; i += nthreads >> 5) {
    const int64_t t = rowmap[c0 + i];
    const float oi = roff[i] * inv_tau;
    const float e2 = expf(lse[t] - oi);
    float rq = 0.f;
    if (resid) {
      const float R = resid[t];
      if (R > 0.f) rq = R / outside_mass[t];
    }
    const float g = 1.f - rq;
    const int* srow = sidx + t * K;
    const float* prow = sp + t * K;
    const float* zrow = zg + t * K;
    __nv_bfloat16* grow = gbuf + i * V;
    for (int k = lane; k < K; k += 32) {
      const int v = srow[k];
      if ((k > 0 && srow[k - 1] == v) || v < 0 || v >= V) continue;
      float P = prow[k];
      int cnt = 1;
      for (int q = k + 1; q < K && srow[q] == v; ++q, ++cnt) P += prow[q];
      const float a = cnt == 1 ? 1.f : 1.f + static_cast<float>(cnt - 1) * rq;
      grow[v] = __float2bfloat16_rn((expf(zrow[k] - oi) * a - P * e2) / g);
    }
  }
}

// Split-K completion for dh rows of a chunk: dh[rowmap[c0 + r]] += sum_s part[s][r]
// in a fixed order, for the chunk's rows r < clamp(*nvalid - c0, 0, cap).  The
// contraction published its split count S and partial block height (rows) in
// split_info; partial s (s < S - 1) starts at part + s * height * 4 * d4.
// d4 = d / 4.
__global__ void kd_split_reduce_rows_kernel(float* __restrict__ dh, const float* __restrict__ part,
                                            const int* __restrict__ split_info,
                                            const int* __restrict__ rowmap,
                                            const int* __restrict__ nvalid, int c0, int cap,
                                            int d4) {
  const int rows = max(0, min(*nvalid - c0, cap));
  const int nparts = split_info[0] - 1;
  if (nparts <= 0) return;
  const int64_t stride4 = static_cast<int64_t>(split_info[1]) * d4;
  const int64_t n = static_cast<int64_t>(rows) * d4;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / d4);
    const int j = static_cast<int>(i - static_cast<int64_t>(r) * d4);
    float4* dst = reinterpret_cast<float4*>(dh) + static_cast<int64_t>(rowmap[c0 + r]) * d4 + j;
    float4 a = *dst;
    for (int s = 0; s < nparts; ++s) {
      const float4 b = reinterpret_cast<const float4*>(part)[s * stride4 + i];
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    *dst = a;
  }
}

// One thread waits, through the pipeline's bounded wait, on an mbarrier that
// nothing arrives on; the wait must give up after limit_ns and report
// KD_ERR_TIMEOUT in *status.
__global__ void kd_wait_selftest_kernel(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile int* af = &abort_flag;
    mbar_wait(&bar, 0, af, status, limit_ns);
  }
}

}  // namespace kd
