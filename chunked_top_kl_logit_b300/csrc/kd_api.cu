// C ABI of the fused top-K KL loss: argument checks, workspace layout,
// TMA tensor maps and the launch sequence.  The library owns no memory; every
// buffer (inputs, outputs, workspace, status word) belongs to the caller.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/kd_topk_kl.h"
#include "kd_filter.cuh"
#include "kd_kernels.cuh"
#include "kd_pair.cuh"
#include "kd_topk_producer.cuh"

using namespace kd;

namespace {

// Split-K and tile-order choices are made for this many SMs (B300) rather
// than the SM count of whatever device is current, so that results do not
// depend on the device's SM count.  Grid sizes do use the live SM count.
constexpr int kPolicySMs = 148;
constexpr int kRasterGroupRows = 32;  // 128-row tiles per raster group (4096 rows of h in L2)
constexpr uint32_t kMaxDynSmem = 232448;  // opt-in dynamic shared memory per block (sm_100 family)

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// bf16 matrix with `inner` contiguous elements per line, `outer` lines,
// line pitch `ld` elements; box = 64 inner x box_outer lines, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
              uint32_t box_outer) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {64, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 matrix of `outer` rows with `inner` contiguous elements (pitch `ld`),
// box = box_inner x box_outer, no swizzle: the dW output of the TMA
// store / reduce-add epilogue.
bool make_map_f32(CUtensorMap* m, void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                  uint32_t box_inner, uint32_t box_outer, bool swizzle128 = false) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 4};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sms(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KD_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return KD_ERR_CUDA;
  if (major != 10 || minor != 3) return KD_ERR_UNSUPPORTED;
  return KD_OK;
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t al256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Largest split count the dh contraction may use (the device picks the actual
// count from the chunk's row count; each split keeps at least 32 k-steps).
constexpr int kMaxDhSplits = 4;
constexpr int kGradBN = 256;  // gradient contractions: 128 hidden units x 256 rows per tile

// Tile width of the dW contraction over the hidden units: the widest multiple
// of 16 up to 256 that divides d (d = 2880 -> 240), so no column is padding.
int dw_tile_width(int64_t d) {
  for (int bn = 256; bn >= 16; bn -= 16)
    if (d % bn == 0) return bn;
  return 64;
}

int dh_max_splits(int64_t V) {
  const int64_t ks = cdiv(V, BK);
  int s = 1;
  while (s < kMaxDhSplits && ks / (s + 1) >= 32) ++s;
  return s;
}

struct Layout {
  size_t nvalid, losspart, sidx, sp, sslot, tterm, resid;  // shared by both passes
  size_t zg, part;                                  // forward
  size_t rowmap, split_info, hc, hct, dz, dhpart;   // backward
  size_t szg, spart, srowkl, sroff, srs, ses, sscal;  // single sweep (sweep layouts only)
  size_t fwd_total, bwd_total;
  int64_t rows_chunk;
  int dh_splits;      // largest split count of the dh contraction
  int64_t part_rows;  // rows of dh partials the split blocks may use
  int64_t hct_ld;     // row pitch (elements) of the transposed h chunk
};

// sweep: the single-sweep training step's layout: the backward's buffers (dz
// holds the chunk's G, and first the forward's values relative to the row
// offsets), then the forward's tables, the chunk's row offsets and scales, and
// per chunk an overflow flag plus the dW factor; bwd_total is its size.
Layout make_layout(int64_t T, int64_t V, int64_t d, int64_t K, int64_t chunk,
                   bool sweep = false) {
  Layout L{};
  size_t off = 0;
  L.nvalid = off;   off += 256;
  L.losspart = off; off += al256(static_cast<size_t>(cdiv(T, 32)) * 8);
  L.sidx = off;     off += al256(static_cast<size_t>(T * K) * 4);
  L.sp = off;       off += al256(static_cast<size_t>(T * K) * 4);
  L.sslot = off;    off += al256(static_cast<size_t>(T * K) * 2);
  L.tterm = off;    off += al256(static_cast<size_t>(T) * 4);
  L.resid = off;    off += al256(static_cast<size_t>(T) * 4);
  const size_t common = off;
  L.zg = off;       off += al256(static_cast<size_t>(T * K) * 4);
  L.part = off;     off += al256(static_cast<size_t>(cdiv(V, ZBN) * T) * 4);
  L.fwd_total = off;
  L.rows_chunk = chunk < T ? chunk : T;
  L.dh_splits = dh_max_splits(V);
  L.part_rows = L.dh_splits > 1 ? (L.dh_splits - 1) * cdiv(L.rows_chunk, kGradBN) * kGradBN : 0;
  off = common;
  L.rowmap = off;     off += al256(static_cast<size_t>(T) * 4);
  L.split_info = off; off += 256;
  L.hc = off;         off += al256(static_cast<size_t>(L.rows_chunk * d) * 2);
  L.hct_ld = cdiv(L.rows_chunk, 8) * 8;  // 16-byte row pitch for the TMA
  L.hct = off;        off += al256(static_cast<size_t>(L.hct_ld * d) * 2);
  L.dz = off;         off += al256(static_cast<size_t>(L.rows_chunk * V) * 2);
  L.dhpart = off;     off += al256(static_cast<size_t>(L.part_rows * d) * 4);
  if (sweep) {
    L.szg = off;      off += al256(static_cast<size_t>(T * K) * 4);
    L.spart = off;    off += al256(static_cast<size_t>(cdiv(V, ZBN) * L.rows_chunk) * 4);
    L.srowkl = off;   off += al256(static_cast<size_t>(T) * 4);
    L.sroff = off;    off += al256(static_cast<size_t>(L.rows_chunk) * 4);
    L.srs = off;      off += al256(static_cast<size_t>(L.rows_chunk) * 4);
    L.ses = off;      off += al256(static_cast<size_t>(L.rows_chunk) * 4);
    L.sscal = off;    off += al256(static_cast<size_t>(cdiv(T, L.rows_chunk) + 1) * 4);
  }
  L.bwd_total = off;
  return L;
}

int check_shape(int64_t T, int64_t V, int64_t d, int32_t K, int64_t chunk) {
  if (T < 1 || V < 1 || d < 1 || K < 1 || chunk < 1) return KD_ERR_INVALID_ARG;
  if (T > INT32_MAX || V > INT32_MAX || d > INT32_MAX || chunk > INT32_MAX)
    return KD_ERR_UNSUPPORTED;
  if (V % 8 != 0 || d % 64 != 0 || K > V || K > 32767) return KD_ERR_UNSUPPORTED;
  if (static_cast<double>(T) * K > 2e9) return KD_ERR_UNSUPPORTED;
  return KD_OK;
}

int check_inputs(const void* h, const void* W, const int32_t* idx, const float* tl,
                 const uint8_t* valid, int64_t T, int64_t V, int64_t d, int32_t K, float tau,
                 int64_t chunk, const void* ws, const int32_t* dev_status) {
  if (!h || !W || !idx || !tl || !valid || !ws || !dev_status) return KD_ERR_INVALID_ARG;
  if (!(tau > 0.f) || !std::isfinite(tau)) return KD_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(W) || !aligned16(ws)) return KD_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(idx) & 3u) || (reinterpret_cast<uintptr_t>(tl) & 3u) ||
      (reinterpret_cast<uintptr_t>(dev_status) & 3u))
    return KD_ERR_INVALID_ARG;
  return check_shape(T, V, d, K, chunk);
}

GemmParams base_params(int a_mn, int b_mn, int BN) {
  GemmParams p{};
  p.a_mn = a_mn;
  p.b_mn = b_mn;
  p.BN = BN;
  p.a_bytes = BM * BK * 2;
  p.b_bytes = static_cast<uint32_t>(BN) * BK * 2;
  p.stage_bytes = p.a_bytes + p.b_bytes;
  p.stages = static_cast<int>((200u * 1024u) / p.stage_bytes);
  if (p.stages > MAX_STAGES) p.stages = MAX_STAGES;
  p.idesc = make_idesc_bf16(BM, BN, a_mn, b_mn);
  p.splits = 1;
  return p;
}

static_assert(static_cast<int>(KD_KERNEL_LOGITS_FWD) == EPI_FWD &&
                  static_cast<int>(KD_KERNEL_LOGITS_BWD) == EPI_DZ &&
                  static_cast<int>(KD_KERNEL_DH) == EPI_DH &&
                  static_cast<int>(KD_KERNEL_DW) == EPI_DW &&
                  static_cast<int>(KD_KERNEL_TOPK_PASS1) == EPI_TMAX,
              "kernel ids of the timing interface follow the epilogue modes");

// Diagnostic launch timing (kd_timing_*): while recording, each contraction
// launch is bracketed by two CUDA events on its stream.
struct TimingRec {
  int kind;
  cudaEvent_t start, stop;
};

struct Timing {
  std::mutex mu;
  bool recording = false;
  int capacity = 0;
  int used = 0;
  std::vector<TimingRec> recs;
};

Timing& timing() {
  static Timing t;
  return t;
}

void destroy_timing_events(Timing& t) {
  for (auto& r : t.recs) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  t.recs.clear();
  t.used = 0;
  t.capacity = 0;
}

// Slot for the next timed launch, or -1 when not recording / out of slots.
int timing_slot(int kind) {
  Timing& t = timing();
  std::lock_guard<std::mutex> lock(t.mu);
  if (!t.recording || t.used >= t.capacity) return -1;
  t.recs[t.used].kind = kind;
  return t.used++;
}

// Opt a kernel into the full dynamic shared-memory limit once per device (a
// function attribute, not a stream operation: keeping it out of the launch
// path lets the calls be captured in a CUDA graph).
template <typename Kernel>
bool ensure_smem_attr(Kernel kernel, std::once_flag* flags, bool* ok) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::call_once(flags[dev], [&] {
    ok[dev] = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(kMaxDynSmem)) == cudaSuccess;
  });
  return ok[dev];
}

// `c` / `dm` are the output tensor maps of EPI_DW (32- and 16-column pieces;
// ignored by the other modes).
template <int MODE>
int launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                const CUtensorMap& dm, GemmParams p, int sms, cudaStream_t st) {
  if (p.num_tiles <= 0) return KD_OK;
  p.epi_smem = (MODE == EPI_DW || MODE == EPI_DZ || MODE == EPI_TMAX || MODE == EPI_FWDZ ||
                MODE == EPI_FWDZ_RESID)
                   ? 4u * 2u * DW_PIECE_FLOATS * 4u
                   : 0u;
  // the stage ring shares the opt-in shared-memory limit with the staging
  const int fit = static_cast<int>((kMaxDynSmem - 1024u - 256u - p.epi_smem) / p.stage_bytes);
  if (p.stages > fit) p.stages = fit;
  const size_t smem = 1024 + static_cast<size_t>(p.stages) * p.stage_bytes + p.epi_smem + 256;
  static std::once_flag attr_once[64];
  static bool attr_ok[64];
  if (!ensure_smem_attr(kd_gemm_kernel<MODE>, attr_once, attr_ok)) return KD_ERR_CUDA;
  const int grid = p.num_tiles < sms ? p.num_tiles : sms;
  // the residual variant's and the single sweep's forwards are timed as the
  // forward logit kernel
  const int slot = MODE == EPI_STORE ? -1
                   : timing_slot((MODE == EPI_FWD_RESID || MODE == EPI_FWDZ ||
                                  MODE == EPI_FWDZ_RESID)
                                     ? EPI_FWD
                                     : MODE);
  if (slot >= 0 && cudaEventRecord(timing().recs[static_cast<size_t>(slot)].start, st) != cudaSuccess)
    return KD_ERR_CUDA;
  kd_gemm_kernel<MODE><<<grid, NUM_THREADS, smem, st>>>(a, b, c, dm, p);
  if (cudaGetLastError() != cudaSuccess) return KD_ERR_CUDA;
  if (slot >= 0 && cudaEventRecord(timing().recs[static_cast<size_t>(slot)].stop, st) != cudaSuccess)
    return KD_ERR_CUDA;
  return KD_OK;
}

// Launch the CTA-pair kernel (clusters of two CTAs) on a pair schedule.
int launch_pair(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, int sms,
                cudaStream_t st) {
  if (p.num_tiles <= 0) return KD_OK;
  const size_t smem = 1024 + static_cast<size_t>(p.stages) * p.stage_bytes + 256;
  static std::once_flag attr_once[64];
  static bool attr_ok[64];
  if (!ensure_smem_attr(kd_gemm_pair_kernel, attr_once, attr_ok)) return KD_ERR_CUDA;
  const int clusters = p.num_tiles < sms / 2 ? p.num_tiles : sms / 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kd_gemm_pair_kernel, a, b, p) != cudaSuccess) return KD_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

// Turn a one-CTA schedule with K-major operands and 128 x BN tiles into the
// CTA-pair schedule: 256 x BN tiles per pair, each CTA loading its 128 rows of
// A and BN/2 rows of B (so B's tensor map box is BN/2 rows), M = 256 MMAs.
void pair_schedule(GemmParams& p, int group_pairs) {
  p.a_bytes = BM * BK * 2;
  p.b_bytes = static_cast<uint32_t>(p.BN / 2) * BK * 2;
  p.stage_bytes = p.a_bytes + p.b_bytes;
  p.stages = static_cast<int>((200u * 1024u) / p.stage_bytes);
  if (p.stages > MAX_STAGES) p.stages = MAX_STAGES;
  p.idesc = make_idesc_bf16(2 * BM, p.BN, 0, 0);
  p.m_tiles = static_cast<int>(cdiv(p.M, 2 * BM));
  p.num_tiles = p.m_tiles * p.n_tiles * p.splits;
  p.group_m = p.m_tiles < group_pairs ? p.m_tiles : group_pairs;
}

struct Ws {
  int* nvalid;
  double* losspart;
  int* sidx;
  float* sp;
  int16_t* sslot;
  float* tterm;
  float* resid;
};

Ws carve(void* ws, const Layout& L) {
  char* w = static_cast<char*>(ws);
  return Ws{reinterpret_cast<int*>(w + L.nvalid), reinterpret_cast<double*>(w + L.losspart),
            reinterpret_cast<int*>(w + L.sidx),   reinterpret_cast<float*>(w + L.sp),
            reinterpret_cast<int16_t*>(w + L.sslot), reinterpret_cast<float*>(w + L.tterm),
            reinterpret_cast<float*>(w + L.resid)};
}

// Normalisation of the teacher's cached entries.  Main loss: all pointers null
// (softmax renormalised over the K entries).  Residual variant: teacher_lse is
// the teacher's full-vocabulary log-normaliser at tau; the forward writes the
// student's mass outside the cached entries to outside_mass_out and the
// backward reads it back from outside_mass_in.
struct Variant {
  const float* teacher_lse = nullptr;
  float* outside_mass_out = nullptr;
  const float* outside_mass_in = nullptr;
  bool residual() const { return teacher_lse != nullptr; }
};

int run_prep(const int32_t* idx, const float* tl, const uint8_t* valid, int64_t T, int32_t K,
             int64_t V, float inv_tau, const Ws& w, const Variant& var, int32_t* dev_status,
             cudaStream_t st) {
  if (cudaMemsetAsync(dev_status, 0, sizeof(int32_t), st) != cudaSuccess) return KD_ERR_CUDA;
  if (cudaMemsetAsync(w.nvalid, 0, sizeof(int), st) != cudaSuccess) return KD_ERR_CUDA;
  const int rows_per_block = 8;
  kd_prep_kernel<<<static_cast<unsigned>(cdiv(T, rows_per_block)), 32 * rows_per_block, 0, st>>>(
      idx, tl, var.teacher_lse, valid, static_cast<int>(T), K, static_cast<int>(V), inv_tau, w.sidx,
      w.sp, w.sslot, w.tterm, var.residual() ? w.resid : nullptr, w.nvalid, dev_status);
  return cudaGetLastError() == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

// Logit-tile schedule shared by the forward, the backward recompute and the
// teacher top-K passes: 128 x 256 tiles, raster groups of 32 row tiles (4096
// rows of h stay L2-resident), vocabulary-major inside a group.  (The CTA-pair
// kernel of kd_gemm_bf16_diag_pair computes the same tiles as 256 x 256 pair
// tiles; under the 1.1 kW power cap it made the whole step 3% slower, so the
// loss keeps one CTA per tile.)
void logit_schedule(GemmParams& p, int64_t rows, int64_t V, int64_t d) {
  p.m_tiles = static_cast<int>(cdiv(rows, BM));
  p.n_tiles = static_cast<int>(cdiv(V, ZBN));
  p.num_tiles = p.m_tiles * p.n_tiles;
  p.k_steps = static_cast<int>(d / BK);
  p.ks_per_split = p.k_steps;
  p.group_m = p.m_tiles < kRasterGroupRows ? p.m_tiles : kRasterGroupRows;
  p.n_fast = 0;
  p.M = static_cast<int>(rows);
  p.N = static_cast<int>(V);
}

// Workspace of the teacher top-K producer, for chunks of C rows.
struct TopkLayout {
  size_t part, tkeys, theta, theta_val, cnt, cand, z, total;
  int64_t C;
  int n_tiles, cap;
};

TopkLayout make_topk_layout(int64_t T, int64_t V, int32_t K, int64_t chunk) {
  TopkLayout L{};
  L.C = chunk < T ? chunk : T;
  L.n_tiles = static_cast<int>(cdiv(V, ZBN));
  // candidates per row: at most (K - 1) full tiles plus the threshold key, or
  // the whole row when it has fewer than K tiles
  const int64_t bound = K <= L.n_tiles ? static_cast<int64_t>(K - 1) * ZBN + 1 : V;
  L.cap = static_cast<int>(bound < V ? bound : V);
  size_t off = 0;
  L.part = off;      off += al256(static_cast<size_t>(L.n_tiles) * L.C * 4);
  L.tkeys = off;     off += al256(static_cast<size_t>(L.C) * L.n_tiles * 8);
  L.theta = off;     off += al256(static_cast<size_t>(L.C) * 8);
  L.theta_val = off; off += al256(static_cast<size_t>(L.C) * 4);
  L.cnt = off;       off += al256(static_cast<size_t>(L.C) * 4);
  L.cand = off;      off += al256(static_cast<size_t>(L.C) * L.cap * 8);
  L.z = off;         off += al256(static_cast<size_t>(L.C) * V * 4);  // the chunk's fp32 logits
  L.total = off;
  return L;
}

}  // namespace

// ------------------------------------------------------------------
// Built-in scratch for kd_topk_kl_forward_noalloc.  Callers that cannot
// allocate device memory get this fixed array as the forward's workspace.
// It lives in the library's device image, so every GPU that loads the
// library holds these bytes until the process exits.
static constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Device address of g_noalloc_scratch on the current device.  The symbol's
// name in host code is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress once per device (with that device current) and
// cached.
void* noalloc_scratch_address(int* rc) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *rc = KD_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      *rc = KD_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" {

const char* kd_topk_kl_status_string(int status) {
  switch (status) {
    case KD_OK: return "ok";
    case KD_ERR_INVALID_ARG: return "invalid argument";
    case KD_ERR_UNSUPPORTED: return "unsupported device or shape";
    case KD_ERR_WORKSPACE: return "workspace too small";
    case KD_ERR_CUDA: return "CUDA call failed";
    case KD_ERR_INDEX_RANGE: return "teacher index outside [0, V)";
    case KD_ERR_TIMEOUT: return "bounded pipeline wait timed out";
    case KD_ERR_SCRATCH_LIMIT: return "shape needs more than the built-in 32 MiB scratch array";
    case KD_ERR_INTERNAL: return "internal bound violated (library bug)";
    case KD_ERR_NONFINITE: return "a row of teacher logits is not finite (NaN or +inf)";
    default: return "unknown status";
  }
}

int kd_topk_kl_workspace_size(int64_t T, int64_t V, int64_t d, int32_t K, int64_t chunk,
                              size_t* fwd_bytes, size_t* bwd_bytes) {
  const int rc = check_shape(T, V, d, K, chunk);
  if (rc != KD_OK) return rc;
  const Layout L = make_layout(T, V, d, K, chunk);
  if (fwd_bytes) *fwd_bytes = L.fwd_total;
  if (bwd_bytes) *bwd_bytes = L.bwd_total;
  return KD_OK;
}

int kd_topk_kl_forward_backward_workspace_size(int64_t T, int64_t V, int64_t d, int32_t K,
                                               int64_t chunk, size_t* bytes, int32_t* launches) {
  const int rc = check_shape(T, V, d, K, chunk);
  if (rc != KD_OK) return rc;
  const Layout L = make_layout(T, V, d, K, chunk, true);
  if (bytes) *bytes = L.bwd_total;
  // prep, row order; per chunk: row gather with offsets, logit GEMM, combine,
  // recompute (returns at once unless the chunk is flagged), cached columns,
  // transposed row gather, dh, [dh split reduce], dW; loss partials, loss
  if (launches)
    *launches = static_cast<int32_t>(2 + cdiv(T, L.rows_chunk) * (L.dh_splits > 1 ? 9 : 8) + 2);
  return KD_OK;
}

int kd_topk_kl_launch_count(int64_t T, int64_t V, int64_t d, int32_t K, int64_t chunk,
                            int32_t* fwd_launches, int32_t* bwd_launches) {
  const int rc = check_shape(T, V, d, K, chunk);
  if (rc != KD_OK) return rc;
  const Layout L = make_layout(T, V, d, K, chunk);
  const int64_t chunks = cdiv(T, L.rows_chunk);
  if (fwd_launches) *fwd_launches = 4;  // prep, logit GEMM, combine, loss
  // prep + row compaction, then per chunk: row gather (plain and transposed),
  // recompute, dh, [dh split reduce], dW
  if (bwd_launches)
    *bwd_launches = static_cast<int32_t>(2 + chunks * (L.dh_splits > 1 ? 6 : 5));
  return KD_OK;
}

}  // extern "C"

namespace {

// The forward's launches after the teacher prep: logit GEMM with the lse /
// gather epilogue, combine, loss.  lse may be null (loss-only evaluation).
int enqueue_forward(const void* h, const void* W, const uint8_t* valid, int64_t T, int64_t V,
                    int64_t d, int32_t K, float tau, const Layout& L, void* ws, const Ws& w,
                    const Variant& var, int sms, float* loss, float* lse, float* row_kl,
                    int32_t* gathered_idx, int32_t* dev_status, cudaStream_t st) {
  int rc = KD_OK;
  char* wb = static_cast<char*>(ws);
  float* zg = reinterpret_cast<float*>(wb + L.zg);
  float* part = reinterpret_cast<float*>(wb + L.part);
  const float inv_tau = 1.0f / tau;
  CUtensorMap ta, tb;
  if (!make_map(&ta, h, d, T, d, BM) || !make_map(&tb, W, d, V, d, ZBN)) return KD_ERR_CUDA;
  GemmParams p = base_params(0, 0, ZBN);
  logit_schedule(p, T, V, d);
  p.status = dev_status;
  p.row0 = 0;
  p.K = K;
  p.sidx = w.sidx;
  p.sp = w.sp;
  p.sslot = w.sslot;
  p.inv_tau = inv_tau;
  p.c_log2 = LOG2E * inv_tau;
  p.part_ld = T;
  p.part = part;
  p.zg = zg;
  p.gidx = gathered_idx;
  rc = var.residual() ? launch_gemm<EPI_FWD_RESID>(ta, tb, ta, ta, p, sms, st)
                      : launch_gemm<EPI_FWD>(ta, tb, ta, ta, p, sms, st);
  if (rc) return rc;

  const int nb = static_cast<int>(cdiv(T, 32));
  kd_combine_kernel<<<nb, dim3(32, COMBINE_SPLIT), 0, st>>>(
      part, T, p.n_tiles, static_cast<int>(T), K, nullptr, 0, w.sidx, w.sp, zg, w.tterm,
      var.residual() ? w.resid : nullptr, valid, lse, row_kl, var.outside_mass_out, w.losspart,
      SweepScales{});
  kd_loss_final_kernel<<<1, 256, 0, st>>>(w.losspart, nb, w.nvalid, loss);
  return cudaGetLastError() == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

// The gradient contractions of one chunk of compacted valid rows [c0, c0 + C)
// (their count clamp(*nvalid - c0, 0, C) stays on the device), given the
// chunk's bf16 G (row pitch g_ld elements) and h_c^T: dh rows through the
// row map, split over V on the device when the chunk has few rows, and dW
// (accumulate: added to dW instead of stored).
int enqueue_grad_contractions(const void* W, int64_t V, int64_t d, const Layout& L, const Ws& w,
                              int sms, const int* rowmap, const __nv_bfloat16* G, int64_t g_ld,
                              const __nv_bfloat16* hct, float* dhpart, int* split_info,
                              int64_t c0, float* dh, float* dW, int accumulate,
                              const float* cscale, const float* oscale, int32_t* dev_status,
                              cudaStream_t st) {
  int rc = KD_OK;
  const int S = L.dh_splits;
  const int64_t C = L.rows_chunk;
  CUtensorMap ta, tb;
  // (2) dh rows of the chunk, computed transposed: dh_c^T = W^T G_c^T, so a
  // tile is 128 hidden units x 256 chunk rows (A = W as an MN-major operand,
  // B = G K-major).  The contraction over V is split on the device when the
  // chunk holds too few rows to fill the GPU.
  if (!make_map(&ta, W, d, V, d, 64) || !make_map(&tb, G, V, C, g_ld, kGradBN))
    return KD_ERR_CUDA;
  GemmParams q = base_params(1, 0, kGradBN);
  q.m_tiles = static_cast<int>(cdiv(d, BM));
  q.n_tiles = static_cast<int>(cdiv(C, kGradBN));
  q.splits = S;
  q.num_tiles = q.m_tiles * q.n_tiles * S;  // upper bound; the device decides
  q.k_steps = static_cast<int>(cdiv(V, BK));
  q.ks_per_split = q.k_steps;
  q.n_fast = 0;
  q.group_m = q.m_tiles;                    // hidden-unit tiles fastest: W slabs shared
  q.M = static_cast<int>(d);
  q.N = static_cast<int>(C);
  q.status = dev_status;
  q.out = dh;
  q.out2 = dhpart;
  q.ld_out = d;
  q.dyn_count = w.nvalid;
  q.dyn_base = static_cast<int>(c0);
  q.dyn_cap = static_cast<int>(C);
  q.dyn_kind = 3;
  q.rowmap = rowmap;
  q.rowmap_base = static_cast<int>(c0);
  q.part_rows = static_cast<int>(L.part_rows);
  q.policy_sms = kPolicySMs;
  q.split_info = split_info;
  q.cscale = cscale;
  if ((rc = launch_gemm<EPI_DH>(ta, tb, ta, ta, q, sms, st))) return rc;
  if (S > 1) {
    kd_split_reduce_rows_kernel<<<sms * 4, 256, 0, st>>>(
        dh, dhpart, split_info, rowmap, w.nvalid, static_cast<int>(c0), static_cast<int>(C),
        static_cast<int>(d / 4));
    if (cudaGetLastError() != cudaSuccess) return KD_ERR_CUDA;
  }

  // (3) dW (+)= G_c^T h_c: tiles of 128 vocabulary rows x BNw hidden units
  // (A = G as an MN-major operand, B = h_c^T K-major), the contraction over
  // the chunk's valid rows; 32 x 32 pieces of the tile are stored or
  // reduce-added into dW by the TMA.
  const int BNw = dw_tile_width(d);
  CUtensorMap tc, td;
  if (!make_map(&ta, G, V, C, g_ld, 64) ||
      !make_map(&tb, hct, C, d, L.hct_ld, static_cast<uint32_t>(BNw)) ||
      !make_map_f32(&tc, dW, d, V, d, 32, 32, true) || !make_map_f32(&td, dW, d, V, d, 16, 32))
    return KD_ERR_CUDA;
  GemmParams r = base_params(1, 0, BNw);
  r.m_tiles = static_cast<int>(cdiv(V, BM));
  r.n_tiles = static_cast<int>(d / BNw);
  r.num_tiles = r.m_tiles * r.n_tiles;
  r.k_steps = static_cast<int>(cdiv(C, BK));
  r.ks_per_split = r.k_steps;
  r.n_fast = 1;                             // hidden-unit tiles fastest: G slabs shared
  r.group_m = 1;
  r.M = static_cast<int>(V);
  r.N = static_cast<int>(d);
  r.status = dev_status;
  r.out = dW;
  r.out2 = nullptr;
  r.ld_out = d;
  r.accumulate = accumulate;
  r.dyn_count = w.nvalid;
  r.dyn_base = static_cast<int>(c0);
  r.dyn_cap = static_cast<int>(C);
  r.dyn_kind = 2;
  r.oscale = oscale;
  return launch_gemm<EPI_DW>(ta, tb, tc, td, r, sms, st);
}

// The chunk's valid rows of h as h_c^T (dW's B operand): hcT[j][i] =
// h[rowmap[c0 + i]][j] for the chunk's valid rows i (times escale[i] when
// escale is not null), zero up to the pitch.
int enqueue_gather_t(const void* h, int64_t d, const Layout& L, const Ws& w, const int* rowmap,
                     int64_t c0, const float* escale, __nv_bfloat16* hct, cudaStream_t st) {
  const int64_t C = L.rows_chunk;
  kd_gather_rows_t_kernel<<<dim3(static_cast<unsigned>(cdiv(d, 32)),
                                 static_cast<unsigned>(cdiv(C, 32))),
                            dim3(32, 8), 0, st>>>(static_cast<const __nv_bfloat16*>(h), rowmap,
                                                  w.nvalid, static_cast<int>(c0),
                                                  static_cast<int>(C), static_cast<int>(L.hct_ld),
                                                  static_cast<int>(d), escale, hct);
  return cudaGetLastError() == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

// The backward's launches after the teacher prep: dh zeroing, row
// compaction, then per chunk of valid rows the recompute, dh and dW
// contractions.  accumulate_dW: the first chunk adds to dW instead of
// overwriting it.
int enqueue_backward(const void* h, const void* W, const uint8_t* valid, int64_t T, int64_t V,
                     int64_t d, int32_t K, float tau, const Layout& L, void* ws, const Ws& w,
                     const Variant& var, int sms, const float* lse, float grad_loss, float* dh,
                     float* dW, int accumulate_dW, int32_t* dev_status, cudaStream_t st) {
  int rc = KD_OK;
  char* wb = static_cast<char*>(ws);
  int* rowmap = reinterpret_cast<int*>(wb + L.rowmap);
  __nv_bfloat16* hc = reinterpret_cast<__nv_bfloat16*>(wb + L.hc);
  __nv_bfloat16* hct = reinterpret_cast<__nv_bfloat16*>(wb + L.hct);
  __nv_bfloat16* dz = reinterpret_cast<__nv_bfloat16*>(wb + L.dz);
  float* dhpart = reinterpret_cast<float*>(wb + L.dhpart);
  int* split_info = reinterpret_cast<int*>(wb + L.split_info);
  const float inv_tau = 1.0f / tau;
  const int64_t C = L.rows_chunk;

  // Rows with valid = 0 have an exactly zero gradient: dh starts at zero and
  // the chunks below run over the valid rows only, compacted in ascending
  // order.  Their count stays on the device; every kernel clamps to it.
  if (cudaMemsetAsync(dh, 0, static_cast<size_t>(T * d) * sizeof(float), st) != cudaSuccess)
    return KD_ERR_CUDA;
  kd_compact_rows_kernel<<<1, 1024, 0, st>>>(valid, static_cast<int>(T), nullptr, rowmap);
  if (cudaGetLastError() != cudaSuccess) return KD_ERR_CUDA;

  for (int64_t c0 = 0; c0 < T; c0 += C) {
    CUtensorMap ta, tb;

    // (0) the chunk's valid rows of h, zero-padded to C rows, and transposed
    kd_gather_rows_kernel<<<sms * 4, 256, 0, st>>>(
        static_cast<const uint4*>(h), rowmap, w.nvalid, static_cast<int>(c0), static_cast<int>(C),
        static_cast<int>(d / 8), reinterpret_cast<uint4*>(hc));
    if (cudaGetLastError() != cudaSuccess) return KD_ERR_CUDA;
    if ((rc = enqueue_gather_t(h, d, L, w, rowmap, c0, nullptr, hct, st))) return rc;

    // (1) recompute the chunk's logit tiles and write G as bf16
    if (!make_map(&ta, hc, d, C, d, BM) || !make_map(&tb, W, d, V, d, ZBN)) return KD_ERR_CUDA;
    GemmParams p = base_params(0, 0, ZBN);
    logit_schedule(p, C, V, d);
    p.status = dev_status;
    p.K = K;
    p.sidx = w.sidx;
    p.sp = w.sp;
    p.sslot = w.sslot;
    p.inv_tau = inv_tau;
    p.c_log2 = LOG2E * inv_tau;
    p.lse = lse;
    p.resid = var.residual() ? w.resid : nullptr;
    p.outside_mass = var.outside_mass_in;
    p.valid = valid;
    p.nvalid = w.nvalid;
    p.grad_loss = grad_loss;
    p.dz = dz;
    p.dz_ld = V;
    p.dyn_count = w.nvalid;
    p.dyn_base = static_cast<int>(c0);
    p.dyn_cap = static_cast<int>(C);
    p.dyn_kind = 1;
    p.rowmap = rowmap;
    p.rowmap_base = static_cast<int>(c0);
    CUtensorMap tg;  // G chunk as the TMA store target (64-column x 32-row boxes)
    if (!make_map(&tg, dz, V, C, V, 32)) return KD_ERR_CUDA;
    if ((rc = launch_gemm<EPI_DZ>(ta, tb, tg, ta, p, sms, st))) return rc;

    // (2), (3) dh and dW of the chunk
    if ((rc = enqueue_grad_contractions(W, V, d, L, w, sms, rowmap, dz, V, hct, dhpart, split_info,
                                        c0, dh, dW, (c0 > 0 || accumulate_dW) ? 1 : 0, nullptr,
                                        nullptr, dev_status, st)))
      return rc;
  }
  return KD_OK;
}

// The single-sweep training step after the teacher prep (one logit GEMM per
// row instead of two): rows in the order valid rows, then invalid rows.  Per
// chunk of C rows of that order: the rows of h and each valid row's offset o
// (the student's logit at the teacher's highest cached entry); the forward
// logit GEMM forms the lse partials and the gather and stores the valid rows'
// logits as bf16 exp((z - o) / tau) into the chunk's G buffer; the combine
// gives lse and row_kl and the scales exp(o / tau - lse); a chunk whose stored
// values would have left their range has its G recomputed from the lse (a
// launch that returns at once otherwise); the cached columns are corrected;
// h_c^T is formed with the rows' scales, and the dh (scaled per row in its
// epilogue) and dW contractions follow as in the backward.  The chunks of
// valid rows are the backward's and the lse arithmetic is the forward's, so
// lse, row_kl and the loss equal forward + backward bit for bit (the loss's
// partial sums are formed over the rows in their original order); dh and dW
// agree to within bf16 rounding.
int enqueue_sweep(const void* h, const void* W, const int32_t* teacher_idx,
                  const float* teacher_logits, const uint8_t* valid, int64_t T, int64_t V,
                  int64_t d, int32_t K, float tau, const Layout& L, void* ws, const Ws& w,
                  const Variant& var, int sms, float grad_loss, int accumulate_dW,
                  int valid_only, float* loss, float* lse, float* row_kl, float* dh, float* dW,
                  int32_t* dev_status, cudaStream_t st) {
  int rc = KD_OK;
  char* wb = static_cast<char*>(ws);
  int* rowmap = reinterpret_cast<int*>(wb + L.rowmap);
  int* split_info = reinterpret_cast<int*>(wb + L.split_info);
  __nv_bfloat16* hc = reinterpret_cast<__nv_bfloat16*>(wb + L.hc);
  __nv_bfloat16* hct = reinterpret_cast<__nv_bfloat16*>(wb + L.hct);
  __nv_bfloat16* G = reinterpret_cast<__nv_bfloat16*>(wb + L.dz);
  float* dhpart = reinterpret_cast<float*>(wb + L.dhpart);
  float* zg = reinterpret_cast<float*>(wb + L.szg);
  float* part = reinterpret_cast<float*>(wb + L.spart);
  float* roff = reinterpret_cast<float*>(wb + L.sroff);
  float* rscale = reinterpret_cast<float*>(wb + L.srs);
  float* escale = reinterpret_cast<float*>(wb + L.ses);
  float* oscale = reinterpret_cast<float*>(wb + L.sscal);  // then one flag per chunk
  int* ovf = reinterpret_cast<int*>(oscale + 1);
  float* rkl = row_kl ? row_kl : reinterpret_cast<float*>(wb + L.srowkl);
  const float inv_tau = 1.0f / tau;
  const int64_t C = L.rows_chunk;
  const int64_t nchunks = cdiv(T, C);

  if (cudaMemsetAsync(dh, 0, static_cast<size_t>(T * d) * sizeof(float), st) != cudaSuccess ||
      cudaMemsetAsync(ovf, 0, static_cast<size_t>(nchunks) * sizeof(int), st) != cudaSuccess)
    return KD_ERR_CUDA;
  kd_compact_rows_kernel<<<1, 1024, 0, st>>>(valid, static_cast<int>(T), w.nvalid, rowmap);
  if (cudaGetLastError() != cudaSuccess) return KD_ERR_CUDA;

  for (int64_t c0 = 0; c0 < T; c0 += C) {
    const int64_t M = (T - c0) < C ? (T - c0) : C;
    int* flag = ovf + c0 / C;
    CUtensorMap ta, tb, ty;
    // (0) the chunk's rows of h in that order, and the valid rows' offsets
    kd_gather_rows_offset_kernel<<<static_cast<unsigned>(cdiv(M, 8)), 256, 0, st>>>(
        static_cast<const uint4*>(h), static_cast<const uint4*>(W), rowmap, w.nvalid, teacher_idx,
        teacher_logits, K, static_cast<int>(V), static_cast<int>(c0), static_cast<int>(M),
        static_cast<int>(d / 8), reinterpret_cast<uint4*>(hc), roff);
    if (cudaGetLastError() != cudaSuccess) return KD_ERR_CUDA;

    // (1) logit tiles: lse partials, gather, the valid rows' values relative to
    // their offsets into the G buffer (64-column x 32-row boxes of bf16)
    if (!make_map(&ta, hc, d, M, d, BM) || !make_map(&tb, W, d, V, d, ZBN) ||
        !make_map(&ty, G, V, M, V, 32))
      return KD_ERR_CUDA;
    GemmParams p = base_params(0, 0, ZBN);
    logit_schedule(p, M, V, d);
    p.status = dev_status;
    p.K = K;
    p.sidx = w.sidx;
    p.sp = w.sp;
    p.sslot = w.sslot;
    p.inv_tau = inv_tau;
    p.c_log2 = LOG2E * inv_tau;
    p.part_ld = C;
    p.part = part;
    p.zg = zg;
    p.gidx = nullptr;
    p.nvalid = w.nvalid;
    p.rowmap = rowmap;
    p.rowmap_base = static_cast<int>(c0);
    p.roff = roff;
    p.ovf = flag;
    if (valid_only) {  // only the chunk's valid rows (the first ones of the row order)
      p.dyn_count = w.nvalid;
      p.dyn_base = static_cast<int>(c0);
      p.dyn_cap = static_cast<int>(M);
      p.dyn_kind = 1;
    }
    rc = var.residual() ? launch_gemm<EPI_FWDZ_RESID>(ta, tb, ty, ta, p, sms, st)
                        : launch_gemm<EPI_FWDZ>(ta, tb, ty, ta, p, sms, st);
    if (rc) return rc;

    // (2) lse and row_kl of the chunk's rows (and the mass outside the cache),
    // and the scales of the stored values
    const float* resid = var.residual() ? w.resid : nullptr;
    const SweepScales sc{roff, flag, w.nvalid, grad_loss, inv_tau, rscale, escale, oscale,
                         valid_only};
    kd_combine_kernel<<<static_cast<unsigned>(cdiv(M, 32)), dim3(32, COMBINE_SPLIT), 0, st>>>(
        part, C, p.n_tiles, static_cast<int>(M), K, rowmap, static_cast<int>(c0), w.sidx, w.sp,
        zg, w.tterm, resid, valid, lse, rkl, var.outside_mass_out, nullptr, sc);
    if (cudaGetLastError() != cudaSuccess) return KD_ERR_CUDA;

    // (3) only for a flagged chunk: G of its valid rows recomputed from the lse
    GemmParams q = base_params(0, 0, ZBN);
    logit_schedule(q, M, V, d);
    q.status = dev_status;
    q.K = K;
    q.sidx = w.sidx;
    q.sp = w.sp;
    q.sslot = w.sslot;
    q.inv_tau = inv_tau;
    q.c_log2 = LOG2E * inv_tau;
    q.lse = lse;
    q.resid = resid;
    q.outside_mass = var.outside_mass_out;
    q.valid = valid;
    q.nvalid = w.nvalid;
    q.grad_loss = grad_loss;
    q.dz = G;
    q.dz_ld = V;
    q.dyn_count = w.nvalid;
    q.dyn_base = static_cast<int>(c0);
    q.dyn_cap = static_cast<int>(M);
    q.dyn_kind = 1;
    q.rowmap = rowmap;
    q.rowmap_base = static_cast<int>(c0);
    q.gate = flag;
    if ((rc = launch_gemm<EPI_DZ>(ta, tb, ty, ta, q, sms, st))) return rc;

    // (4) the cached columns (and zero rows after the valid ones, up to the next
    // multiple of 64)
    const int slot = timing_slot(KD_KERNEL_SWEEP_FIX);
    if (slot >= 0 &&
        cudaEventRecord(timing().recs[static_cast<size_t>(slot)].start, st) != cudaSuccess)
      return KD_ERR_CUDA;
    kd_fix_cached_kernel<<<static_cast<unsigned>(cdiv(C, FIX_WARPS)), 32 * FIX_WARPS, 0, st>>>(
        G, static_cast<int>(V), static_cast<int>(c0), static_cast<int>(C), rowmap, w.nvalid, w.sidx,
        w.sp, zg, K, lse, roff, inv_tau, resid, var.outside_mass_out, flag, rscale, escale,
        oscale);
    if (cudaGetLastError() != cudaSuccess) return KD_ERR_CUDA;
    if (slot >= 0 &&
        cudaEventRecord(timing().recs[static_cast<size_t>(slot)].stop, st) != cudaSuccess)
      return KD_ERR_CUDA;

    // (5) h_c^T with the rows' scales, then dh and dW of the chunk
    if ((rc = enqueue_gather_t(h, d, L, w, rowmap, c0, escale, hct, st))) return rc;
    if ((rc = enqueue_grad_contractions(W, V, d, L, w, sms, rowmap, G, V, hct, dhpart, split_info,
                                        c0, dh, dW, (c0 > 0 || accumulate_dW) ? 1 : 0, rscale,
                                        oscale, dev_status, st)))
      return rc;
  }
  const int nb = static_cast<int>(cdiv(T, 32));
  kd_loss_blocks_kernel<<<static_cast<unsigned>(cdiv(nb, 256)), 256, 0, st>>>(
      rkl, static_cast<int>(T), w.losspart);
  kd_loss_final_kernel<<<1, 256, 0, st>>>(w.losspart, nb, w.nvalid, loss);
  return cudaGetLastError() == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

}  // namespace

extern "C" {

int kd_topk_kl_forward(const void* h, const void* W, const int32_t* teacher_idx,
                       const float* teacher_logits, const uint8_t* valid, int64_t T, int64_t V,
                       int64_t d, int32_t K, float tau, int64_t chunk, float* loss, float* lse,
                       float* row_kl, int32_t* gathered_idx, void* ws, size_t ws_bytes,
                       int32_t* dev_status, struct CUstream_st* stream) {
  int rc = check_inputs(h, W, teacher_idx, teacher_logits, valid, T, V, d, K, tau, chunk, ws,
                        dev_status);
  if (rc != KD_OK) return rc;
  if (!loss) return KD_ERR_INVALID_ARG;
  const Layout L = make_layout(T, V, d, K, chunk);
  if (ws_bytes < L.fwd_total) return KD_ERR_WORKSPACE;
  int sms = 0;
  if ((rc = device_sms(&sms)) != KD_OK) return rc;
  if (!encode_fn()) return KD_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const Ws w = carve(ws, L);
  const Variant var;
  if ((rc = run_prep(teacher_idx, teacher_logits, valid, T, K, V, 1.0f / tau, w, var, dev_status,
                     st)))
    return rc;
  return enqueue_forward(h, W, valid, T, V, d, K, tau, L, ws, w, var, sms, loss, lse, row_kl,
                         gathered_idx, dev_status, st);
}

int kd_topk_kl_backward(const void* h, const void* W, const int32_t* teacher_idx,
                        const float* teacher_logits, const uint8_t* valid, int64_t T, int64_t V,
                        int64_t d, int32_t K, float tau, int64_t chunk, const float* lse,
                        float grad_loss, float* dh, float* dW, void* ws, size_t ws_bytes,
                        int32_t* dev_status, struct CUstream_st* stream) {
  int rc = check_inputs(h, W, teacher_idx, teacher_logits, valid, T, V, d, K, tau, chunk, ws,
                        dev_status);
  if (rc != KD_OK) return rc;
  if (!lse || !dh || !dW || !aligned16(dh) || !aligned16(dW)) return KD_ERR_INVALID_ARG;
  if (!std::isfinite(grad_loss)) return KD_ERR_INVALID_ARG;
  const Layout L = make_layout(T, V, d, K, chunk);
  if (ws_bytes < L.bwd_total) return KD_ERR_WORKSPACE;
  int sms = 0;
  if ((rc = device_sms(&sms)) != KD_OK) return rc;
  if (!encode_fn()) return KD_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const Ws w = carve(ws, L);
  const Variant var;
  if ((rc = run_prep(teacher_idx, teacher_logits, valid, T, K, V, 1.0f / tau, w, var, dev_status,
                     st)))
    return rc;
  return enqueue_backward(h, W, valid, T, V, d, K, tau, L, ws, w, var, sms, lse, grad_loss, dh, dW,
                          0, dev_status, st);
}

int kd_topk_kl_forward_backward(const void* h, const void* W, const int32_t* teacher_idx,
                                const float* teacher_logits, const uint8_t* valid, int64_t T,
                                int64_t V, int64_t d, int32_t K, float tau, int64_t chunk,
                                float grad_loss, uint32_t flags, float* loss, float* lse,
                                float* row_kl, float* dh, float* dW, void* ws, size_t ws_bytes,
                                int32_t* dev_status, struct CUstream_st* stream) {
  int rc = check_inputs(h, W, teacher_idx, teacher_logits, valid, T, V, d, K, tau, chunk, ws,
                        dev_status);
  if (rc != KD_OK) return rc;
  if (!loss || !lse || !dh || !dW || !aligned16(dh) || !aligned16(dW)) return KD_ERR_INVALID_ARG;
  if (!std::isfinite(grad_loss) ||
      (flags & ~static_cast<uint32_t>(KD_ACCUMULATE_DW | KD_VALID_ROWS_ONLY)))
    return KD_ERR_INVALID_ARG;
  const Layout L = make_layout(T, V, d, K, chunk, true);
  if (ws_bytes < L.bwd_total) return KD_ERR_WORKSPACE;
  int sms = 0;
  if ((rc = device_sms(&sms)) != KD_OK) return rc;
  if (!encode_fn()) return KD_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const Ws w = carve(ws, L);
  const Variant var;
  if ((rc = run_prep(teacher_idx, teacher_logits, valid, T, K, V, 1.0f / tau, w, var, dev_status,
                     st)))
    return rc;
  return enqueue_sweep(h, W, teacher_idx, teacher_logits, valid, T, V, d, K, tau, L, ws, w, var,
                       sms, grad_loss, (flags & KD_ACCUMULATE_DW) ? 1 : 0,
                       (flags & KD_VALID_ROWS_ONLY) ? 1 : 0, loss, lse, row_kl, dh, dW, dev_status,
                       st);
}

int kd_gemm_bf16_diag(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t Kd,
                      int32_t a_mn, int32_t b_mn, int32_t* dev_status,
                      struct CUstream_st* stream) {
  if (!A || !B || !C || !dev_status) return KD_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || Kd < 1 || (a_mn != 0 && a_mn != 1) || (b_mn != 0 && b_mn != 1))
    return KD_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return KD_ERR_INVALID_ARG;
  if (M % 8 || N % 8 || Kd % 8 || M > INT32_MAX || N > INT32_MAX || Kd > INT32_MAX)
    return KD_ERR_UNSUPPORTED;
  int sms = 0;
  int rc = device_sms(&sms);
  if (rc != KD_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int BN = N >= 256 ? 256 : static_cast<int>(cdiv(N, 64) * 64);
  CUtensorMap ta, tb;
  const bool okA = a_mn ? make_map(&ta, A, M, Kd, M, 64) : make_map(&ta, A, Kd, M, Kd, BM);
  const bool okB = b_mn ? make_map(&tb, B, N, Kd, N, 64) : make_map(&tb, B, Kd, N, Kd, BN);
  if (!okA || !okB) return KD_ERR_CUDA;
  GemmParams p = base_params(a_mn, b_mn, BN);
  p.m_tiles = static_cast<int>(cdiv(M, BM));
  p.n_tiles = static_cast<int>(cdiv(N, BN));
  p.num_tiles = p.m_tiles * p.n_tiles;
  p.k_steps = static_cast<int>(cdiv(Kd, BK));
  p.ks_per_split = p.k_steps;
  // the shorter tile dimension runs fastest, so that the CTAs running
  // together share the operand slabs of the longer one
  p.n_fast = p.n_tiles <= p.m_tiles ? 1 : 0;
  p.group_m = p.m_tiles;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.status = dev_status;
  p.out = C;
  p.ld_out = N;
  if (cudaMemsetAsync(dev_status, 0, sizeof(int32_t), st) != cudaSuccess) return KD_ERR_CUDA;
  return launch_gemm<EPI_STORE>(ta, tb, ta, ta, p, sms, st);
}

int kd_gemm_bf16_diag_pair(const void* A, const void* B, float* C, int64_t M, int64_t N,
                           int64_t Kd, int32_t* dev_status, struct CUstream_st* stream) {
  if (!A || !B || !C || !dev_status) return KD_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || Kd < 1) return KD_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return KD_ERR_INVALID_ARG;
  if (M % 8 || N % 8 || Kd % 8 || M > INT32_MAX || N > INT32_MAX || Kd > INT32_MAX)
    return KD_ERR_UNSUPPORTED;
  int sms = 0;
  int rc = device_sms(&sms);
  if (rc != KD_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int BN = N >= 256 ? 256 : static_cast<int>(cdiv(N, 64) * 64);
  CUtensorMap ta, tb;
  if (!make_map(&ta, A, Kd, M, Kd, BM) || !make_map(&tb, B, Kd, N, Kd, BN / 2)) return KD_ERR_CUDA;
  GemmParams p = base_params(0, 0, BN);
  p.m_tiles = static_cast<int>(cdiv(M, BM));
  p.n_tiles = static_cast<int>(cdiv(N, BN));
  p.k_steps = static_cast<int>(cdiv(Kd, BK));
  p.ks_per_split = p.k_steps;
  p.n_fast = 0;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  pair_schedule(p, 16);
  p.status = dev_status;
  p.out = C;
  p.ld_out = N;
  if (cudaMemsetAsync(dev_status, 0, sizeof(int32_t), st) != cudaSuccess) return KD_ERR_CUDA;
  return launch_pair(ta, tb, p, sms, st);
}

int kd_pipeline_wait_selftest(uint64_t limit_ns, int32_t* dev_status,
                              struct CUstream_st* stream) {
  if (!dev_status || limit_ns == 0 || limit_ns > 1000000000ull) return KD_ERR_INVALID_ARG;
  int sms = 0;
  const int rc = device_sms(&sms);
  if (rc != KD_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(dev_status, 0, sizeof(int32_t), st) != cudaSuccess) return KD_ERR_CUDA;
  kd_wait_selftest_kernel<<<1, 32, 0, st>>>(limit_ns, dev_status);
  return cudaGetLastError() == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

int kd_topk_kl_forward_noalloc(const void* h, const void* W, const int32_t* teacher_idx,
                               const float* teacher_logits, const uint8_t* valid, int64_t T,
                               int64_t V, int64_t d, int32_t K, float tau, float* loss, float* lse,
                               float* row_kl, int32_t* gathered_idx, int32_t* dev_status,
                               struct CUstream_st* stream) {
  int rc = check_shape(T, V, d, K, 1);
  if (rc != KD_OK) return rc;
  if (make_layout(T, V, d, K, 1).fwd_total > kNoAllocScratchBytes) return KD_ERR_SCRATCH_LIMIT;
  int sms = 0;
  if ((rc = device_sms(&sms)) != KD_OK) return rc;
  void* ws = noalloc_scratch_address(&rc);
  if (!ws) return rc;
  // The forward resets, on `stream`, the valid-row counter and the status word
  // it accumulates into, and overwrites every other scratch entry it reads.
  return kd_topk_kl_forward(h, W, teacher_idx, teacher_logits, valid, T, V, d, K, tau, 1, loss,
                            lse, row_kl, gathered_idx, ws, kNoAllocScratchBytes, dev_status,
                            stream);
}


int kd_timing_start(int32_t capacity) {
  if (capacity < 1 || capacity > 1000000) return KD_ERR_INVALID_ARG;
  Timing& t = timing();
  std::lock_guard<std::mutex> lock(t.mu);
  destroy_timing_events(t);
  t.recs.resize(static_cast<size_t>(capacity));
  for (int i = 0; i < capacity; ++i) {
    t.recs[i].kind = -1;
    if (cudaEventCreate(&t.recs[i].start) != cudaSuccess ||
        cudaEventCreate(&t.recs[i].stop) != cudaSuccess) {
      t.recs.resize(static_cast<size_t>(i));  // keep only fully created pairs
      destroy_timing_events(t);
      t.recording = false;
      return KD_ERR_CUDA;
    }
  }
  t.capacity = capacity;
  t.used = 0;
  t.recording = true;
  return KD_OK;
}

int kd_timing_stop(void) {
  Timing& t = timing();
  std::lock_guard<std::mutex> lock(t.mu);
  t.recording = false;
  return KD_OK;
}

int kd_timing_query(int32_t kernel, int32_t* launches, double* total_ms) {
  if (!launches || !total_ms) return KD_ERR_INVALID_ARG;
  Timing& t = timing();
  std::lock_guard<std::mutex> lock(t.mu);
  int n = 0;
  double ms = 0.0;
  for (int i = 0; i < t.used; ++i) {
    if (t.recs[i].kind != kernel) continue;
    if (cudaEventSynchronize(t.recs[i].stop) != cudaSuccess) return KD_ERR_CUDA;
    float e = 0.f;
    if (cudaEventElapsedTime(&e, t.recs[i].start, t.recs[i].stop) != cudaSuccess)
      return KD_ERR_CUDA;
    ++n;
    ms += e;
  }
  *launches = n;
  *total_ms = ms;
  return KD_OK;
}

int kd_timing_release(void) {
  Timing& t = timing();
  std::lock_guard<std::mutex> lock(t.mu);
  t.recording = false;
  destroy_timing_events(t);
  return KD_OK;
}

int kd_topk_kl_forward_residual(const void* h, const void* W, const int32_t* teacher_idx,
                                const float* teacher_logits, const float* teacher_lse,
                                const uint8_t* valid, int64_t T, int64_t V, int64_t d, int32_t K,
                                float tau, int64_t chunk, float* loss, float* lse, float* row_kl,
                                float* outside_mass, void* ws, size_t ws_bytes,
                                int32_t* dev_status,
                                struct CUstream_st* stream) {
  int rc = check_inputs(h, W, teacher_idx, teacher_logits, valid, T, V, d, K, tau, chunk, ws,
                        dev_status);
  if (rc != KD_OK) return rc;
  if (!loss || !teacher_lse || (reinterpret_cast<uintptr_t>(teacher_lse) & 3u))
    return KD_ERR_INVALID_ARG;
  const Layout L = make_layout(T, V, d, K, chunk);
  if (ws_bytes < L.fwd_total) return KD_ERR_WORKSPACE;
  int sms = 0;
  if ((rc = device_sms(&sms)) != KD_OK) return rc;
  if (!encode_fn()) return KD_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const Ws w = carve(ws, L);
  Variant var;
  var.teacher_lse = teacher_lse;
  var.outside_mass_out = outside_mass;
  if ((rc = run_prep(teacher_idx, teacher_logits, valid, T, K, V, 1.0f / tau, w, var, dev_status,
                     st)))
    return rc;
  return enqueue_forward(h, W, valid, T, V, d, K, tau, L, ws, w, var, sms, loss, lse, row_kl,
                         nullptr, dev_status, st);
}

int kd_topk_kl_backward_residual(const void* h, const void* W, const int32_t* teacher_idx,
                                 const float* teacher_logits, const float* teacher_lse,
                                 const uint8_t* valid, int64_t T, int64_t V, int64_t d, int32_t K,
                                 float tau, int64_t chunk, const float* lse,
                                 const float* outside_mass, float grad_loss, float* dh, float* dW,
                                 void* ws, size_t ws_bytes, int32_t* dev_status,
                                 struct CUstream_st* stream) {
  int rc = check_inputs(h, W, teacher_idx, teacher_logits, valid, T, V, d, K, tau, chunk, ws,
                        dev_status);
  if (rc != KD_OK) return rc;
  if (!lse || !outside_mass || !teacher_lse || !dh || !dW || !aligned16(dh) || !aligned16(dW) ||
      (reinterpret_cast<uintptr_t>(teacher_lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(outside_mass) & 3u))
    return KD_ERR_INVALID_ARG;
  if (!std::isfinite(grad_loss)) return KD_ERR_INVALID_ARG;
  const Layout L = make_layout(T, V, d, K, chunk);
  if (ws_bytes < L.bwd_total) return KD_ERR_WORKSPACE;
  int sms = 0;
  if ((rc = device_sms(&sms)) != KD_OK) return rc;
  if (!encode_fn()) return KD_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const Ws w = carve(ws, L);
  Variant var;
  var.teacher_lse = teacher_lse;
  var.outside_mass_in = outside_mass;
  if ((rc = run_prep(teacher_idx, teacher_logits, valid, T, K, V, 1.0f / tau, w, var, dev_status,
                     st)))
    return rc;
  return enqueue_backward(h, W, valid, T, V, d, K, tau, L, ws, w, var, sms, lse, grad_loss, dh, dW,
                          0, dev_status, st);
}

int kd_topk_kl_forward_backward_residual(const void* h, const void* W, const int32_t* teacher_idx,
                                         const float* teacher_logits, const float* teacher_lse,
                                         const uint8_t* valid, int64_t T, int64_t V, int64_t d,
                                         int32_t K, float tau, int64_t chunk, float grad_loss,
                                         uint32_t flags, float* loss, float* lse, float* row_kl,
                                         float* outside_mass, float* dh, float* dW, void* ws,
                                         size_t ws_bytes, int32_t* dev_status,
                                         struct CUstream_st* stream) {
  int rc = check_inputs(h, W, teacher_idx, teacher_logits, valid, T, V, d, K, tau, chunk, ws,
                        dev_status);
  if (rc != KD_OK) return rc;
  if (!loss || !lse || !outside_mass || !dh || !dW || !aligned16(dh) || !aligned16(dW) ||
      !teacher_lse || (reinterpret_cast<uintptr_t>(teacher_lse) & 3u))
    return KD_ERR_INVALID_ARG;
  if (!std::isfinite(grad_loss) ||
      (flags & ~static_cast<uint32_t>(KD_ACCUMULATE_DW | KD_VALID_ROWS_ONLY)))
    return KD_ERR_INVALID_ARG;
  const Layout L = make_layout(T, V, d, K, chunk, true);
  if (ws_bytes < L.bwd_total) return KD_ERR_WORKSPACE;
  int sms = 0;
  if ((rc = device_sms(&sms)) != KD_OK) return rc;
  if (!encode_fn()) return KD_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const Ws w = carve(ws, L);
  Variant var;
  var.teacher_lse = teacher_lse;
  var.outside_mass_out = outside_mass;
  if ((rc = run_prep(teacher_idx, teacher_logits, valid, T, K, V, 1.0f / tau, w, var, dev_status,
                     st)))
    return rc;
  return enqueue_sweep(h, W, teacher_idx, teacher_logits, valid, T, V, d, K, tau, L, ws, w, var,
                       sms, grad_loss, (flags & KD_ACCUMULATE_DW) ? 1 : 0,
                       (flags & KD_VALID_ROWS_ONLY) ? 1 : 0, loss, lse, row_kl, dh, dW,
                       dev_status, st);
}

int kd_teacher_topk_workspace_size(int64_t T, int64_t V, int64_t d, int32_t K, int64_t chunk,
                                   size_t* bytes) {
  const int rc = check_shape(T, V, d, K, chunk);
  if (rc != KD_OK) return rc;
  if (!bytes) return KD_ERR_INVALID_ARG;
  *bytes = make_topk_layout(T, V, K, chunk).total;
  return KD_OK;
}

int kd_teacher_topk(const void* h, const void* W, int64_t T, int64_t V, int64_t d, int32_t K,
                    float tau, int64_t chunk, int32_t* topk_idx, float* topk_logits,
                    float* full_lse, void* ws, size_t ws_bytes, int32_t* dev_status,
                    struct CUstream_st* stream) {
  if (!h || !W || !topk_idx || !topk_logits || !ws || !dev_status) return KD_ERR_INVALID_ARG;
  if (!(tau > 0.f) || !std::isfinite(tau)) return KD_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(W) || !aligned16(ws) ||
      (reinterpret_cast<uintptr_t>(topk_idx) & 3u) ||
      (reinterpret_cast<uintptr_t>(topk_logits) & 3u) ||
      (reinterpret_cast<uintptr_t>(full_lse) & 3u) || (reinterpret_cast<uintptr_t>(dev_status) & 3u))
    return KD_ERR_INVALID_ARG;
  int rc = check_shape(T, V, d, K, chunk);
  if (rc != KD_OK) return rc;
  const TopkLayout L = make_topk_layout(T, V, K, chunk);
  if (ws_bytes < L.total) return KD_ERR_WORKSPACE;
  int sms = 0;
  if ((rc = device_sms(&sms)) != KD_OK) return rc;
  if (!encode_fn()) return KD_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* wb = static_cast<char*>(ws);
  float* part = reinterpret_cast<float*>(wb + L.part);
  uint64_t* tkeys = reinterpret_cast<uint64_t*>(wb + L.tkeys);
  uint64_t* theta = reinterpret_cast<uint64_t*>(wb + L.theta);
  float* theta_val = reinterpret_cast<float*>(wb + L.theta_val);
  int* cnt = reinterpret_cast<int*>(wb + L.cnt);
  uint64_t* cand = reinterpret_cast<uint64_t*>(wb + L.cand);
  float* z = reinterpret_cast<float*>(wb + L.z);
  if (cudaMemsetAsync(dev_status, 0, sizeof(int32_t), st) != cudaSuccess) return KD_ERR_CUDA;
  const float inv_tau = 1.0f / tau;
  for (int64_t c0 = 0; c0 < T; c0 += L.C) {
    const int64_t rows = (T - c0) < L.C ? (T - c0) : L.C;
    const void* hc = static_cast<const __nv_bfloat16*>(h) + c0 * d;
    CUtensorMap ta, tb, tz;
    if (!make_map(&ta, hc, d, rows, d, BM) || !make_map(&tb, W, d, V, d, ZBN) ||
        !make_map_f32(&tz, z, V, rows, V, 32, 32, true))
      return KD_ERR_CUDA;
    // the contraction: tile maxima, lse partials, and the logits into z
    GemmParams p = base_params(0, 0, ZBN);
    logit_schedule(p, rows, V, d);
    p.status = dev_status;
    p.inv_tau = inv_tau;
    p.c_log2 = LOG2E * inv_tau;
    p.part = part;
    p.part_ld = rows;
    p.tkeys = tkeys;
    if ((rc = launch_gemm<EPI_TMAX>(ta, tb, tz, ta, p, sms, st))) return rc;
    const unsigned blocks = static_cast<unsigned>(cdiv(rows, TOPK_WARPS));
    kd_topk_threshold_kernel<<<blocks, 32 * TOPK_WARPS, 0, st>>>(
        tkeys, part, rows, static_cast<int>(rows), L.n_tiles, K, theta, theta_val,
        full_lse ? full_lse + c0 : nullptr, dev_status);
    if (cudaMemsetAsync(cnt, 0, static_cast<size_t>(rows) * 4, st) != cudaSuccess)
      return KD_ERR_CUDA;
    // candidates at or above the threshold, from the stored logits
    const int slot = timing_slot(KD_KERNEL_TOPK_SCAN);
    if (slot >= 0 &&
        cudaEventRecord(timing().recs[static_cast<size_t>(slot)].start, st) != cudaSuccess)
      return KD_ERR_CUDA;
    kd_topk_scan_kernel<<<static_cast<unsigned>(rows), SCAN_THREADS, 0, st>>>(
        z, V, static_cast<int>(V), theta, theta_val, cand, cnt, L.cap, dev_status);
    if (slot >= 0 &&
        cudaEventRecord(timing().recs[static_cast<size_t>(slot)].stop, st) != cudaSuccess)
      return KD_ERR_CUDA;
    kd_topk_finalize_kernel<<<blocks, 32 * TOPK_WARPS, 0, st>>>(
        cand, cnt, L.cap, theta_val, static_cast<int>(rows), K, topk_idx + c0 * K,
        topk_logits + c0 * K, dev_status);
    if (cudaGetLastError() != cudaSuccess) return KD_ERR_CUDA;
  }
  return KD_OK;
}

int kd_entropy_filter_workspace_size(int64_t T, size_t* bytes) {
  if (T < 1 || !bytes) return KD_ERR_INVALID_ARG;
  if (T > INT32_MAX) return KD_ERR_UNSUPPORTED;
  *bytes = al256(static_cast<size_t>(T + 3) / 4 * 16);  // keys, padded to whole uint4
  return KD_OK;
}

int kd_entropy_filter(const float* teacher_logits, const uint8_t* valid_in, int64_t T, int32_t K,
                      float tau, int32_t keep_num, int32_t keep_den, uint8_t* valid_out,
                      float* entropy, void* ws, size_t ws_bytes, int32_t* dev_status,
                      struct CUstream_st* stream) {
  if (!teacher_logits || !valid_in || !valid_out || !ws || !dev_status) return KD_ERR_INVALID_ARG;
  if (T < 1 || K < 1 || !(tau > 0.f) || !std::isfinite(tau)) return KD_ERR_INVALID_ARG;
  if (keep_den < 1 || keep_num < 0 || keep_num > keep_den) return KD_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(teacher_logits) & 3u) ||
      (reinterpret_cast<uintptr_t>(entropy) & 3u) || (reinterpret_cast<uintptr_t>(ws) & 255u) ||
      (reinterpret_cast<uintptr_t>(dev_status) & 3u))
    return KD_ERR_INVALID_ARG;
  if (T > INT32_MAX || static_cast<double>(T) * K > 2e9) return KD_ERR_UNSUPPORTED;
  if (ws_bytes < al256(static_cast<size_t>(T + 3) / 4 * 16)) return KD_ERR_WORKSPACE;
  int sms = 0;
  const int rc = device_sms(&sms);
  if (rc != KD_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(dev_status, 0, sizeof(int32_t), st) != cudaSuccess) return KD_ERR_CUDA;
  uint32_t* keys = static_cast<uint32_t*>(ws);
  const int rows_per_block = 8;
  kd_entropy_kernel<<<static_cast<unsigned>(cdiv(T, rows_per_block)), 32 * rows_per_block, 0,
                      st>>>(teacher_logits, valid_in, static_cast<int>(T), K, 1.0f / tau, entropy,
                            keys);
  kd_entropy_select_kernel<<<1, FILTER_THREADS, 0, st>>>(keys, static_cast<int>(T), keep_num,
                                                         keep_den, valid_out);
  return cudaGetLastError() == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

}  // extern "C"
