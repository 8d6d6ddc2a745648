// C-ABI of the fused linear cross-entropy library: argument validation,
// workspace planning, TMA tensor-map encoding and the stream-ordered launch
// sequence of the forward and backward passes.
//
// Forward (one call):  gemm<kLse>  ->  lse_merge  ->  loss_finalize
// Backward (one call): grad_scale, then for each vocabulary chunk
//                      [v0, v0 + Cv):  gemm<kDz> (recompute Z, write dZ chunk)
//                                      gemm<kStore> dW[v0:v0+Cv] = dZ^T X
//                                      gemm<kStore> dX_acc += dZ W[v0:v0+Cv]
//                      then dx_finalize (bf16 inputs).
// Merged backward (opt-in, CTA-pair tiles without the optional features):
// gemm<kDz> for chunk 0 alone, then one bwd_fused launch per chunk c running
// dW(c), dX(c) and the dZ recompute of chunk c+1 from one tile list; the dZ
// scratch is two N x Cv buffers used in turn.
// Running the vocabulary chunks outermost lets the dW GEMM contract over all
// N tokens at once, so every dW row is written exactly once per call (no
// read-modify-write of the V x H fp32 gradient), while the N x Cv bf16
// gradient chunk stays the only logit-shaped buffer -- the bounded
// "scratchpad" of "Chunked and Fused Cross-Entropy ...", step 1, with the
// roles of rows and vocabulary swapped.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <numeric>
#include <string>
#include <vector>

#include "flce.h"
#include "aux_kernels.cuh"
#include "bwd_fused.cuh"
#include "gemm_core.cuh"
#include "ptx.cuh"

using namespace flce;

namespace {

constexpr int kStages = 4;       // 1-CTA tiles: 4 x 48 KB stages
constexpr int kPairStages = 6;   // CTA-pair tiles: 6 x 32 KB stages per CTA
constexpr int64_t kPartialsBudget = 32ll << 20;   // bytes of forward partials
constexpr int64_t kDzBudgetMin = 256ll << 20;     // bytes of all dZ chunk buffers, at least
constexpr int64_t kDzRowsEquiv = 1024;            // ... and as many as this many rows of logits
constexpr unsigned long long kTimeoutNs = 2000000000ull;
constexpr size_t kAlign = 256;

thread_local std::string g_last_cuda_error;
thread_local int g_launches = 0;
thread_local int g_quad_launches = 0;  // launches of the last call that took the QUAD walk
// Process-wide defaults of the launch settings; a call whose options set a
// field itself does not read the matching default.
std::atomic<int64_t> g_vocab_chunk{0};
std::atomic<int> g_cta_pair{1};
std::atomic<int> g_bwd_merge{0};
std::atomic<int> g_l2_hints{0};
std::atomic<int> g_cluster_mcast{1};

// Launch settings of one call, resolved once at its entry from its options
// and the process-wide defaults, and used for both the workspace plan and the
// launches.
struct Tuning {
  bool pair;           // 256 x 256 CTA-pair tiles (else 128 x 256 single-CTA)
  int merge;           // backward layout (pair tiles only): 0 three launches per chunk,
                       // 1 dW(c) + dX(c) + dZ(c+1) merged (two dZ buffers),
                       // 2 dW(c) + dX(c) merged after dZ(c) (one dZ buffer)
  bool l2_hints;       // evict_last policy on the re-read operand
  int64_t chunk_set;   // requested vocabulary chunk width (0 = automatic)
  bool mcast;          // pair launches may take 4-CTA clusters with operand multicast
};

Tuning default_tuning() {
  return Tuning{g_cta_pair.load() != 0, g_bwd_merge.load(), g_l2_hints.load() != 0,
                g_vocab_chunk.load(), g_cluster_mcast.load() != 0};
}

// Optional per-kernel timing: CUDA events recorded on the caller's stream
// around every GEMM launch (kinds: forward logits+LSE, dZ recompute, dW, dX,
// merged backward).
constexpr int kProfKinds = 5;
struct ProfRec {
  int kind;
  cudaEvent_t start, stop;
};
thread_local bool g_prof_on = false;
thread_local std::vector<ProfRec> g_prof_pending;
thread_local std::vector<cudaEvent_t> g_prof_pool;
thread_local double g_prof_ms[kProfKinds] = {};
thread_local int g_prof_n[kProfKinds] = {};

cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

flce_status cuda_fail(cudaError_t e, const char* what) {
  char buf[256];
  snprintf(buf, sizeof buf, "%s: %s", what, cudaGetErrorString(e));
  g_last_cuda_error = buf;
  return FLCE_ERR_CUDA;
}

#define FLCE_CUDA(call)                                  \
  do {                                                   \
    cudaError_t e_ = (call);                             \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call);  \
  } while (0)

// ---------------------------------------------------------------------------
// Workspace plan: depends only on the shape, dtype, mode and chunk setting.
// ---------------------------------------------------------------------------
struct Plan {
  int64_t N, H, V;
  int m_blocks, m_pad, v_tiles, group_len, n_groups, merge_blocks;
  int64_t chunk;
  int n_chunks;
  int dz_bufs;  // 2 when the merged backward may run (dZ of chunk c+1 beside chunk c)
  bool counters;  // one tile counter per chunk (merged launches of either layout)
  size_t off_scalars, off_blocks, off_partials, off_block_loss, off_block_valid, off_dz,
      off_dz2, off_counters, off_dxacc, off_xcast, off_wcast, off_mask_x, off_mask_w, total;
  // gradient-filter masks (sized for 128-row tiles, the smaller tile shape)
  int mask_x_ld, mask_w_ld;
  int n_blocks128;  // token blocks of 128 rows (the finest skip granularity)
};

bool shape_ok(int64_t N, int64_t H, int64_t V) {
  if (N < 0 || H <= 0 || V <= 0) return false;
  if (H % 8 != 0) return false;
  // TMA coordinates and the kernels' tile indices are 32-bit.
  if (N > (int64_t)INT32_MAX - 1024 || V > (int64_t)INT32_MAX - 1024 || H > (int64_t)INT32_MAX)
    return false;
  return true;
}

// Whether backward calls may take the merged launches of dW(c), dX(c) and
// dZ(c+1) (CTA-pair tiles only); their workspace then holds two dZ buffers.
bool merge_planned(const Tuning& t) { return t.merge == 1 && t.pair; }
// Whether backward calls may merge only dW(c) and dX(c) (one dZ buffer).
bool merge_dwdx_planned(const Tuning& t) { return t.merge == 2 && t.pair; }
int dz_buffers(const Tuning& t) { return merge_planned(t) ? 2 : 1; }

// CTA pairs of a persistent launch on the current device (76 on a 152-SM
// GB300, also the value when no device can be queried).
int64_t device_pairs() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      sms >= 2)
    return sms / 2;
  (void)cudaGetLastError();  // clear the failed query's error
  return 76;
}

// Three-launch backward: the dW launch of a chunk has (Cv / 256) x ceil(H / 256)
// tiles, whose last wave of CTA pairs is partly idle unless the count is a
// whole number of waves.  Among the widths that keep at least 7/8 of the
// budget width -- multiples of 256, of 512 when ceil(H / 256) is odd (so the
// dW launch's row blocks pair up for the multicast walk) -- the one whose dW
// launch fills its last wave best is taken (the widest within half a point
// of the best), but the widest width stays unless that best fill beats its
// fill by 2.5 points.  Measured on a GB300: Llama-3 shape 16384 ->
// 14592 (912 tiles, 12 whole waves; 2.6% faster dW launches); Qwen-2.5 shape
// 9216 -> 8192 (dW at 9216 ran 2.5% slower, its last wave 95% full against 98%).
int64_t wave_fit(int64_t c, int64_t H) {
  const int64_t pairs = device_pairs();
  const int64_t hb = ceil_div(H, BN);
  const int64_t unit = (hb % 2) ? 512 : 256;
  auto fill = [&](int64_t w) {
    const int64_t tiles = (w / 256) * hb;
    return (double)tiles / (double)(ceil_div(tiles, pairs) * pairs);
  };
  const int64_t widest = c / unit * unit;
  if (widest < unit) return std::max<int64_t>(256, c / 256 * 256);
  double top = 0.0;
  for (int64_t w = widest; w >= unit && w * 8 >= c * 7; w -= unit) top = std::max(top, fill(w));
  if (top <= fill(widest) + 0.025) return widest;
  for (int64_t w = widest; w >= unit && w * 8 >= c * 7; w -= unit)
    if (fill(w) >= top - 0.005) return w;
  return widest;
}

// Bytes the dZ buffers may take together by default: as much as 1024 token
// rows of bf16 logits over the whole vocabulary -- the fully fused chunk of
// "Fused cross-entropy -- the memory kernel" (a B*T chunk of 1024 rows, 0.26 GB
// at V = 128256) -- and at least 256 MiB.  The N x Cv chunk then holds the same
// bytes as the pages' 1024 x V one, with the roles of tokens and vocabulary
// swapped.
int64_t dz_budget(int64_t V) { return std::max<int64_t>(kDzBudgetMin, kDzRowsEquiv * V * 2); }

// Cv: the dZ buffers together take at most dz_budget(V) (default) and at most
// half of the N x V logits (each buffer at most V / (2 * buffers) columns).
// The default width is a multiple of 512 (an even number of 256-column blocks,
// so the weight-gradient launch's row blocks pair up for the multicast walk)
// and is wave-aligned for the three-launch backward.
int64_t auto_chunk(int64_t N, int64_t H, int64_t V, const Tuning& t) {
  const int bufs = dz_buffers(t);
  const int64_t half = std::max<int64_t>(256, (V / (2 * bufs)) / 256 * 256);
  const int64_t set = t.chunk_set;
  if (set > 0) return std::min(std::max<int64_t>(ceil_div(set, 256) * 256, 256), half);
  int64_t c = (dz_budget(V) / bufs / (std::max<int64_t>(N, 1) * 2)) / 512 * 512;
  c = std::min(std::max<int64_t>(c, 256), half);
  return merge_planned(t) ? c : wave_fit(c, H);
}

bool make_plan(int64_t N, int64_t H, int64_t V, flce_dtype dtype, int mode, const Tuning& t,
               Plan* pl) {
  if (!shape_ok(N, H, V)) return false;
  if (dtype != FLCE_BF16 && dtype != FLCE_FP32) return false;
  if (mode < FLCE_MODE_FWD || mode > FLCE_MODE_FWD_BWD) return false;
  Plan& p = *pl;
  p.N = N;
  p.H = H;
  p.V = V;
  p.m_blocks = (int)ceil_div(std::max<int64_t>(N, 1), 2 * BM);
  p.m_pad = p.m_blocks * 2 * BM;  // covers the row padding of either tile shape
  p.v_tiles = (int)ceil_div(V, BN);
  int L = 1;
  while ((int64_t)ceil_div(p.v_tiles, L) * p.m_pad * 16 > kPartialsBudget && L < p.v_tiles) L *= 2;
  p.group_len = L;
  p.n_groups = (int)ceil_div(p.v_tiles, L);
  p.merge_blocks = (int)merge_block_count(N);
  p.chunk = auto_chunk(N, H, V, t);
  p.n_chunks = (int)ceil_div(V, p.chunk);
  p.dz_bufs = dz_buffers(t);
  p.counters = merge_planned(t) || merge_dwdx_planned(t);
  const bool fwd = mode & FLCE_MODE_FWD;
  const bool bwd = mode & FLCE_MODE_BWD;
  size_t off = 0;
  p.off_scalars = off;
  off += kAlign;
  // skip lists: flags[nb], list[nb], count -- nb counted at 128-row granularity
  p.n_blocks128 = (int)ceil_div(std::max<int64_t>(N, 1), BM);
  p.off_blocks = off;
  off = align_up(off + (size_t)(2 * p.n_blocks128 + 1) * sizeof(int), kAlign);
  p.off_partials = p.off_block_loss = p.off_block_valid = 0;
  if (fwd) {
    p.off_partials = off;
    off = align_up(off + (size_t)p.n_groups * p.m_pad * sizeof(float4), kAlign);
    p.off_block_loss = off;
    off = align_up(off + (size_t)p.merge_blocks * sizeof(double), kAlign);
    p.off_block_valid = off;
    off = align_up(off + (size_t)p.merge_blocks * sizeof(int), kAlign);
  }
  p.off_dz = p.off_dz2 = p.off_counters = p.off_dxacc = 0;
  if (bwd) {
    p.off_dz = off;
    off = align_up(off + (size_t)std::max<int64_t>(N, 1) * p.chunk * 2, kAlign);
    if (p.dz_bufs == 2) {
      p.off_dz2 = off;
      off = align_up(off + (size_t)std::max<int64_t>(N, 1) * p.chunk * 2, kAlign);
    }
    if (p.counters) {
      p.off_counters = off;  // one tile counter per merged launch
      off = align_up(off + (size_t)p.n_chunks * sizeof(int), kAlign);
    }
    if (dtype == FLCE_BF16) {
      p.off_dxacc = off;
      off = align_up(off + (size_t)N * H * 4, kAlign);
    }
    p.mask_x_ld = (int)align_up((size_t)ceil_div(p.chunk, BK), 16);
    p.mask_w_ld = (int)align_up((size_t)ceil_div(std::max<int64_t>(N, 1), BK), 16);
    p.off_mask_x = off;
    off = align_up(off + (size_t)ceil_div(std::max<int64_t>(N, 1), BM) * p.mask_x_ld, kAlign);
    p.off_mask_w = off;
    off = align_up(off + (size_t)ceil_div(p.chunk, BM) * p.mask_w_ld, kAlign);
  }
  p.off_xcast = p.off_wcast = 0;
  if (dtype == FLCE_FP32) {
    p.off_xcast = off;
    off = align_up(off + (size_t)N * H * 2, kAlign);
    p.off_wcast = off;
    off = align_up(off + (size_t)V * H * 2, kAlign);
  }
  p.total = off;
  return true;
}

#ifdef FLCE_DEBUG
// Debug build: the regions a call of `mode` uses lie inside the plan's total,
// in ascending order, without overlap, and the dZ chunk width is at most half
// the vocabulary (or the 256-column minimum).
bool plan_regions_ok(const Plan& p, flce_dtype dtype, int mode) {
  struct R {
    size_t off, bytes;
  };
  const size_t n1 = (size_t)std::max<int64_t>(p.N, 1);
  std::vector<R> rs;
  rs.push_back({p.off_scalars, kAlign});
  rs.push_back({p.off_blocks, (size_t)(2 * p.n_blocks128 + 1) * sizeof(int)});
  if (mode & FLCE_MODE_FWD) {
    rs.push_back({p.off_partials, (size_t)p.n_groups * p.m_pad * sizeof(float4)});
    rs.push_back({p.off_block_loss, (size_t)p.merge_blocks * sizeof(double)});
    rs.push_back({p.off_block_valid, (size_t)p.merge_blocks * sizeof(int)});
  }
  if (mode & FLCE_MODE_BWD) {
    rs.push_back({p.off_dz, n1 * (size_t)p.chunk * 2});
    if (p.dz_bufs == 2) rs.push_back({p.off_dz2, n1 * (size_t)p.chunk * 2});
    if (p.counters) rs.push_back({p.off_counters, (size_t)p.n_chunks * sizeof(int)});
    if (dtype == FLCE_BF16) rs.push_back({p.off_dxacc, (size_t)p.N * p.H * 4});
    rs.push_back({p.off_mask_x, (size_t)ceil_div((int64_t)n1, BM) * p.mask_x_ld});
    rs.push_back({p.off_mask_w, (size_t)ceil_div(p.chunk, BM) * p.mask_w_ld});
  }
  if (dtype == FLCE_FP32) {
    rs.push_back({p.off_xcast, (size_t)p.N * p.H * 2});
    rs.push_back({p.off_wcast, (size_t)p.V * p.H * 2});
  }
  size_t end = 0;
  for (const R& r : rs) {
    if (r.off < end || r.off % kAlign != 0 || r.off + r.bytes > p.total) return false;
    end = r.off + r.bytes;
  }
  return p.chunk >= 256 && p.chunk % 256 == 0 && p.chunk <= std::max<int64_t>(256, p.V / 2) &&
         p.n_chunks * p.chunk >= p.V && (int64_t)p.m_pad >= p.N;
}
#endif

// ---------------------------------------------------------------------------
// Device properties and kernel attributes (cached per device).
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
int g_num_sms[kMaxDevices] = {0};
bool g_dev_ok[kMaxDevices] = {false};

flce_status device_check(int* dev_out, int* sms_out) {
  int dev = 0;
  FLCE_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return FLCE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_dev_mutex);
  if (!g_num_sms[dev]) {
    int major = 0, minor = 0, sms = 0;
    FLCE_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    FLCE_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    FLCE_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    g_dev_ok[dev] = (major == 10 && minor == 3);
    g_num_sms[dev] = sms;
  }
  if (!g_dev_ok[dev]) return FLCE_ERR_UNSUPPORTED;
  *dev_out = dev;
  *sms_out = g_num_sms[dev];
  return FLCE_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D tiled tensor map, 128-byte swizzle.  inner/outer in elements.
flce_status make_map(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* base,
                     uint64_t inner, uint64_t outer, uint64_t pitch_bytes, uint32_t box_inner,
                     uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) {
    g_last_cuda_error = "cuTensorMapEncodeTiled entry point unavailable";
    return FLCE_ERR_CUDA;
  }
  (void)elem_bytes;
  cuuint64_t dims[2] = {inner, std::max<uint64_t>(outer, 1)};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[200];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d): inner=%llu outer=%llu pitch=%llu",
             (int)r, (unsigned long long)inner, (unsigned long long)outer,
             (unsigned long long)pitch_bytes);
    g_last_cuda_error = buf;
    return FLCE_ERR_CUDA;
  }
  return FLCE_OK;
}

// bf16 operand maps
flce_status map_kmajor(CUtensorMap* m, const void* base, uint64_t k, uint64_t rows,
                       uint64_t pitch_elems, uint32_t box_rows) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, k, rows, pitch_elems * 2, BK,
                  box_rows);
}
flce_status map_mnmajor(CUtensorMap* m, const void* base, uint64_t mn, uint64_t k,
                        uint64_t pitch_elems) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, mn, k, pitch_elems * 2, 64, BK);
}
// dZ chunk store map: 64 bf16 columns x 32 rows
flce_status map_dz_store(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                         uint64_t pitch_elems) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, cols, rows, pitch_elems * 2, 64,
                  32);
}
// fp32 output map: 32 columns x 32 rows
flce_status map_f32_out(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                        uint64_t pitch_elems) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, cols, rows, pitch_elems * 4, 32,
                  32);
}

// One-time set-up of a kernel on one device: its dynamic shared-memory limit
// and, for cluster kernels, how many 2-CTA clusters of it fit at once.  Done
// under call_once, and the outcome -- a CUDA error included -- is kept, so
// every later call on that device sees the same result.
struct KernelSetup {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  const char* what = "";
  int max_clusters = 0;
};

template <typename Kern>
void setup_kernel(KernelSetup& ks, Kern kern, int smem, bool cluster, int num_sms) {
  std::call_once(ks.once, [&] {
    ks.err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    ks.what = "cudaFuncSetAttribute";
    if (ks.err != cudaSuccess || !cluster) return;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    int n = 0;
    ks.err = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    ks.what = "cudaOccupancyMaxActiveClusters";
    ks.max_clusters = std::max(1, std::min(n, num_sms / 2));
  });
}

// Persistent launches take their work units round robin, so a launch lasts
// ceil(units / workers) rounds.  The fewest workers (a multiple of `step`)
// that keep that round count leave the other SMs idle for the whole launch
// rather than for its last round; under the GB300's power cap the power they
// leave goes to the clock of the busy ones (measured: 0.8% faster steps at
// the Gemma-2 shape, whose dW and dX launches end on partial rounds; no
// change at the other shapes).
int fewest_workers(int units, int max_workers, int step) {
  const int w = std::min(units, max_workers) / step * step;
  if (w < step) return std::min(units, max_workers);
  const int rounds = (units + w - 1) / w;
  const int need = (units + rounds - 1) / rounds;
  return std::min(w, (need + step - 1) / step * step);
}

template <Epi EPI, bool A_MN, bool B_MN, bool PAIR, bool EXT>
flce_status launch_gemm(int dev, int num_sms, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& out, const GemmParams& p, cudaStream_t st,
                        int prof_kind = -1) {
  constexpr int stages = PAIR ? kPairStages : kStages;
  auto kern = [] {
    if constexpr (PAIR)
      return gemm_pair_kernel<EPI, A_MN, B_MN, stages, EXT>;
    else
      return gemm_kernel<EPI, A_MN, B_MN, stages, EXT>;
  }();
  constexpr int smem = gemm_smem_bytes<EPI, stages, PAIR, EXT>();
  static KernelSetup setup[kMaxDevices];
  setup_kernel(setup[dev], kern, smem, PAIR, num_sms);
  if (setup[dev].err != cudaSuccess) return cuda_fail(setup[dev].err, setup[dev].what);
  if (p.num_units <= 0) return FLCE_OK;
  // One CTA per SM (one cluster per SM pair), persistent over the work units.
  // A persistent grid must be co-resident, so pairs are capped by how many
  // 2-CTA clusters of this size fit on the device at once.
  int grid = fewest_workers(p.num_units, num_sms, 1);
  if constexpr (PAIR) grid = 2 * fewest_workers(p.num_units, setup[dev].max_clusters, 1);
  ProfRec rec{prof_kind, nullptr, nullptr};
  if (g_prof_on && prof_kind >= 0) {
    rec.start = prof_event();
    rec.stop = prof_event();
    if (rec.start && rec.stop) FLCE_CUDA(cudaEventRecord(rec.start, st));
  }
  kern<<<grid, NUM_THREADS, smem, st>>>(a, b, out, p);
  ++g_launches;
  FLCE_CUDA(cudaGetLastError());
  if (rec.start && rec.stop) {
    FLCE_CUDA(cudaEventRecord(rec.stop, st));
    g_prof_pending.push_back(rec);
  }
  return FLCE_OK;
}

// The walk of a CTA-pair launch: plain pairs (2-CTA clusters), or the QUAD
// walk (4-CTA clusters preferred, the two pairs of a cluster multicasting the
// operand their tiles share; see gemm_core.cuh).
struct Walk {
  bool quad = false;
  bool share_b = false;  // QUAD: the pairs share B (differ in row block), else A
};

// QUAD needs whole groups of two pairs whose units pair up exactly: units
// 2v and 2v+1 must differ only in the row block (share B) or only in the
// column group (share A, group length 1), and every unit needs its partner.
Walk pick_walk(const Tuning& t, bool pair, bool ext, const GemmParams& p) {
  Walk w;
  if (!pair || ext || !t.mcast || p.num_units < 4 || p.num_units % 2 != 0) return w;
  if (p.m_fastest) {
    const bool banded = p.m_band > 0 && p.m_band < p.m_blocks;
    if (p.m_blocks % 2 != 0 || (banded && p.m_band % 2 != 0)) return w;
    w.quad = w.share_b = true;
  } else if (p.group_len == 1 && p.n_groups % 2 == 0) {
    w.quad = true;
  } else if (p.m_blocks % 2 == 0) {
    w.quad = w.share_b = true;
  }
  return w;
}

// Rows of a K-major operand box: QUAD loads every operand half as two 64-row
// boxes; pairs load their 128 rows of A and of B in one box each, single CTAs
// 128 rows of A and 256 of B.
uint32_t a_box_rows(const Walk& w) { return w.quad ? 64 : BM; }
uint32_t b_box_rows(bool pair, const Walk& w) { return w.quad ? 64 : (pair ? BN / 2 : BN); }

template <Epi EPI, bool A_MN, bool B_MN, bool SHARE_B>
flce_status launch_quad(int dev, int num_sms, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& out, const GemmParams& p, cudaStream_t st,
                        int prof_kind) {
  auto kern = gemm_quad_kernel<EPI, A_MN, B_MN, kPairStages, SHARE_B>;
  constexpr int smem = gemm_smem_bytes<EPI, kPairStages, true, false>();
  static KernelSetup setup[kMaxDevices];
  setup_kernel(setup[dev], kern, smem, false, num_sms);
  if (setup[dev].err != cudaSuccess) return cuda_fail(setup[dev].err, setup[dev].what);
  if (p.num_units <= 0) return FLCE_OK;
  // An even number of pairs (the fewest that keep the round count), so that
  // the two pairs of every group of four CTAs take partner units; the
  // hardware groups each four into one 4-CTA cluster where it can, else into
  // two 2-CTA clusters (no multicast).
  const int pairs = fewest_workers(p.num_units, num_sms / 2, 2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributePreferredClusterDimension;
  at[1].val.preferredClusterDim.x = 4;
  at[1].val.preferredClusterDim.y = 1;
  at[1].val.preferredClusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  ProfRec rec{prof_kind, nullptr, nullptr};
  if (g_prof_on && prof_kind >= 0) {
    rec.start = prof_event();
    rec.stop = prof_event();
    if (rec.start && rec.stop) FLCE_CUDA(cudaEventRecord(rec.start, st));
  }
  FLCE_CUDA(cudaLaunchKernelEx(&cfg, kern, a, b, out, p));
  ++g_launches;
  ++g_quad_launches;
  if (rec.start && rec.stop) {
    FLCE_CUDA(cudaEventRecord(rec.stop, st));
    g_prof_pending.push_back(rec);
  }
  return FLCE_OK;
}

// Run-time choice between the 1-CTA (128 x 256), CTA-pair (256 x 256) and
// QUAD kernels.
template <Epi EPI, bool A_MN, bool B_MN>
flce_status launch_tile(bool pair, bool ext, const Walk& w, int dev, int num_sms,
                        const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& out,
                        const GemmParams& p, cudaStream_t st, int prof_kind = -1) {
  if (w.quad)
    return w.share_b ? launch_quad<EPI, A_MN, B_MN, true>(dev, num_sms, a, b, out, p, st, prof_kind)
                     : launch_quad<EPI, A_MN, B_MN, false>(dev, num_sms, a, b, out, p, st, prof_kind);
  if (ext)
    return pair ? launch_gemm<EPI, A_MN, B_MN, true, true>(dev, num_sms, a, b, out, p, st, prof_kind)
                : launch_gemm<EPI, A_MN, B_MN, false, true>(dev, num_sms, a, b, out, p, st, prof_kind);
  return pair ? launch_gemm<EPI, A_MN, B_MN, true, false>(dev, num_sms, a, b, out, p, st, prof_kind)
              : launch_gemm<EPI, A_MN, B_MN, false, false>(dev, num_sms, a, b, out, p, st, prof_kind);
}

// One merged backward launch (CTA pairs, persistent; the list's tiles go round
// robin except the last DYNAMIC_ROUNDS rounds, taken from a global counter).
flce_status launch_fused(int dev, int num_sms, const FusedMaps& maps, const FusedParams& p,
                         cudaStream_t st) {
  constexpr int smem = fused_smem_bytes<kPairStages>();
  auto kern = bwd_fused_kernel<kPairStages>;
  static KernelSetup setup[kMaxDevices];
  setup_kernel(setup[dev], kern, smem, true, num_sms);
  if (setup[dev].err != cudaSuccess) return cuda_fail(setup[dev].err, setup[dev].what);
  if (p.total_tiles <= 0) return FLCE_OK;
  const int pairs = std::min(p.total_tiles, setup[dev].max_clusters);
  const int grid = 2 * pairs;
  // all but the last DYNAMIC_ROUNDS rounds of tiles go round robin
  FusedParams pp = p;
  pp.static_tiles = std::max(0, (p.total_tiles - DYNAMIC_ROUNDS * pairs) / pairs * pairs);
  ProfRec rec{4, nullptr, nullptr};
  if (g_prof_on) {
    rec.start = prof_event();
    rec.stop = prof_event();
    if (rec.start && rec.stop) FLCE_CUDA(cudaEventRecord(rec.start, st));
  }
  kern<<<grid, NUM_THREADS, smem, st>>>(maps, pp);
  ++g_launches;
  FLCE_CUDA(cudaGetLastError());
  if (rec.start && rec.stop) {
    FLCE_CUDA(cudaEventRecord(rec.stop, st));
    g_prof_pending.push_back(rec);
  }
  return FLCE_OK;
}

// Row-block bands for the launches that re-read X (forward, dZ recompute):
// with all row blocks in flight, X (N x H bf16) competes in L2 with the
// streamed W tiles and is re-read from DRAM several times.  Splitting the row
// blocks into ceil(X / 40 MiB) bands (at most 4) walked one after another costs
// one more pass over W per band but keeps each band's X resident; measured on
// a GB300 it cut the dZ launch's DRAM reads from ~1.0 to 0.42 GB at the
// Llama-3 shape and sped the step up ~2% (Llama-3 and Gemma-2 shapes).
int x_band(int64_t N, int64_t H, int m_blocks) {
  const double x_bytes = (double)N * H * 2;
  if (x_bytes <= 48.0 * (1 << 20)) return 0;
  const int bands = (int)std::min(4.0, std::ceil(x_bytes / (40.0 * (1 << 20))));
  return bands > 1 ? (m_blocks + bands - 1) / bands : 0;
}

// Fraction of the reused operand's lines kept in L2 with evict_last priority:
// about 64 MB of the 129 MB L2 is given to it, the rest streams.
float l2_keep_fraction(const Tuning& t, double operand_bytes) {
  if (!t.l2_hints || operand_bytes <= 0) return 0.f;
  return (float)std::min(1.0, (64.0 * (1 << 20)) / operand_bytes);
}
int tile_rows(bool pair) { return pair ? 2 * BM : BM; }
uint32_t b_box_rows(bool pair) { return pair ? BN / 2 : BN; }

#define FLCE_TRY(expr)                   \
  do {                                   \
    flce_status s_ = (expr);             \
    if (s_ != FLCE_OK) return s_;        \
  } while (0)

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Common {
  const void* X;
  const void* W;
  const int64_t* labels;
  int64_t N, H, V, ignore_index;
  float smoothing;
  float z_loss;
  float* row_loss;
  int skip_ignored;
  float grad_filter;
  flce_dtype dtype;
  flce_reduction reduction;
  void* ws;
  size_t ws_bytes;
  int32_t* err_word;
  cudaStream_t st;
  // vocabulary-parallel shards: W holds rows [vocab_offset, vocab_offset + V)
  // of a vocabulary of vocab_total; the backward then returns an fp32 partial dX
  int64_t vocab_offset = 0;
  int64_t vocab_total = 0;
  bool dx_partial_f32 = false;
  Tuning tun{};
};

flce_status validate_common(const Common& c, int mode, Plan* pl) {
  if (!shape_ok(c.N, c.H, c.V)) return FLCE_ERR_ARG;
  if (c.dtype != FLCE_BF16 && c.dtype != FLCE_FP32) return FLCE_ERR_ARG;
  if (c.reduction != FLCE_MEAN && c.reduction != FLCE_SUM) return FLCE_ERR_ARG;
  if (!(c.smoothing >= 0.f && c.smoothing < 1.f)) return FLCE_ERR_ARG;
  if (!(c.z_loss >= 0.f && c.z_loss < 1e30f)) return FLCE_ERR_ARG;
  if (!(c.grad_filter >= 0.f && c.grad_filter < 1.f)) return FLCE_ERR_ARG;
  if (c.row_loss && !aligned(c.row_loss, 4)) return FLCE_ERR_ARG;
  if (!c.err_word) return FLCE_ERR_ARG;
  if (c.N > 0) {
    if (!c.X || !c.labels) return FLCE_ERR_ARG;
    if (!aligned(c.X, 16) || !aligned(c.labels, 8)) return FLCE_ERR_ARG;
  }
  if (!c.W || !aligned(c.W, 16)) return FLCE_ERR_ARG;
  if (!aligned(c.err_word, 4)) return FLCE_ERR_ARG;
  if (!make_plan(c.N, c.H, c.V, c.dtype, mode, c.tun, pl)) return FLCE_ERR_ARG;
  if (!c.ws || !aligned(c.ws, kAlign)) return FLCE_ERR_WORKSPACE;
  if (c.ws_bytes < pl->total) return FLCE_ERR_WORKSPACE;
#ifdef FLCE_DEBUG
  if (!plan_regions_ok(*pl, c.dtype, mode)) {
    g_last_cuda_error = "debug build: workspace plan regions overlap or overrun";
    return FLCE_ERR_BOUNDS;
  }
#endif
  return FLCE_OK;
}

// Whether a call needs the kernels' optional features compiled in.
bool ext_features(const Common& c) {
  return c.skip_ignored || c.grad_filter > 0.f || c.tun.l2_hints;
}

// Skip lists for SFT-style masking: token blocks of `tile_rows(pair)` rows with
// at least one label other than ignore_index.
struct SkipLists {
  const int* flags = nullptr;
  const int* list = nullptr;
  const int* count = nullptr;
  int block_rows = 1;
};

flce_status build_skip_lists(const Common& c, const Plan& pl, bool pair, SkipLists* out) {
  *out = SkipLists{};
  if (!c.skip_ignored || c.N == 0) return FLCE_OK;
  int* base = reinterpret_cast<int*>(static_cast<uint8_t*>(c.ws) + pl.off_blocks);
  const int rows = tile_rows(pair);
  const int nb = (int)ceil_div(c.N, rows);
  active_blocks_kernel<<<1, MERGE_THREADS, 0, c.st>>>(c.labels, (int)c.N, c.ignore_index, rows,
                                                       nb, base, base + pl.n_blocks128,
                                                       base + 2 * pl.n_blocks128);
  ++g_launches;
  FLCE_CUDA(cudaGetLastError());
  out->flags = base;
  out->list = base + pl.n_blocks128;
  out->count = base + 2 * pl.n_blocks128;
  out->block_rows = rows;
  return FLCE_OK;
}

// fp32 inputs: one rounding to bf16 into the workspace.
flce_status cast_inputs(const Common& c, const Plan& pl, int sms, const void** Xb,
                        const void** Wb) {
  if (c.dtype == FLCE_BF16) {
    *Xb = c.X;
    *Wb = c.W;
    return FLCE_OK;
  }
  uint8_t* ws = static_cast<uint8_t*>(c.ws);
  void* xo = ws + pl.off_xcast;
  void* wo = ws + pl.off_wcast;
  const size_t nx4 = (size_t)c.N * c.H / 4, nw4 = (size_t)c.V * c.H / 4;
  if (nx4) {
    cast_f32_bf16_kernel<<<convert_blocks(nx4, sms), CONVERT_THREADS, 0, c.st>>>(
        static_cast<const float4*>(c.X), static_cast<uint2*>(xo), nx4);
    ++g_launches;
    FLCE_CUDA(cudaGetLastError());
  }
  cast_f32_bf16_kernel<<<convert_blocks(nw4, sms), CONVERT_THREADS, 0, c.st>>>(
      static_cast<const float4*>(c.W), static_cast<uint2*>(wo), nw4);
  ++g_launches;
  FLCE_CUDA(cudaGetLastError());
  *Xb = xo;
  *Wb = wo;
  return FLCE_OK;
}

flce_status run_forward(const Common& c, const Plan& pl, int dev, int sms, const void* Xb,
                        const void* Wb, float* loss, float* lse, int32_t* valid_count,
                        float4* shard_out = nullptr) {
  uint8_t* ws = static_cast<uint8_t*>(c.ws);
  double* block_loss = reinterpret_cast<double*>(ws + pl.off_block_loss);
  int* block_valid = reinterpret_cast<int*>(ws + pl.off_block_valid);
  if (c.N > 0) {
    const bool pair = c.tun.pair;
    SkipLists sk;
    FLCE_TRY(build_skip_lists(c, pl, pair, &sk));
    GemmParams p{};
    p.m_size = (int)c.N;
    p.n_size = (int)c.V;
    p.k_size = (int)c.H;
    p.m_blocks = (int)ceil_div(c.N, tile_rows(pair));
    p.n_blocks = pl.v_tiles;
    p.group_len = pl.group_len;
    p.n_groups = pl.n_groups;
    p.num_units = p.m_blocks * pl.n_groups;
    p.m_fastest = 1;
    p.m_band = x_band(c.N, c.H, p.m_blocks);
    p.labels = c.labels;
    p.ignore_index = c.ignore_index;
    p.vocab = (int)c.vocab_total;
    p.col_base = (int)c.vocab_offset;
    p.col_limit = (int)c.V;
    p.smoothing = c.smoothing;
    p.partials = reinterpret_cast<float4*>(ws + pl.off_partials);
    p.m_pad = pl.m_pad;
    p.l2_keep_b = 0;
    p.l2_keep_frac = l2_keep_fraction(c.tun, (double)c.N * c.H * 2);
    p.row_list = sk.list;
    p.row_count = sk.count;
    p.list_cap = pl.n_blocks128;
    p.err_word = c.err_word;
    p.timeout_ns = kTimeoutNs;
    const bool ext = ext_features(c);
    const Walk walk = pick_walk(c.tun, pair, ext, p);
    CUtensorMap tmX, tmW;
    FLCE_TRY(map_kmajor(&tmX, Xb, c.H, c.N, c.H, a_box_rows(walk)));
    FLCE_TRY(map_kmajor(&tmW, Wb, c.H, c.V, c.H, b_box_rows(pair, walk)));
    FLCE_TRY((launch_tile<Epi::kLse, false, false>(pair, ext, walk, dev, sms, tmX, tmW, tmX, p,
                                                  c.st, 0)));
    if (shard_out) {
      // vocabulary shard: one merged partial per row, no loss yet
      shard_partial_kernel<<<pl.merge_blocks, MERGE_THREADS, 0, c.st>>>(
          p.partials, pl.n_groups, pl.m_pad, (int)c.N, shard_out);
      ++g_launches;
      FLCE_CUDA(cudaGetLastError());
      return FLCE_OK;
    }
    lse_merge_kernel<<<pl.merge_blocks, MERGE_THREADS, 0, c.st>>>(
        p.partials, pl.n_groups, pl.m_pad, (int)c.N, (int)c.V, c.labels, c.ignore_index,
        c.smoothing, c.z_loss, lse, c.row_loss, block_loss, block_valid, c.err_word, sk.flags,
        sk.block_rows);
    ++g_launches;
    FLCE_CUDA(cudaGetLastError());
  }
  loss_finalize_kernel<<<1, MERGE_THREADS, 0, c.st>>>(block_loss, block_valid,
                                                       c.N > 0 ? pl.merge_blocks : 0,
                                                       c.reduction == FLCE_SUM, loss, valid_count);
  ++g_launches;
  FLCE_CUDA(cudaGetLastError());
  return FLCE_OK;
}

flce_status run_backward(const Common& c, const Plan& pl, int dev, int sms, const void* Xb,
                         const void* Wb, const float* lse, const int32_t* valid_count,
                         const float* grad_loss, void* dX, float* dW, int accumulate) {
  uint8_t* ws = static_cast<uint8_t*>(c.ws);
  float* scale = reinterpret_cast<float*>(ws + pl.off_scalars);
  grad_scale_kernel<<<1, 1, 0, c.st>>>(valid_count, grad_loss, c.reduction == FLCE_SUM, scale);
  ++g_launches;
  FLCE_CUDA(cudaGetLastError());
  if (c.N == 0) {
    if (!accumulate) FLCE_CUDA(cudaMemsetAsync(dW, 0, (size_t)c.V * c.H * 4, c.st));
    return FLCE_OK;
  }
  const int64_t N = c.N, H = c.H, V = c.V, Cv = pl.chunk;
  void* dz = ws + pl.off_dz;
  float* dx_acc = (c.dtype == FLCE_BF16 && !c.dx_partial_f32)
                      ? reinterpret_cast<float*>(ws + pl.off_dxacc)
                      : static_cast<float*>(dX);
  const auto* Wb16 = static_cast<const uint16_t*>(Wb);

  // X as the K-major A operand of the dZ recompute: 128-row boxes (pairs, the
  // merged launches) or 64-row boxes (QUAD walks)
  CUtensorMap tmX_k, tmX_k64, tmX_mn, tmDxAcc;
  FLCE_TRY(map_kmajor(&tmX_k, Xb, H, N, H, BM));
  FLCE_TRY(map_kmajor(&tmX_k64, Xb, H, N, H, 64));
  FLCE_TRY(map_mnmajor(&tmX_mn, Xb, H, N, H));
  FLCE_TRY(map_f32_out(&tmDxAcc, dx_acc, H, N, H));

  const bool pair = c.tun.pair;
  const bool ext = ext_features(c);
  const int m_blocks_tok = (int)ceil_div(N, tile_rows(pair));
  SkipLists sk;
  FLCE_TRY(build_skip_lists(c, pl, pair, &sk));
  if (sk.flags) {
    zero_skipped_rows_kernel<<<2 * sms, 256, 0, c.st>>>(sk.flags, sk.block_rows, dx_acc, (int)N,
                                                         (int)H);
    ++g_launches;
    FLCE_CUDA(cudaGetLastError());
  }
  const int h_blocks = (int)ceil_div(H, BN);
  // gradient filtering: keep masks, one k-loop of a tile must fit the smem keep bytes
  const bool filt = c.grad_filter > 0.f;
  if (filt && (ceil_div(Cv, BK) > FILTER_MAX_KB || ceil_div(N, BK) > FILTER_MAX_KB))
    return FLCE_ERR_UNSUPPORTED;
  uint8_t* mask_x = ws + pl.off_mask_x;
  uint8_t* mask_w = ws + pl.off_mask_w;
  const size_t mask_x_bytes = (size_t)ceil_div(N, BM) * pl.mask_x_ld;
  const size_t mask_w_bytes = (size_t)ceil_div(Cv, BM) * pl.mask_w_ld;
  // K3 parameters: recompute Z[:, v0:v0+w] and write dZ (bf16) into a chunk buffer.
  auto dz_params = [&](int64_t v0, int64_t w) {
    GemmParams p3{};
    p3.m_size = (int)N;
    p3.n_size = (int)w;
    p3.k_size = (int)H;
    p3.m_blocks = m_blocks_tok;
    p3.n_blocks = (int)ceil_div(w, BN);
    p3.group_len = 1;
    p3.n_groups = p3.n_blocks;
    p3.num_units = p3.m_blocks * p3.n_groups;
    p3.m_fastest = 1;
    p3.m_band = x_band(N, H, p3.m_blocks);
    p3.labels = c.labels;
    p3.ignore_index = c.ignore_index;
    p3.vocab = (int)c.vocab_total;
    p3.col_base = (int)(c.vocab_offset + v0);
    p3.col_limit = (int)w;
    p3.smoothing = c.smoothing;
    p3.z_loss = c.z_loss;
    p3.row_list = sk.list;
    p3.row_count = sk.count;
    p3.list_cap = pl.n_blocks128;
    if (filt) {
      p3.mask_x_out = mask_x;
      p3.mask_w_out = mask_w;
      p3.mask_x_ld = pl.mask_x_ld;
      p3.mask_w_ld = pl.mask_w_ld;
      p3.mask_tile = tile_rows(pair);
      p3.filter_thr = c.grad_filter;
      p3.mask_x_bytes = (long long)mask_x_bytes;
      p3.mask_w_bytes = (long long)mask_w_bytes;
    }
    p3.lse = lse;
    p3.scale = scale;
    p3.l2_keep_b = 0;  // X is reused by every wave; the W tile is shared within one
    p3.l2_keep_frac = l2_keep_fraction(c.tun, (double)N * H * 2);
    p3.err_word = c.err_word;
    p3.timeout_ns = kTimeoutNs;
    return p3;
  };
  // One merged launch for chunk c: the dW(c) and dX(c) tiles, reading dZ(c)
  // from `cur`, and -- when `next_buf` is set and a chunk c+1 exists -- the dZ
  // recompute of chunk c+1 into `next_buf`, all from one tile list.
  int* counters = reinterpret_cast<int*>(ws + pl.off_counters);
  auto merged_launch = [&](int ci, const void* cur, void* next_buf) -> flce_status {
    const int64_t v0 = (int64_t)ci * Cv;
    const int64_t w = std::min(Cv, V - v0);
    const bool next = next_buf != nullptr && ci + 1 < pl.n_chunks;
    const int64_t v1 = v0 + Cv;
    const int64_t w1 = next ? std::min(Cv, V - v1) : 0;
    const void* Wc = Wb16 + v0 * H;
    FusedMaps fm;
    FLCE_TRY(map_mnmajor(&fm.a[kFusedDw], cur, w, N, Cv));
    fm.b[kFusedDw] = tmX_mn;
    FLCE_TRY(map_f32_out(&fm.out[kFusedDw], dW + v0 * H, H, w, H));
    FLCE_TRY(map_kmajor(&fm.a[kFusedDx], cur, w, N, Cv, BM));
    FLCE_TRY(map_mnmajor(&fm.b[kFusedDx], Wc, H, w, H));
    fm.out[kFusedDx] = tmDxAcc;
    fm.a[kFusedDz] = tmX_k;
    if (next) {
      FLCE_TRY(map_kmajor(&fm.b[kFusedDz], Wb16 + v1 * H, H, w1, H, b_box_rows(pair)));
      FLCE_TRY(map_dz_store(&fm.out[kFusedDz], next_buf, w1, N, Cv));
    } else {  // no dZ tiles: valid maps for the prefetch only
      fm.b[kFusedDz] = tmX_k;
      fm.out[kFusedDz] = tmX_k;
    }
    FusedSeg segs[3];
    int n_seg = 0;
    auto seg = [&](int kind, int m_size, int n_size, int k_size, int m_fastest, int m_band,
                   int reduce_add) {
      FusedSeg g{};
      g.kind = kind;
      g.m_size = m_size;
      g.n_size = n_size;
      g.k_size = k_size;
      g.m_blocks = (int)ceil_div(m_size, 2 * BM);
      g.n_blocks = (int)ceil_div(n_size, BN);
      g.num_tiles = g.m_blocks * g.n_blocks;
      g.m_fastest = m_fastest;
      g.m_band = m_band;
      g.reduce_add = reduce_add;
      segs[n_seg++] = g;
    };
    // dX first among equals: its tiles hold a whole row block of dX_acc
    seg(kFusedDx, (int)N, (int)H, (int)w, 0, 0, ci > 0 ? 1 : 0);
    seg(kFusedDw, (int)w, (int)H, (int)N, 0, 0, accumulate ? 1 : 0);
    if (next) seg(kFusedDz, (int)N, (int)w1, (int)H, 1, x_band(N, H, m_blocks_tok), 0);
    // longest k-loop first, so the list ends on the shortest tiles
    std::stable_sort(segs, segs + n_seg, [](const FusedSeg& a, const FusedSeg& b) {
      return ceil_div(a.k_size, BK) > ceil_div(b.k_size, BK);
    });
    FusedParams fp{};
    int first = 0;
    for (int i = 0; i < n_seg; ++i) {
      segs[i].first = first;
      first += segs[i].num_tiles;
      fp.seg[i] = segs[i];
    }
    fp.n_seg = n_seg;
    fp.total_tiles = first;
    fp.tile_counter = counters + ci;
    fp.labels = c.labels;
    fp.ignore_index = c.ignore_index;
    fp.vocab = (int)c.vocab_total;
    fp.col_base = (int)(c.vocab_offset + v1);
    fp.col_limit = (int)w1;
    fp.smoothing = c.smoothing;
    fp.z_loss = c.z_loss;
    fp.lse = lse;
    fp.scale = scale;
    fp.err_word = c.err_word;
    fp.timeout_ns = kTimeoutNs;
    return launch_fused(dev, sms, fm, fp, c.st);
  };
  // K3 alone for chunk ci: recompute Z[:, v0:v0+w] and write dZ into `buf`.
  auto dz_launch = [&](int ci, void* buf, bool ext_kernel) -> flce_status {
    const int64_t v0 = (int64_t)ci * Cv;
    const int64_t w = std::min(Cv, V - v0);
    const GemmParams p3 = dz_params(v0, w);
    const Walk w3 = pick_walk(c.tun, pair, ext_kernel, p3);
    CUtensorMap tmWc_k, tmDzSt;
    FLCE_TRY(map_kmajor(&tmWc_k, Wb16 + v0 * H, H, w, H, b_box_rows(pair, w3)));
    FLCE_TRY(map_dz_store(&tmDzSt, buf, w, N, Cv));
    return launch_tile<Epi::kDz, false, false>(pair, ext_kernel, w3, dev, sms,
                                               w3.quad ? tmX_k64 : tmX_k, tmWc_k, tmDzSt, p3,
                                               c.st, 1);
  };
  if (pair && !ext && pl.dz_bufs == 2) {
    // Merged backward: dZ of chunk 0 alone, then per chunk c one launch of
    // dW(c), dX(c) and dZ(c+1), the dZ buffers taken in turn.
    FLCE_CUDA(cudaMemsetAsync(counters, 0, (size_t)pl.n_chunks * sizeof(int), c.st));
    void* dz_buf[2] = {ws + pl.off_dz, ws + pl.off_dz2};
    FLCE_TRY(dz_launch(0, dz_buf[0], false));
    for (int ci = 0; ci < pl.n_chunks; ++ci)
      FLCE_TRY(merged_launch(ci, dz_buf[ci & 1], dz_buf[(ci + 1) & 1]));
  } else if (pair && !ext && pl.counters) {
    // dW(c) and dX(c) merged: per chunk the dZ recompute alone, then one
    // launch of both GEMMs that read it (one dZ buffer).
    FLCE_CUDA(cudaMemsetAsync(counters, 0, (size_t)pl.n_chunks * sizeof(int), c.st));
    for (int ci = 0; ci < pl.n_chunks; ++ci) {
      FLCE_TRY(dz_launch(ci, dz, false));
      FLCE_TRY(merged_launch(ci, dz, nullptr));
    }
  } else {
    for (int ci = 0; ci < pl.n_chunks; ++ci) {
      const int64_t v0 = (int64_t)ci * Cv;
      const int64_t w = std::min(Cv, V - v0);
      if (filt) {
        FLCE_CUDA(cudaMemsetAsync(mask_x, 0, mask_x_bytes, c.st));
        FLCE_CUDA(cudaMemsetAsync(mask_w, 0, mask_w_bytes, c.st));
      }
      const void* Wc = Wb16 + v0 * H;
      const GemmParams p3 = dz_params(v0, w);
      const Walk w3 = pick_walk(c.tun, pair, ext, p3);
      CUtensorMap tmWc_k, tmWc_mn, tmDzSt, tmDz_mn, tmDz_k, tmDw;
      FLCE_TRY(map_kmajor(&tmWc_k, Wc, H, w, H, b_box_rows(pair, w3)));
      FLCE_TRY(map_mnmajor(&tmWc_mn, Wc, H, w, H));
      FLCE_TRY(map_dz_store(&tmDzSt, dz, w, N, Cv));
      FLCE_TRY(map_mnmajor(&tmDz_mn, dz, w, N, Cv));
      FLCE_TRY(map_f32_out(&tmDw, dW + v0 * H, H, w, H));

      // K3: recompute Z[:, v0:v0+w] and write dZ (bf16) into the chunk scratch.
      FLCE_TRY((launch_tile<Epi::kDz, false, false>(pair, ext, w3, dev, sms,
                                                    w3.quad ? tmX_k64 : tmX_k, tmWc_k, tmDzSt,
                                                    p3, c.st, 1)));

      // K4: dW[v0:v0+w, :] = dZ_chunk^T X   (K = N tokens)
      GemmParams p4{};
      p4.m_size = (int)w;
      p4.n_size = (int)H;
      p4.k_size = (int)N;
      p4.m_blocks = (int)ceil_div(w, tile_rows(pair));
      p4.n_blocks = h_blocks;
      p4.group_len = 1;
      p4.n_groups = h_blocks;
      p4.num_units = p4.m_blocks * h_blocks;
      p4.m_fastest = 0;
      p4.reduce_add = accumulate ? 1 : 0;
      p4.k_list = sk.list;
      p4.k_count = sk.count;
      p4.k_per_entry = tile_rows(pair) / BK;
      p4.list_cap = pl.n_blocks128;
      if (filt) {
        p4.fmask = mask_w;
        p4.fmask_ld = pl.mask_w_ld;
        p4.fmask_bytes = (long long)mask_w_bytes;
      }
      p4.l2_keep_b = 1;  // X again; the dZ column block is shared within one wave
      p4.l2_keep_frac = l2_keep_fraction(c.tun, (double)N * H * 2);
      p4.err_word = c.err_word;
      p4.timeout_ns = kTimeoutNs;
      FLCE_TRY((launch_tile<Epi::kStore, true, true>(pair, ext, pick_walk(c.tun, pair, ext, p4),
                                                     dev, sms, tmDz_mn, tmX_mn, tmDw, p4, c.st,
                                                     2)));

      // K5: dX_acc (+)= dZ_chunk W[v0:v0+w, :]   (K = w vocabulary columns)
      GemmParams p5{};
      p5.m_size = (int)N;
      p5.n_size = (int)H;
      p5.k_size = (int)w;
      p5.m_blocks = m_blocks_tok;
      p5.n_blocks = h_blocks;
      p5.group_len = 1;
      p5.n_groups = h_blocks;
      p5.num_units = m_blocks_tok * h_blocks;
      p5.m_fastest = 0;
      p5.reduce_add = ci > 0 ? 1 : 0;
      p5.row_list = sk.list;
      p5.row_count = sk.count;
      p5.list_cap = pl.n_blocks128;
      if (filt) {
        p5.fmask = mask_x;
        p5.fmask_ld = pl.mask_x_ld;
        p5.fmask_bytes = (long long)mask_x_bytes;
      }
      p5.l2_keep_b = 1;  // the W chunk; the dZ row block is shared within one wave
      p5.l2_keep_frac = l2_keep_fraction(c.tun, (double)w * H * 2);
      p5.err_word = c.err_word;
      p5.timeout_ns = kTimeoutNs;
      const Walk w5 = pick_walk(c.tun, pair, ext, p5);
      FLCE_TRY(map_kmajor(&tmDz_k, dz, w, N, Cv, a_box_rows(w5)));
      FLCE_TRY((launch_tile<Epi::kStore, false, true>(pair, ext, w5, dev, sms, tmDz_k, tmWc_mn,
                                                      tmDxAcc, p5, c.st, 3)));
    }
  }
  if (c.dtype == FLCE_BF16 && !c.dx_partial_f32) {
    const size_t n4 = (size_t)N * H / 4;
    dx_finalize_bf16_kernel<<<convert_blocks(n4, sms), CONVERT_THREADS, 0, c.st>>>(
        reinterpret_cast<const float4*>(dx_acc), static_cast<uint2*>(dX), n4);
    ++g_launches;
    FLCE_CUDA(cudaGetLastError());
  }
  return FLCE_OK;
}

}  // namespace

// ===========================================================================
// Exported C ABI
// ===========================================================================
extern "C" {

int flce_abi_version(void) { return 106; }

const char* flce_status_string(flce_status s) {
  switch (s) {
    case FLCE_OK: return "FLCE_OK";
    case FLCE_ERR_ARG: return "FLCE_ERR_ARG: invalid argument";
    case FLCE_ERR_UNSUPPORTED: return "FLCE_ERR_UNSUPPORTED: device or size not supported";
    case FLCE_ERR_WORKSPACE: return "FLCE_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case FLCE_ERR_LABEL: return "FLCE_ERR_LABEL: label outside [0, V) and not ignore_index";
    case FLCE_ERR_TIMEOUT: return "FLCE_ERR_TIMEOUT: a bounded device wait expired";
    case FLCE_ERR_CUDA: return "FLCE_ERR_CUDA: CUDA call failed";
    case FLCE_ERR_BOUNDS: return "FLCE_ERR_BOUNDS: an index check of the debug build failed";
  }
  return "unknown flce_status";
}

const char* flce_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

int flce_last_launch_count(void) { return g_launches; }

int flce_debug_last_multicast_launches(void) { return g_quad_launches; }

flce_status flce_profile_enable(int on) {
  g_prof_on = on != 0;
  return FLCE_OK;
}

flce_status flce_profile_read(int kind, double* total_ms, int* launches) {
  if (kind < 0 || kind >= kProfKinds || !total_ms || !launches) return FLCE_ERR_ARG;
  for (const ProfRec& r : g_prof_pending) {
    FLCE_CUDA(cudaEventSynchronize(r.stop));
    float ms = 0.f;
    FLCE_CUDA(cudaEventElapsedTime(&ms, r.start, r.stop));
    g_prof_ms[r.kind] += ms;
    g_prof_n[r.kind] += 1;
    g_prof_pool.push_back(r.start);
    g_prof_pool.push_back(r.stop);
  }
  g_prof_pending.clear();
  *total_ms = g_prof_ms[kind];
  *launches = g_prof_n[kind];
  return FLCE_OK;
}

void flce_profile_reset(void) {
  for (const ProfRec& r : g_prof_pending) {
    g_prof_pool.push_back(r.start);
    g_prof_pool.push_back(r.stop);
  }
  g_prof_pending.clear();
  for (int k = 0; k < kProfKinds; ++k) {
    g_prof_ms[k] = 0.0;
    g_prof_n[k] = 0;
  }
}

flce_status flce_set_l2_hints(int on) {
  g_l2_hints.store(on != 0 ? 1 : 0);
  return FLCE_OK;
}

flce_status flce_set_cta_pair(int on) {
  g_cta_pair.store(on != 0 ? 1 : 0);
  return FLCE_OK;
}

int flce_cta_pair(void) { return g_cta_pair.load(); }

flce_status flce_set_cluster_multicast(int on) {
  g_cluster_mcast.store(on != 0 ? 1 : 0);
  return FLCE_OK;
}

int flce_cluster_multicast(void) { return g_cluster_mcast.load(); }

flce_status flce_set_backward_merge(int on) {
  if (on < 0 || on > 2) return FLCE_ERR_ARG;
  g_bwd_merge.store(on);
  return FLCE_OK;
}

int flce_backward_merge(void) { return g_bwd_merge.load(); }

flce_status flce_set_vocab_chunk(int64_t cols) {
  if (cols < 0) return FLCE_ERR_ARG;
  g_vocab_chunk.store(cols);
  return FLCE_OK;
}

int64_t flce_vocab_chunk(int64_t N, int64_t H, int64_t V) {
  if (N < 0 || H <= 0 || V <= 0) return 0;
  return auto_chunk(N, H, V, default_tuning());
}

size_t flce_workspace_size(int64_t N, int64_t H, int64_t V, flce_dtype dtype, int mode) {
  Plan pl;
  if (!make_plan(N, H, V, dtype, mode, default_tuning(), &pl)) return 0;
  return pl.total;
}

void flce_options_init(flce_options* opt) {
  if (!opt) return;
  opt->struct_size = sizeof(flce_options);
  opt->ignore_index = -100;
  opt->smoothing = 0.f;
  opt->z_loss = 0.f;
  opt->reduction = FLCE_MEAN;
  opt->row_loss = nullptr;
  opt->skip_ignored_blocks = 0;
  opt->grad_filter = 0.f;
  opt->cta_pair = -1;
  opt->backward_merge = -1;
  opt->l2_hints = -1;
  opt->vocab_chunk = -1;
  opt->cluster_multicast = -1;
}

}  // extern "C"

namespace {

// Size of the options struct of ABI 1.05, before the launch settings.
constexpr size_t kOptionsV105Size = offsetof(flce_options, cta_pair);

bool options_ok(const flce_options* opt) {
  if (!opt) return false;
  if (opt->struct_size == kOptionsV105Size) return true;
  if (opt->struct_size != sizeof(flce_options)) return false;
  auto tri = [](int v) { return v >= -1 && v <= 1; };
  return tri(opt->cta_pair) && opt->backward_merge >= -1 && opt->backward_merge <= 2 &&
         tri(opt->l2_hints) && tri(opt->cluster_multicast) &&
         opt->vocab_chunk >= -1;
}

// The launch settings of a call: each options field that is not -1 overrides
// the process-wide default (a 1.05-sized struct has no such fields).
Tuning resolve_tuning(const flce_options* opt) {
  Tuning t = default_tuning();
  if (!opt || opt->struct_size < sizeof(flce_options)) return t;
  if (opt->cta_pair >= 0) t.pair = opt->cta_pair != 0;
  if (opt->backward_merge >= 0) t.merge = opt->backward_merge;
  if (opt->l2_hints >= 0) t.l2_hints = opt->l2_hints != 0;
  if (opt->vocab_chunk >= 0) t.chunk_set = opt->vocab_chunk;
  if (opt->cluster_multicast >= 0) t.mcast = opt->cluster_multicast != 0;
  return t;
}

Common make_common(const void* X, const void* W, const int64_t* labels, int64_t N, int64_t H,
                   int64_t V, flce_dtype dtype, const flce_options* o, void* ws, size_t ws_bytes,
                   int32_t* err_word, void* stream) {
  return Common{X,
                W,
                labels,
                N,
                H,
                V,
                o->ignore_index,
                o->smoothing,
                o->z_loss,
                o->row_loss,
                o->skip_ignored_blocks,
                o->grad_filter,
                dtype,
                o->reduction,
                ws,
                ws_bytes,
                err_word,
                static_cast<cudaStream_t>(stream),
                0,
                V,
                false,
                resolve_tuning(o)};
}

flce_options defaults(int64_t ignore_index, float smoothing, flce_reduction reduction) {
  flce_options o;
  flce_options_init(&o);
  o.ignore_index = ignore_index;
  o.smoothing = smoothing;
  o.reduction = reduction;
  return o;
}

}  // namespace

extern "C" {

size_t flce_workspace_size_ex(int64_t N, int64_t H, int64_t V, flce_dtype dtype, int mode,
                              const flce_options* opt) {
  if (opt && !options_ok(opt)) return 0;
  Plan pl;
  if (!make_plan(N, H, V, dtype, mode, resolve_tuning(opt), &pl)) return 0;
  return pl.total;
}

int64_t flce_vocab_chunk_ex(int64_t N, int64_t H, int64_t V, const flce_options* opt) {
  if (N < 0 || H <= 0 || V <= 0) return 0;
  if (opt && !options_ok(opt)) return 0;
  return auto_chunk(N, H, V, resolve_tuning(opt));
}

flce_status flce_forward_ex(const void* X, const void* W, const int64_t* labels, int64_t N,
                            int64_t H, int64_t V, flce_dtype dtype, const flce_options* opt,
                            float* loss, float* lse, int32_t* valid_count, void* workspace,
                            size_t ws_bytes, int32_t* err_word, void* stream) {
  g_launches = 0;
  g_quad_launches = 0;
  if (!options_ok(opt)) return FLCE_ERR_ARG;
  Common c = make_common(X, W, labels, N, H, V, dtype, opt, workspace, ws_bytes, err_word, stream);
  Plan pl;
  FLCE_TRY(validate_common(c, FLCE_MODE_FWD, &pl));
  if (!loss || !valid_count || (N > 0 && !lse)) return FLCE_ERR_ARG;
  int dev, sms;
  FLCE_TRY(device_check(&dev, &sms));
  const void *Xb, *Wb;
  FLCE_TRY(cast_inputs(c, pl, sms, &Xb, &Wb));
  return run_forward(c, pl, dev, sms, Xb, Wb, loss, lse, valid_count);
}

flce_status flce_backward_ex(const void* X, const void* W, const int64_t* labels, int64_t N,
                             int64_t H, int64_t V, flce_dtype dtype, const flce_options* opt,
                             const float* lse, const int32_t* valid_count,
                             const float* grad_loss, void* dX, float* dW, int accumulate_dW,
                             void* workspace, size_t ws_bytes, int32_t* err_word, void* stream) {
  g_launches = 0;
  g_quad_launches = 0;
  if (!options_ok(opt)) return FLCE_ERR_ARG;
  Common c = make_common(X, W, labels, N, H, V, dtype, opt, workspace, ws_bytes, err_word, stream);
  Plan pl;
  FLCE_TRY(validate_common(c, FLCE_MODE_BWD, &pl));
  if (!valid_count || !dW || !aligned(dW, 16)) return FLCE_ERR_ARG;
  if (N > 0 && (!lse || !dX || !aligned(dX, 16))) return FLCE_ERR_ARG;
  int dev, sms;
  FLCE_TRY(device_check(&dev, &sms));
  const void *Xb, *Wb;
  FLCE_TRY(cast_inputs(c, pl, sms, &Xb, &Wb));
  return run_backward(c, pl, dev, sms, Xb, Wb, lse, valid_count, grad_loss, dX, dW,
                      accumulate_dW);
}

flce_status flce_fwd_bwd_ex(const void* X, const void* W, const int64_t* labels, int64_t N,
                            int64_t H, int64_t V, flce_dtype dtype, const flce_options* opt,
                            const float* grad_loss, float* loss, float* lse,
                            int32_t* valid_count, void* dX, float* dW, int accumulate_dW,
                            void* workspace, size_t ws_bytes, int32_t* err_word, void* stream) {
  g_launches = 0;
  g_quad_launches = 0;
  if (!options_ok(opt)) return FLCE_ERR_ARG;
  Common c = make_common(X, W, labels, N, H, V, dtype, opt, workspace, ws_bytes, err_word, stream);
  Plan pl;
  FLCE_TRY(validate_common(c, FLCE_MODE_FWD_BWD, &pl));
  if (!loss || !valid_count || !dW || !aligned(dW, 16)) return FLCE_ERR_ARG;
  if (N > 0 && (!lse || !dX || !aligned(dX, 16))) return FLCE_ERR_ARG;
  int dev, sms;
  FLCE_TRY(device_check(&dev, &sms));
  const void *Xb, *Wb;
  FLCE_TRY(cast_inputs(c, pl, sms, &Xb, &Wb));
  FLCE_TRY(run_forward(c, pl, dev, sms, Xb, Wb, loss, lse, valid_count));
  return run_backward(c, pl, dev, sms, Xb, Wb, lse, valid_count, grad_loss, dX, dW,
                      accumulate_dW);
}

flce_status flce_forward(const void* X, const void* W, const int64_t* labels, int64_t N,
                         int64_t H, int64_t V, int64_t ignore_index, float smoothing,
                         flce_dtype dtype, flce_reduction reduction, float* loss, float* lse,
                         int32_t* valid_count, void* workspace, size_t ws_bytes,
                         int32_t* err_word, void* stream) {
  const flce_options o = defaults(ignore_index, smoothing, reduction);
  return flce_forward_ex(X, W, labels, N, H, V, dtype, &o, loss, lse, valid_count, workspace,
                         ws_bytes, err_word, stream);
}

flce_status flce_backward(const void* X, const void* W, const int64_t* labels, int64_t N,
                          int64_t H, int64_t V, int64_t ignore_index, float smoothing,
                          flce_dtype dtype, flce_reduction reduction, const float* lse,
                          const int32_t* valid_count, const float* grad_loss, void* dX,
                          float* dW, int accumulate_dW, void* workspace, size_t ws_bytes,
                          int32_t* err_word, void* stream) {
  const flce_options o = defaults(ignore_index, smoothing, reduction);
  return flce_backward_ex(X, W, labels, N, H, V, dtype, &o, lse, valid_count, grad_loss, dX, dW,
                          accumulate_dW, workspace, ws_bytes, err_word, stream);
}

flce_status flce_fwd_bwd(const void* X, const void* W, const int64_t* labels, int64_t N,
                         int64_t H, int64_t V, int64_t ignore_index, float smoothing,
                         flce_dtype dtype, flce_reduction reduction, const float* grad_loss,
                         float* loss, float* lse, int32_t* valid_count, void* dX, float* dW,
                         int accumulate_dW, void* workspace, size_t ws_bytes, int32_t* err_word,
                         void* stream) {
  const flce_options o = defaults(ignore_index, smoothing, reduction);
  return flce_fwd_bwd_ex(X, W, labels, N, H, V, dtype, &o, grad_loss, loss, lse, valid_count, dX,
                         dW, accumulate_dW, workspace, ws_bytes, err_word, stream);
}

// ---------------------------------------------------------------------------
// Vocabulary-parallel shards
// ---------------------------------------------------------------------------
}  // extern "C"

namespace {

flce_status shard_common(const void* X, const void* W_shard, const int64_t* labels, int64_t N,
                         int64_t H, int64_t V_shard, int64_t vocab_offset, int64_t vocab_total,
                         flce_dtype dtype, const flce_options* opt, void* ws, size_t ws_bytes,
                         int32_t* err_word, void* stream, Common* out) {
  if (!options_ok(opt)) return FLCE_ERR_ARG;
  if (opt->skip_ignored_blocks || opt->row_loss) return FLCE_ERR_ARG;
  if (vocab_offset < 0 || V_shard <= 0 || vocab_total < vocab_offset + V_shard ||
      vocab_total > (int64_t)INT32_MAX - 1024)
    return FLCE_ERR_ARG;
  *out = make_common(X, W_shard, labels, N, H, V_shard, dtype, opt, ws, ws_bytes, err_word,
                     stream);
  out->vocab_offset = vocab_offset;
  out->vocab_total = vocab_total;
  return FLCE_OK;
}

}  // namespace

extern "C" {

flce_status flce_forward_vocab_shard(const void* X, const void* W_shard, const int64_t* labels,
                                     int64_t N, int64_t H, int64_t V_shard, int64_t vocab_offset,
                                     int64_t vocab_total, flce_dtype dtype,
                                     const flce_options* opt, float* partials, void* workspace,
                                     size_t ws_bytes, int32_t* err_word, void* stream) {
  g_launches = 0;
  g_quad_launches = 0;
  Common c;
  FLCE_TRY(shard_common(X, W_shard, labels, N, H, V_shard, vocab_offset, vocab_total, dtype, opt,
                        workspace, ws_bytes, err_word, stream, &c));
  Plan pl;
  FLCE_TRY(validate_common(c, FLCE_MODE_FWD, &pl));
  if (N > 0 && (!partials || !aligned(partials, 16))) return FLCE_ERR_ARG;
  if (N == 0) return FLCE_OK;
  int dev, sms;
  FLCE_TRY(device_check(&dev, &sms));
  const void *Xb, *Wb;
  FLCE_TRY(cast_inputs(c, pl, sms, &Xb, &Wb));
  return run_forward(c, pl, dev, sms, Xb, Wb, nullptr, nullptr, nullptr,
                     reinterpret_cast<float4*>(partials));
}

size_t flce_combine_workspace_size(int64_t N) {
  if (N < 0) return 0;
  const size_t nb = (size_t)merge_block_count(N);
  return align_up(nb * sizeof(double), kAlign) + align_up(nb * sizeof(int), kAlign);
}

flce_status flce_combine_vocab_shards(const float* partials, int n_shards, int64_t N,
                                      const int64_t* labels, int64_t vocab_total,
                                      const flce_options* opt, float* loss, float* lse,
                                      int32_t* valid_count, void* workspace, size_t ws_bytes,
                                      int32_t* err_word, void* stream) {
  g_launches = 0;
  g_quad_launches = 0;
  if (!options_ok(opt) || opt->skip_ignored_blocks) return FLCE_ERR_ARG;
  if (n_shards <= 0 || N < 0 || N > (int64_t)INT32_MAX - 1024 || vocab_total <= 0 ||
      vocab_total > (int64_t)INT32_MAX - 1024)
    return FLCE_ERR_ARG;
  if (opt->reduction != FLCE_MEAN && opt->reduction != FLCE_SUM) return FLCE_ERR_ARG;
  if (!(opt->smoothing >= 0.f && opt->smoothing < 1.f) || !(opt->z_loss >= 0.f))
    return FLCE_ERR_ARG;
  if (!loss || !valid_count || !err_word) return FLCE_ERR_ARG;
  if (N > 0 && (!partials || !labels || !lse || !aligned(partials, 16))) return FLCE_ERR_ARG;
  if (opt->row_loss && !aligned(opt->row_loss, 4)) return FLCE_ERR_ARG;
  if (!workspace || !aligned(workspace, kAlign) || ws_bytes < flce_combine_workspace_size(N))
    return FLCE_ERR_WORKSPACE;
  int dev, sms;
  FLCE_TRY(device_check(&dev, &sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int nb = (int)merge_block_count(N);
  double* block_loss = static_cast<double*>(workspace);
  int* block_valid = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) +
                                            align_up(nb * sizeof(double), kAlign));
  if (N > 0) {
    // the LSE-combine of the shards is the merge of n_shards partials per row
    lse_merge_kernel<<<nb, MERGE_THREADS, 0, st>>>(
        reinterpret_cast<const float4*>(partials), n_shards, (int)N, (int)N, (int)vocab_total,
        labels, opt->ignore_index, opt->smoothing, opt->z_loss, lse, opt->row_loss, block_loss,
        block_valid, err_word, nullptr, 1);
    ++g_launches;
    FLCE_CUDA(cudaGetLastError());
  }
  loss_finalize_kernel<<<1, MERGE_THREADS, 0, st>>>(block_loss, block_valid, N > 0 ? nb : 0,
                                                     opt->reduction == FLCE_SUM, loss,
                                                     valid_count);
  ++g_launches;
  FLCE_CUDA(cudaGetLastError());
  return FLCE_OK;
}

flce_status flce_backward_vocab_shard(const void* X, const void* W_shard, const int64_t* labels,
                                      int64_t N, int64_t H, int64_t V_shard,
                                      int64_t vocab_offset, int64_t vocab_total,
                                      flce_dtype dtype, const flce_options* opt,
                                      const float* lse, const int32_t* valid_count,
                                      const float* grad_loss, float* dX_partial,
                                      float* dW_shard, int accumulate_dW, void* workspace,
                                      size_t ws_bytes, int32_t* err_word, void* stream) {
  g_launches = 0;
  g_quad_launches = 0;
  Common c;
  FLCE_TRY(shard_common(X, W_shard, labels, N, H, V_shard, vocab_offset, vocab_total, dtype, opt,
                        workspace, ws_bytes, err_word, stream, &c));
  c.dx_partial_f32 = true;
  Plan pl;
  FLCE_TRY(validate_common(c, FLCE_MODE_BWD, &pl));
  if (!valid_count || !dW_shard || !aligned(dW_shard, 16)) return FLCE_ERR_ARG;
  if (N > 0 && (!lse || !dX_partial || !aligned(dX_partial, 16))) return FLCE_ERR_ARG;
  int dev, sms;
  FLCE_TRY(device_check(&dev, &sms));
  const void *Xb, *Wb;
  FLCE_TRY(cast_inputs(c, pl, sms, &Xb, &Wb));
  return run_backward(c, pl, dev, sms, Xb, Wb, lse, valid_count, grad_loss, dX_partial, dW_shard,
                      accumulate_dW);
}

flce_status flce_debug_wait_timeout(int32_t* err_word, uint64_t timeout_ns,
                                    int32_t* waited_us, void* stream) {
  g_launches = 0;
  g_quad_launches = 0;
  if (!err_word || !waited_us || timeout_ns == 0 || timeout_ns > 10000000000ull)
    return FLCE_ERR_ARG;
  int dev, sms;
  FLCE_TRY(device_check(&dev, &sms));
  wait_timeout_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err_word, timeout_ns,
                                                                             waited_us);
  ++g_launches;
  FLCE_CUDA(cudaGetLastError());
  return FLCE_OK;
}

flce_status flce_debug_gemm(const void* A, const void* B, float* D, int64_t M, int64_t Nn,
                            int64_t K, int a_mn, int b_mn, int accumulate, int32_t* err_word,
                            void* stream) {
  g_launches = 0;
  g_quad_launches = 0;
  if (!A || !B || !D || !err_word) return FLCE_ERR_ARG;
  if (M <= 0 || Nn <= 0 || K <= 0 || M > INT32_MAX / 2 || Nn > INT32_MAX / 2 ||
      K > INT32_MAX / 2)
    return FLCE_ERR_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(D, 16)) return FLCE_ERR_ARG;
  // inner extents of every operand must be 16-byte multiples
  if ((a_mn ? M : K) % 8 || (b_mn ? Nn : K) % 8 || Nn % 4) return FLCE_ERR_ARG;
  int dev, sms;
  FLCE_TRY(device_check(&dev, &sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Tuning tun = default_tuning();
  const bool pair = tun.pair;
  GemmParams p{};
  p.m_size = (int)M;
  p.n_size = (int)Nn;
  p.k_size = (int)K;
  p.m_blocks = (int)ceil_div(M, tile_rows(pair));
  p.n_blocks = (int)ceil_div(Nn, BN);
  p.group_len = 1;
  p.n_groups = p.n_blocks;
  p.num_units = p.m_blocks * p.n_blocks;
  p.m_fastest = 0;
  p.reduce_add = accumulate ? 1 : 0;
  p.err_word = err_word;
  p.timeout_ns = kTimeoutNs;
  const Walk w = pick_walk(tun, pair, false, p);
  CUtensorMap ta, tb, td;
  if (a_mn) FLCE_TRY(map_mnmajor(&ta, A, M, K, M));
  else FLCE_TRY(map_kmajor(&ta, A, K, M, K, a_box_rows(w)));
  if (b_mn) FLCE_TRY(map_mnmajor(&tb, B, Nn, K, Nn));
  else FLCE_TRY(map_kmajor(&tb, B, K, Nn, K, b_box_rows(pair, w)));
  FLCE_TRY(map_f32_out(&td, D, Nn, M, Nn));
  if (!a_mn && !b_mn) return launch_tile<Epi::kStore, false, false>(pair, false, w, dev, sms, ta, tb, td, p, st);
  if (!a_mn && b_mn) return launch_tile<Epi::kStore, false, true>(pair, false, w, dev, sms, ta, tb, td, p, st);
  if (a_mn && !b_mn) return launch_tile<Epi::kStore, true, false>(pair, false, w, dev, sms, ta, tb, td, p, st);
  return launch_tile<Epi::kStore, true, true>(pair, false, w, dev, sms, ta, tb, td, p, st);
}

}  // extern "C"
