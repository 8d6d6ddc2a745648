// flce_forward_noalloc: the forward pass for callers that cannot allocate
// device memory and cannot hand the library a workspace.
//
// Who needs it: code that runs inside a host application that owns every
// byte of device memory through its own pool (a serving process or engine
// with a fixed memory budget, where a stray cudaMalloc either fails or
// fragments the pool), code on a path that must not allocate after start-up
// (cudaMalloc can synchronise the device and stall a latency-critical loop),
// and plain C callers that have no allocator at hand or no way to size and
// keep a workspace buffer between calls.  Such a caller still passes its
// inputs and outputs; the only scratch this entry point needs lives in the
// fixed array below.
//
// The scratch is a file-scope device array of FLCE_NOALLOC_SCRATCH_BYTES
// (16 MiB).  Every GPU on which this entry point runs keeps it allocated
// until the process exits.  In host code the array's name is only a host-side
// stand-in, not a device address, so the first call on each device looks the
// real address up with cudaGetSymbolAddress (with that device current) and
// caches it; make that first call before any stream capture.
//
// All calls share the one array and it keeps the last call's contents.
// Nothing in it has to start at zero: in a call that completes normally,
// every slot the merge reads was written earlier in that same call.  After a
// bounded wait expired (FLCE_ERR_TIMEOUT in the error word) the GEMM skips
// its partial writes, so the merge may read an earlier call's partials: loss
// and lse are then undefined, as the header states.  Two calls whose kernels
// overlap on the GPU (different streams, or different host threads) race on
// the array and give wrong results; serialise them.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <mutex>
#include <string>

#include "flce.h"
#include "aux_kernels.cuh"
#include "gemm_core.cuh"
#include "ptx.cuh"

using namespace flce;

static __device__ __align__(256) unsigned char flce_noalloc_scratch[FLCE_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kNaStages = 4;
constexpr int kNaMaxDevices = 64;
constexpr unsigned long long kNaTimeoutNs = 2000000000ull;

std::mutex g_na_mutex;
void* g_na_scratch[kNaMaxDevices] = {nullptr};
int g_na_sms[kNaMaxDevices] = {0};
bool g_na_attr[kNaMaxDevices] = {false};
thread_local std::string g_na_error;

int64_t na_ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t na_align(size_t x) { return (x + 255) / 256 * 256; }

flce_status na_cuda_fail(cudaError_t e, const char* what) {
  char buf[256];
  snprintf(buf, sizeof buf, "%s: %s", what, cudaGetErrorString(e));
  g_na_error = buf;
  return FLCE_ERR_CUDA;
}

// Forward partials and merge block sums of one call, laid out in the array.
struct NaPlan {
  int m_blocks, m_pad, v_tiles, group_len, n_groups, merge_blocks;
  size_t off_block_loss, off_block_valid, total;
};

// Smallest power-of-two vocabulary group length whose partials fit.
bool na_plan(int64_t N, int64_t V, NaPlan* p) {
  p->m_blocks = (int)na_ceil_div(std::max<int64_t>(N, 1), BM);
  p->m_pad = p->m_blocks * BM;
  p->v_tiles = (int)na_ceil_div(V, BN);
  p->merge_blocks = (int)merge_block_count(N);
  const size_t sums = na_align((size_t)p->merge_blocks * sizeof(double)) +
                      na_align((size_t)p->merge_blocks * sizeof(int));
  for (int L = 1;; L *= 2) {
    const int groups = (int)na_ceil_div(p->v_tiles, L);
    const size_t parts = na_align((size_t)groups * p->m_pad * sizeof(float4));
    if (parts + sums <= FLCE_NOALLOC_SCRATCH_BYTES) {
      p->group_len = L;
      p->n_groups = groups;
      p->off_block_loss = parts;
      p->off_block_valid = parts + na_align((size_t)p->merge_blocks * sizeof(double));
      p->total = parts + sums;
      return true;
    }
    if (groups == 1) return false;
  }
}

// Once per device, with that device current: the array's device address.
flce_status na_setup(int* scratch_sms, void** scratch_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return na_cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kNaMaxDevices) return FLCE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_na_mutex);
  if (!g_na_scratch[dev]) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return na_cuda_fail(e, "cudaDeviceGetAttribute");
    if (!(major == 10 && minor == 3)) return FLCE_ERR_UNSUPPORTED;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, flce_noalloc_scratch);
    if (e != cudaSuccess) return na_cuda_fail(e, "cudaGetSymbolAddress");
    if (p == nullptr) {
      g_na_error = "cudaGetSymbolAddress returned a null address";
      return FLCE_ERR_CUDA;
    }
    g_na_sms[dev] = sms;
    g_na_scratch[dev] = p;
  }
  if (!g_na_attr[dev]) {
    e = cudaFuncSetAttribute(gemm_kernel<Epi::kLse, false, false, kNaStages>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             gemm_smem_bytes<Epi::kLse, kNaStages, false, false>());
    if (e != cudaSuccess) return na_cuda_fail(e, "cudaFuncSetAttribute");
    g_na_attr[dev] = true;
  }
  *scratch_sms = g_na_sms[dev];
  *scratch_out = g_na_scratch[dev];
  return FLCE_OK;
}

flce_status na_map(CUtensorMap* m, const void* base, uint64_t k, uint64_t rows,
                   uint32_t box_rows) {
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
  if (!fn) {
    g_na_error = "cuTensorMapEncodeTiled entry point unavailable";
    return FLCE_ERR_CUDA;
  }
  cuuint64_t dims[2] = {k, std::max<uint64_t>(rows, 1)};
  cuuint64_t strides[1] = {k * 2};
  cuuint32_t box[2] = {BK, box_rows};
  cuuint32_t es[2] = {1, 1};
  if (fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
    g_na_error = "cuTensorMapEncodeTiled failed";
    return FLCE_ERR_CUDA;
  }
  return FLCE_OK;
}

bool na_aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace

extern "C" flce_status flce_forward_noalloc(const void* X, const void* W, const int64_t* labels,
                                            int64_t N, int64_t H, int64_t V,
                                            int64_t ignore_index, float smoothing,
                                            flce_reduction reduction, float* loss, float* lse,
                                            int32_t* valid_count, int32_t* err_word,
                                            void* stream) {
  // Host-side checks first: nothing is launched on an error.
  if (N < 0 || H <= 0 || V <= 0 || H % 8 != 0) return FLCE_ERR_ARG;
  if (N > (int64_t)INT32_MAX - 1024 || V > (int64_t)INT32_MAX - 1024 || H > (int64_t)INT32_MAX)
    return FLCE_ERR_ARG;
  if (reduction != FLCE_MEAN && reduction != FLCE_SUM) return FLCE_ERR_ARG;
  if (!(smoothing >= 0.f && smoothing < 1.f)) return FLCE_ERR_ARG;
  if (!W || !na_aligned(W, 16) || !loss || !valid_count || !err_word) return FLCE_ERR_ARG;
  // the merge and loss kernels store these as 32-bit words
  if (!na_aligned(err_word, 4) || !na_aligned(loss, 4) || !na_aligned(valid_count, 4))
    return FLCE_ERR_ARG;
  if (N > 0 && (!X || !labels || !lse || !na_aligned(X, 16) || !na_aligned(labels, 8) ||
                !na_aligned(lse, 4)))
    return FLCE_ERR_ARG;
  NaPlan pl;
  if (!na_plan(N, V, &pl)) {
    char buf[200];
    snprintf(buf, sizeof buf,
             "flce_forward_noalloc: N=%lld needs more than the fixed %u-byte scratch", (long long)N,
             (unsigned)FLCE_NOALLOC_SCRATCH_BYTES);
    g_na_error = buf;
    return FLCE_ERR_WORKSPACE;
  }
  int sms = 0;
  void* scratch = nullptr;
  flce_status s = na_setup(&sms, &scratch);
  if (s != FLCE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(scratch);
  double* block_loss = reinterpret_cast<double*>(base + pl.off_block_loss);
  int* block_valid = reinterpret_cast<int*>(base + pl.off_block_valid);
  cudaError_t e;
  if (N > 0) {
    CUtensorMap tmX, tmW;
    if ((s = na_map(&tmX, X, H, N, BM)) != FLCE_OK) return s;
    if ((s = na_map(&tmW, W, H, V, BN)) != FLCE_OK) return s;
    GemmParams p{};
    p.m_size = (int)N;
    p.n_size = (int)V;
    p.k_size = (int)H;
    p.m_blocks = pl.m_blocks;
    p.n_blocks = pl.v_tiles;
    p.group_len = pl.group_len;
    p.n_groups = pl.n_groups;
    p.num_units = pl.m_blocks * pl.n_groups;
    p.m_fastest = 1;
    p.labels = labels;
    p.ignore_index = ignore_index;
    p.vocab = (int)V;
    p.col_base = 0;
    p.col_limit = (int)V;
    p.smoothing = smoothing;
    p.partials = reinterpret_cast<float4*>(base);
    p.m_pad = pl.m_pad;
    p.err_word = err_word;
    p.timeout_ns = kNaTimeoutNs;
    const int grid = std::min(p.num_units, sms);
    gemm_kernel<Epi::kLse, false, false, kNaStages>
        <<<grid, NUM_THREADS, gemm_smem_bytes<Epi::kLse, kNaStages, false, false>(), st>>>(tmX, tmW, tmX, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return na_cuda_fail(e, "forward GEMM launch");
    lse_merge_kernel<<<pl.merge_blocks, MERGE_THREADS, 0, st>>>(
        p.partials, pl.n_groups, pl.m_pad, (int)N, (int)V, labels, ignore_index, smoothing, 0.f,
        lse, nullptr, block_loss, block_valid, err_word, nullptr, 1);
    if ((e = cudaGetLastError()) != cudaSuccess) return na_cuda_fail(e, "merge launch");
  }
  loss_finalize_kernel<<<1, MERGE_THREADS, 0, st>>>(block_loss, block_valid,
                                                     N > 0 ? pl.merge_blocks : 0,
                                                     reduction == FLCE_SUM, loss, valid_count);
  if ((e = cudaGetLastError()) != cudaSuccess) return na_cuda_fail(e, "loss launch");
  return FLCE_OK;
}

extern "C" const char* flce_noalloc_last_error(void) { return g_na_error.c_str(); }
