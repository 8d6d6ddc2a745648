// Small kernels around the GEMMs: merge of the per-group log-sum-exp
// partials, the deterministic loss reduction, the gradient scale, the dX
// down-conversion and the fp32 -> bf16 input cast.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include "ptx.cuh"

namespace flce {

constexpr int MERGE_THREADS = 256;
constexpr int MERGE_ROWS = 32;                             // token rows per merge block
constexpr int MERGE_SLICES = MERGE_THREADS / MERGE_ROWS;  // warps, each over a slice of the groups
constexpr float LN2 = 0.6931471805599453f;

// Blocks of the merge kernels for N token rows.
inline int64_t merge_block_count(int64_t N) {
  return ((N > 0 ? N : 1) + MERGE_ROWS - 1) / MERGE_ROWS;
}

// One slice of one row's vocabulary-group partials: groups slice,
// slice + MERGE_SLICES, ... merged online into (max*log2e, sum rescaled to
// that max, target logit, logit sum).  A group with no column (-inf max)
// adds nothing to the sum.
__device__ __forceinline__ float4 merge_slice(const float4* __restrict__ partials, int n_groups,
                                              int m_pad, int row, int slice) {
  float m = -INFINITY, s = 0.f, zy = 0.f, zs = 0.f;
#pragma unroll 4
  for (int g = slice; g < n_groups; g += MERGE_SLICES) {
    const float4 q = partials[(size_t)g * m_pad + row];
    if (q.x > m) {
      s = s * ex2_approx(m - q.x) + q.y;
      m = q.x;
    } else if (q.x > -INFINITY) {
      s += q.y * ex2_approx(q.x - m);
    }
    zy += q.z;
    zs += q.w;
  }
  return make_float4(m, s, zy, zs);
}

// The MERGE_SLICES slice results of row r, combined in slice order.
__device__ __forceinline__ float4 combine_slices(const float4 (*part)[MERGE_ROWS], int r) {
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < MERGE_SLICES; ++k) M = fmaxf(M, part[k][r].x);
  float S = 0.f, zy = 0.f, zs = 0.f;
#pragma unroll
  for (int k = 0; k < MERGE_SLICES; ++k) {
    const float4 q = part[k][r];
    if (q.x > -INFINITY) S += q.y * ex2_approx(q.x - M);
    zy += q.z;
    zs += q.w;
  }
  return make_float4(M, S, zy, zs);
}

// MERGE_ROWS token rows per block; warp k merges groups k, k + MERGE_SLICES,
// ... of every row (coalesced: a warp reads 32 consecutive rows of one group),
// warp 0 combines the slices.  Merges the vocabulary-group partials
// (max*log2e, rescaled exp-sum, target logit, logit sum) into
//   lse_i = m_i + log d_i       ("Chunked and Fused Cross-Entropy ...",
//                                 "Mathematical Mechanics ...", step 2)
//   l_i   = valid_i * (lse_i - (1-eps) z_{i,y_i} - (eps/V) sum_j z_ij
//                    + alpha lse_i^2)            (z-loss term when alpha > 0)
// writes l_i per row when asked, and reduces l_i and valid_i over the block in
// a fixed tree order.  Every order is fixed, so the results are deterministic.
// A label outside [0, V) that is not ignore_index sets FLCE_ERR_LABEL and
// the row counts as ignored.
static __global__ void __launch_bounds__(MERGE_THREADS)
    lse_merge_kernel(const float4* __restrict__ partials, int n_groups, int m_pad, int N, int V,
                     const int64_t* __restrict__ labels, long long ignore_index, float smoothing,
                     float z_loss, float* __restrict__ lse_out, float* __restrict__ row_loss,
                     double* __restrict__ block_loss, int* __restrict__ block_valid,
                     int* err_word, const int* __restrict__ block_active, int block_rows) {
  __shared__ float4 s_part[MERGE_SLICES][MERGE_ROWS];
  const int r = threadIdx.x % MERGE_ROWS;
  const int slice = threadIdx.x / MERGE_ROWS;
  const int row = blockIdx.x * MERGE_ROWS + r;
  // a skipped block: every label in it is ignore_index, its logits were not formed
  const bool skipped = row < N && block_active && !block_active[row / block_rows];
  if (row < N && !skipped) s_part[slice][r] = merge_slice(partials, n_groups, m_pad, row, slice);
  __syncthreads();
  if (slice != 0) return;
  double loss = 0.0;
  int valid = 0;
  if (skipped) {
    lse_out[row] = __int_as_float(0x7fc00000);
    if (row_loss) row_loss[row] = 0.f;
  } else if (row < N) {
    const float4 t = combine_slices(s_part, r);
    const float lse = (t.x + log2f(t.y)) * LN2;
    lse_out[row] = lse;
    const long long y = labels[row];
    if (y != ignore_index) {
      if (y < 0 || y >= V) {
        record_error(err_word, kErrLabel);
      } else {
        valid = 1;
        double l = (double)lse - (1.0 - (double)smoothing) * (double)t.z;
        if (smoothing != 0.f) l -= (double)smoothing / (double)V * (double)t.w;
        if (z_loss != 0.f) l += (double)z_loss * (double)lse * (double)lse;
        loss = l;
      }
    }
    if (row_loss) row_loss[row] = (float)loss;
  }
#pragma unroll
  for (int o = MERGE_ROWS / 2; o > 0; o >>= 1) {
    loss += __shfl_xor_sync(0xffffffffu, loss, o);
    valid += __shfl_xor_sync(0xffffffffu, valid, o);
  }
  if (r == 0) {
    block_loss[blockIdx.x] = loss;
    block_valid[blockIdx.x] = valid;
  }
}

// Merge the vocabulary-group partials of ONE vocabulary shard into a single
// (max*log2e, rescaled sum, z_y, sum_z) per row -- the statistic shards
// exchange in the vocabulary-parallel layout.  Same geometry as
// lse_merge_kernel.
static __global__ void __launch_bounds__(MERGE_THREADS)
    shard_partial_kernel(const float4* __restrict__ partials, int n_groups, int m_pad, int N,
                         float4* __restrict__ out) {
  __shared__ float4 s_part[MERGE_SLICES][MERGE_ROWS];
  const int r = threadIdx.x % MERGE_ROWS;
  const int slice = threadIdx.x / MERGE_ROWS;
  const int row = blockIdx.x * MERGE_ROWS + r;
  if (row < N) s_part[slice][r] = merge_slice(partials, n_groups, m_pad, row, slice);
  __syncthreads();
  if (slice == 0 && row < N) out[row] = combine_slices(s_part, r);
}

// Single block: fixed-order sum of the block partials, then the mean over
// valid tokens (0 when none are valid: the chunked reference divides by
// max(valid_token_count, 1)) or the plain sum.
static __global__ void __launch_bounds__(MERGE_THREADS)
    loss_finalize_kernel(const double* __restrict__ block_loss, const int* __restrict__ block_valid,
                         int nblocks, int reduction_sum, float* loss_out, int* valid_out) {
  __shared__ double s_loss[MERGE_THREADS];
  __shared__ long long s_valid[MERGE_THREADS];
  double l = 0.0;
  long long v = 0;
  for (int b = threadIdx.x; b < nblocks; b += MERGE_THREADS) {
    l += block_loss[b];
    v += block_valid[b];
  }
  s_loss[threadIdx.x] = l;
  s_valid[threadIdx.x] = v;
  __syncthreads();
  for (int w = MERGE_THREADS / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      s_loss[threadIdx.x] += s_loss[threadIdx.x + w];
      s_valid[threadIdx.x] += s_valid[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double total = s_loss[0];
    const long long nv = s_valid[0];
    double out = total;
    if (!reduction_sum) out = nv > 0 ? total / (double)nv : 0.0;
    *loss_out = (float)out;
    *valid_out = (int)nv;
  }
}

// c = grad / N_valid (mean; 0 when N_valid = 0) or grad (sum); grad defaults to 1.
static __global__ void grad_scale_kernel(const int* valid_count, const float* grad_loss,
                                  int reduction_sum, float* scale_out) {
  const float g = grad_loss ? *grad_loss : 1.f;
  float c = g;
  if (!reduction_sum) {
    const int nv = *valid_count;
    c = nv > 0 ? (float)((double)g / (double)nv) : 0.f;
  }
  *scale_out = c;
}

// fp32 -> bf16 (round to nearest even) of n4 float4 groups: every thread
// issues CONVERT_UNROLL independent 16-byte loads before its stores, so a
// launch of a few blocks per SM keeps enough reads in flight to stream at
// HBM speed.  The source is read once (evict-first loads).
constexpr int CONVERT_THREADS = 256;
constexpr int CONVERT_UNROLL = 4;

__device__ __forceinline__ void convert_f32_bf16(const float4* __restrict__ in,
                                                 uint2* __restrict__ out, size_t n4) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i0 = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i0 < n4;
       i0 += stride * CONVERT_UNROLL) {
    float4 v[CONVERT_UNROLL];
#pragma unroll
    for (int u = 0; u < CONVERT_UNROLL; ++u) {
      const size_t i = i0 + u * stride;
      if (i < n4) v[u] = __ldcs(in + i);
    }
#pragma unroll
    for (int u = 0; u < CONVERT_UNROLL; ++u) {
      const size_t i = i0 + u * stride;
      if (i < n4) out[i] = make_uint2(pack_bf16x2(v[u].x, v[u].y), pack_bf16x2(v[u].z, v[u].w));
    }
  }
}

// Blocks of a conversion launch over n4 float4 groups on `sms` SMs.
inline unsigned convert_blocks(size_t n4, int sms) {
  const size_t per_block = (size_t)CONVERT_THREADS * CONVERT_UNROLL;
  const size_t want = (n4 + per_block - 1) / per_block;
  const size_t cap = (size_t)(sms > 0 ? sms : 1) * 8;
  return (unsigned)(want < 1 ? 1 : (want < cap ? want : cap));
}

// dX = bf16(dX_acc).
static __global__ void __launch_bounds__(CONVERT_THREADS)
    dx_finalize_bf16_kernel(const float4* __restrict__ acc, uint2* __restrict__ out, size_t n4) {
  convert_f32_bf16(acc, out, n4);
}

// fp32 inputs -> bf16 operands.
static __global__ void __launch_bounds__(CONVERT_THREADS)
    cast_f32_bf16_kernel(const float4* __restrict__ in, uint2* __restrict__ out, size_t n4) {
  convert_f32_bf16(in, out, n4);
}

// Token blocks of `block_rows` rows that hold at least one label other than
// ignore_index: per-block flag, and the ascending list of active blocks with
// its length (a single block of threads; the scan runs in block order).
static __global__ void __launch_bounds__(MERGE_THREADS)
    active_blocks_kernel(const int64_t* __restrict__ labels, int N, long long ignore_index,
                         int block_rows, int n_blocks, int* __restrict__ flags,
                         int* __restrict__ list, int* __restrict__ count) {
  __shared__ int s_base;
  __shared__ int s_flag[MERGE_THREADS];
  if (threadIdx.x == 0) s_base = 0;
  __syncthreads();
  for (int b0 = 0; b0 < n_blocks; b0 += MERGE_THREADS) {
    const int b = b0 + threadIdx.x;
    int active = 0;
    if (b < n_blocks) {
      const int r1 = min(N, (b + 1) * block_rows);
      for (int r = b * block_rows; r < r1 && !active; ++r) active = labels[r] != ignore_index;
      flags[b] = active;
    }
    s_flag[threadIdx.x] = active;
    __syncthreads();
    if (threadIdx.x == 0) {
      int base = s_base;
      for (int t = 0; t < MERGE_THREADS && b0 + t < n_blocks; ++t)
        if (s_flag[t]) list[base++] = b0 + t;
      s_base = base;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) *count = s_base;
}

// dX_acc rows of skipped blocks are zero (their dZ rows are).
static __global__ void zero_skipped_rows_kernel(const int* __restrict__ flags, int block_rows,
                                                float* __restrict__ acc, int N, int H) {
  const size_t total = (size_t)N * H;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int row = (int)(i / H);
    if (!flags[row / block_rows]) acc[i] = 0.f;
  }
}

// Test-only: one bounded wait on an mbarrier that nothing arrives on.  It must
// give up after `timeout_ns`, record FLCE_ERR_TIMEOUT and return -- the path
// every pipeline wait of the GEMM kernels takes when its partner never comes.
static __global__ void wait_timeout_probe_kernel(int* err_word, unsigned long long timeout_ns,
                                                 int* waited_out) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtx ctx{&abort_flag, err_word, timeout_ns};
    const uint64_t t0 = global_timer_ns();
    const bool ok = mbar_wait(&bar, 0, ctx);
    *waited_out = ok ? -1 : (int)((global_timer_ns() - t0) / 1000ull);  // microseconds
  }
}

}  // namespace flce
