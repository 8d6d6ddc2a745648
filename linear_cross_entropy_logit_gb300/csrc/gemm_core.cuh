// Warp-specialised tcgen05 GEMM for sm_103a with the epilogues of the fused
// linear cross-entropy path.
//
// Persistent, one CTA per SM, 6 warps:
//   warp 0      TMA producer (one elected lane): fills a ring of shared-memory
//               stages with bf16 operand tiles (128-byte swizzle)
//   warp 1      TMEM allocator, then MMA issuer (one elected lane): tcgen05.mma
//               with a double-buffered fp32 accumulator in TMEM (2 x 256
//               columns = all 512), so the epilogue of tile t overlaps the main
//               loop of tile t+1
//   warps 2..5  epilogue: warp w reads TMEM lanes 32*(w%4) .. +31, so each
//               thread owns one accumulator row
//
// Two tile shapes:
//   PAIR = false  one CTA computes a 128 x 256 tile (tcgen05.mma.cta_group::1,
//                 M = 128); a stage holds 128 x 64 of A and 256 x 64 of B.
//   PAIR = true   a cluster of two CTAs on two SMs computes a 256 x 256 tile
//                 (tcgen05.mma.cta_group::2, M = 256).  Each CTA loads its own
//                 128 rows of A and its half (128 rows) of B, so a stage is
//                 32 KB per SM instead of 48 KB; the leader CTA (rank 0) issues
//                 the MMAs, which read both CTAs' shared memory and write each
//                 CTA's 128 accumulator rows into its own TMEM.
//   QUAD (CL = 4) the pair tiles, launched with 4-CTA clusters preferred: the
//                 two pairs of a 4-CTA cluster take two tiles that share one
//                 operand (B when they differ in row block, A when they differ
//                 in column block) and walk them in step, each CTA loading one
//                 64-row half of its share of that operand and multicasting it
//                 to its counterpart in the other pair (rank ^ 2).  Operand
//                 traffic from L2 drops by a quarter.  CTAs the hardware places
//                 in 2-CTA clusters run the same tiles without multicast.
//
// D = A * B^T with A: M x K and B: N x K as the MMA sees them.  Either operand
// may be K-major (K contiguous in memory) or MN-major (M/N contiguous):
//   forward logits / dZ recompute   Z = X W^T        A = X (K-major), B = W (K-major)
//   weight gradient                 dW = dZ^T X      A = dZ (MN-major), B = X (MN-major)
//   input gradient                  dX += dZ W       A = dZ (K-major), B = W (MN-major)
//
// Epilogues:
//   kLse   online log-sum-exp over the tile's vocabulary columns ("Chunked and
//          Fused Cross-Entropy ...", "Mathematical Mechanics of Chunked Online
//          Cross-Entropy", step 2; "Fused cross-entropy -- the memory kernel",
//          "Trick 1 - online softmax"): each thread keeps its row's running max
//          and rescaled exp-sum across the tiles of a work unit, plus the
//          target logit and the row sum of logits (label smoothing), and
//          writes one partial per (vocabulary group, row).  No logit leaves
//          the SM.
//   kDz    dZ = c * valid * (exp(z - lse) - (1-eps) 1[j=y] - eps/V)
//          ("Mathematical Mechanics ...", step 3; "The gradient that makes
//          fusion trivial"), rounded to bf16 in shared memory and written by
//          TMA into the bounded N x Cv chunk scratch.
//   kStore fp32 tile written (or reduce-added) by TMA: the dW and dX GEMMs of
//          step 4 ("Backward Hidden and Weight Accumulation").
#pragma once
#include <cstdint>
#include <cuda.h>
#include "ptx.cuh"

namespace flce {

constexpr int BM = 128;                // accumulator rows per CTA (TMEM lanes)
constexpr int BN = 256;                // tile columns (TMEM columns per buffer)
constexpr int BK = 64;                 // bf16 elements per 128-byte row
constexpr int MN_BOX_BYTES = 64 * 128;  // one MN-major box: 64 MN elements x 64 k rows
constexpr int NUM_THREADS = 192;
constexpr int NUM_EPI_WARPS = 4;
constexpr int STAGING_BUF_BYTES = 32 * 128;               // 32 rows x 128 bytes
constexpr int STAGING_BYTES = NUM_EPI_WARPS * 2 * STAGING_BUF_BYTES;
constexpr int TMEM_COLS = 2 * BN;
constexpr int BARRIER_BYTES = 256;
constexpr int STAGES_META = 8;          // >= STAGES of any instantiation
constexpr int FILTER_MAX_KB = 1024;     // k-blocks of one filtered tile (keep bytes in smem)
constexpr float LOG2E = 1.4426950408889634f;

// Tile geometry of the two variants.
template <bool PAIR>
struct TileCfg {
  static constexpr int TILE_M = PAIR ? 2 * BM : BM;    // rows of D per (pair of) CTA(s)
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;    // rows of B this CTA loads
  static constexpr int A_STAGE = BM * 128;             // bytes of A per stage
  static constexpr int B_STAGE = B_ROWS * 128;         // bytes of B per stage
  static constexpr int STAGE = A_STAGE + B_STAGE;
};

enum class Epi : int { kLse = 0, kDz = 1, kStore = 2 };

struct GemmParams {
  int m_size;      // rows of D
  int n_size;      // columns of D
  int k_size;      // contraction length
  int m_blocks;    // ceil(m_size / TILE_M)
  int n_blocks;    // ceil(n_size / BN)
  int group_len;   // consecutive column tiles per work unit
  int n_groups;    // ceil(n_blocks / group_len)
  int num_units;   // m_blocks * n_groups
  int m_fastest;   // 1: consecutive units walk row blocks (share B); 0: walk column groups
  int m_band;      // m_fastest: walk row blocks in bands of this many (0 = all at once)
  int n_band;      // !m_fastest: walk column groups in bands of this many (0 = all at once)
  // kLse / kDz
  const int64_t* labels;  // per D row (token)
  long long ignore_index;
  int vocab;              // V
  int col_base;           // vocabulary index of D column 0
  int col_limit;          // D columns >= col_limit do not exist
  float smoothing;        // eps
  float z_loss;           // kDz: z-loss weight alpha (softmax term scaled by 1 + 2 alpha lse)
  float4* partials;       // kLse: [n_groups][m_pad] of (max*log2e, sum, z_y, sum_z)
  int m_pad;              // m_blocks * TILE_M
  const float* lse;       // kDz: per-row log-sum-exp
  const float* scale;     // kDz: device scalar c = grad / N_valid
  // kStore
  int reduce_add;         // 1: TMA reduce-add onto the output, 0: overwrite
  // Skipping fully ignored token blocks (SFT-style masking).  When row_list is
  // set, units walk only the row blocks it lists (device count *row_count, in
  // units of TILE_M rows).  When k_list is set, the contraction walks only the
  // token blocks it lists (*k_count entries of k_per_entry k-blocks each); a
  // tile with no active k-block is written as zeros.
  const int* row_list;
  const int* row_count;
  const int* k_list;
  const int* k_count;
  int k_per_entry;
  int list_cap;       // entries row_list / k_list hold (index checks of the debug build)
  // Gradient filtering (CCE-style).  The kDz launch marks, for every
  // 32-token x 64-column block of dZ that holds a probability >= filter_thr
  // or a target, maskX[token tile][vocab k-block] and maskW[vocab tile][token
  // k-block] (tiles of mask_tile rows; the masks start zeroed).  A kStore
  // launch given `fmask` (its own mask, row stride fmask_ld) walks only the
  // k-blocks marked for its tile; the first k-block of a tile always runs.
  uint8_t* mask_x_out;
  uint8_t* mask_w_out;
  int mask_x_ld;      // vocabulary k-blocks per token tile
  int mask_w_ld;      // token k-blocks per vocabulary tile
  int mask_tile;      // rows of the dX / dW tiles the masks describe
  float filter_thr;
  long long mask_x_bytes;  // sizes of the two masks (index checks of the debug build)
  long long mask_w_bytes;
  const uint8_t* fmask;
  int fmask_ld;
  long long fmask_bytes;   // size of fmask (index checks of the debug build)
  // L2 residency: the operand reused across waves of tiles (0 = A, 1 = B) is
  // loaded with an evict_last policy covering `l2_keep_frac` of its lines.
  int l2_keep_b;
  float l2_keep_frac;
  // control
  int* err_word;
  unsigned long long timeout_ns;
};

// EXT = the optional features (token-block skip lists, gradient filtering,
// L2 hints) are compiled in.  Calls that use none of them run EXT = false,
// whose loops carry no trace of them.
template <Epi EPI, int STAGES, bool PAIR, bool EXT>
constexpr int gemm_smem_bytes() {
  return STAGES * TileCfg<PAIR>::STAGE + (EPI == Epi::kLse ? 0 : STAGING_BYTES) + BARRIER_BYTES +
         ((EXT && EPI == Epi::kStore) ? FILTER_MAX_KB : 0) + 1024;
}

// Row-block count and unit count of this launch (after skipping, if any).
struct UnitSpace {
  int m_blocks;
  int num_units;
};

__device__ __forceinline__ UnitSpace unit_space(const GemmParams& p) {
  if (p.row_list) {
    int cnt = *p.row_count;
    if (!dbg_ok(cnt >= 0 && cnt <= p.list_cap, p.err_word)) cnt = 0;
    return {cnt, cnt * p.n_groups};
  }
  return {p.m_blocks, p.num_units};
}

template <bool EXT>
__device__ __forceinline__ void unit_coords(const GemmParams& p, const UnitSpace& us, int u,
                                            int& mb, int& nb0, int& nb1, int& g) {
  if (p.m_fastest) {
    if (p.m_band > 0 && p.m_band < us.m_blocks) {
      // bands of m_band row blocks, each walked over all column groups
      const int band_units = p.m_band * p.n_groups;
      const int band = u / band_units;
      const int ub = u - band * band_units;
      const int mb0 = band * p.m_band;
      const int mbn = min(p.m_band, us.m_blocks - mb0);
      mb = mb0 + ub % mbn;
      g = ub / mbn;
    } else {
      mb = u % us.m_blocks;
      g = u / us.m_blocks;
    }
  } else if (p.n_band > 0 && p.n_band < p.n_groups) {
    // bands of n_band column groups, each walked over all row blocks: the B
    // operand of one band is re-read by every row block while it is in L2
    const int band_units = p.n_band * us.m_blocks;
    const int band = u / band_units;
    const int ub = u - band * band_units;
    const int g0 = band * p.n_band;
    const int gn = min(p.n_band, p.n_groups - g0);
    g = g0 + ub % gn;
    mb = ub / gn;
  } else {
    g = u % p.n_groups;
    mb = u / p.n_groups;
  }
  if constexpr (EXT) {
    if (p.row_list) mb = dbg_ok(mb >= 0 && mb < us.m_blocks, p.err_word) ? p.row_list[mb] : 0;
  }
  nb0 = g * p.group_len;
  nb1 = min(nb0 + p.group_len, p.n_blocks);
  // debug build: a unit outside the tile grid gets no tiles (every role of
  // the CTA computes the same coordinates, so all of them skip it)
  if (!dbg_ok(mb >= 0 && mb < p.m_blocks && g >= 0 && g < p.n_groups && nb0 < p.n_blocks,
              p.err_word)) {
    mb = 0;
    g = 0;
    nb0 = nb1 = 0;
  }
}

// Number of k-blocks the contraction walks, and the i-th of them.
__device__ __forceinline__ int kblock_count(const GemmParams& p, int num_kb) {
  if (!p.k_list) return num_kb;
  int cnt = *p.k_count;
  if (!dbg_ok(cnt >= 0 && cnt <= p.list_cap, p.err_word)) cnt = 0;
  return cnt * p.k_per_entry;
}

// (debug build: a k-block outside [0, ceil(k_size / BK)) is replaced by 0)
__device__ __forceinline__ int kblock_at(const GemmParams& p, int i) {
  if (!p.k_list) return i;
  const int e = i / p.k_per_entry;
  if (!dbg_ok(e >= 0 && e < p.list_cap, p.err_word)) return 0;
  const int kb = p.k_list[e] * p.k_per_entry + i % p.k_per_entry;
  return dbg_ok(kb >= 0 && kb < (p.k_size + BK - 1) / BK, p.err_word) ? kb : 0;
}

// Gradient filtering: copy the keep bytes of row block mb's tile into shared
// memory, indexed like the k loop (i-th walked k-block), and return the index
// of the last kept one.  The first walked k-block always runs.
__device__ __forceinline__ int load_tile_keep(const GemmParams& p, int mb, int num_kb,
                                              uint8_t* keep) {
  const uint8_t* row = p.fmask + (size_t)mb * p.fmask_ld;
  if (!p.k_list) {
    const uint4* src = reinterpret_cast<const uint4*>(row);
    const int n16 = (num_kb + 15) / 16;
    if (dbg_ok((long long)mb * p.fmask_ld + n16 * 16 <= p.fmask_bytes && n16 * 16 <= FILTER_MAX_KB,
               p.err_word)) {
#pragma unroll 4
      for (int i = 0; i < n16; ++i) reinterpret_cast<uint4*>(keep)[i] = __ldg(src + i);
    } else {
      for (int i = 0; i < num_kb && i < FILTER_MAX_KB; ++i) keep[i] = 1;
    }
  } else {
#pragma unroll 4
    for (int i = 0; i < num_kb; ++i) {
      const int kb = kblock_at(p, i);
      keep[i] = dbg_ok(i < FILTER_MAX_KB && kb < p.fmask_ld &&
                           (long long)mb * p.fmask_ld + kb < p.fmask_bytes,
                       p.err_word)
                    ? __ldg(row + kb)
                    : (uint8_t)1;
    }
  }
  keep[0] = 1;
  int last = num_kb - 1;
  while (last > 0 && !keep[last]) --last;
  return last;
}


// tcgen05.wait::ld with the loaded registers as operands, so no use of them
// can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// tcgen05.wait::ld with the 64 loaded registers as operands, so no use of
// them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait_regs64(uint32_t (&r)[64]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]),
                 "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]),
                 "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]),
                 "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]),
                 "+r"(r[54]), "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]),
                 "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63])
               :
               : "memory");
}

// One warp-uniform bounded wait: lane 0 polls, the result is broadcast.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtx& ctx,
                                          int lane) {
  int ok = 0;
  if (lane == 0) ok = mbar_wait(bar, parity, ctx) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

// Write one 32-bit-word row of 128 bytes (32 words) into a 128B-swizzled
// staging buffer: 16-byte chunk c of row r lands at chunk c ^ (r & 7).
__device__ __forceinline__ void staging_write_row(uint32_t buf, int row, const uint32_t* w) {
  const uint32_t base = buf + row * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    st_shared_v4(base + ((c ^ (row & 7)) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2],
                 w[4 * c + 3]);
  }
}

// Per-row constants of the dZ epilogue: dZ = pcoef * p - eps_v - tgt * 1[j = y]
// with p = exp2(z * log2(e) + neg_lse2), c = grad / N_valid, valid = 0 for
// ignored and padding rows.
struct DzRow {
  float pcoef;     // c * valid * (1 + 2 alpha lse)
  float neg_lse2;  // -lse * log2(e)
  float eps_v;     // c * valid * eps / V
  float tgt;       // c * valid * (1 - eps)
  float arg0;      // neg_lse2 + log2(pcoef) (-inf when pcoef = 0): pcoef * p = exp2(z log2 e + arg0)
};

__device__ __forceinline__ DzRow dz_row(bool valid, float lse_r, float c, float eps, float z_loss,
                                        int vocab) {
  const float coef = valid ? c : 0.f;
  const float pcoef = coef * fmaf(2.f * z_loss, lse_r, 1.f);
  const float neg_lse2 = -lse_r * LOG2E;
  return {pcoef, neg_lse2, coef * eps / (float)vocab, coef * (1.f - eps),
          neg_lse2 + __log2f(pcoef)};
}

// dZ of one 64-column slice of this thread's row: TMEM columns taddr .. +63 in,
// 32 packed bf16 pairs out; `off` = label - first column of the slice.
// Returns the largest probability of the slice when PMAX (gradient filtering).
// All 32 lanes of the warp must call it together (the target check is a
// warp vote: only a slice holding some lane's target walks the select chain).
template <bool PMAX>
__device__ __forceinline__ float dz_slice(uint32_t taddr, const DzRow& d, long long off,
                                          uint32_t (&w)[32]) {
  uint32_t r[64];
  tmem_ld_32x32b_x64(taddr, r);
  tmem_ld_wait_regs64(r);
  float pm[2] = {0.f, 0.f};
  // Without smoothing and with a non-negative scale on every lane's row the
  // scale folds into the exponent: pcoef * p = exp2(z log2 e + arg0), one FFMA
  // and one exp2 per element (warp-uniform choice).
  if (!PMAX && __all_sync(0xffffffffu, d.eps_v == 0.f && d.pcoef >= 0.f)) {
#pragma unroll
    for (int j = 0; j < 64; ++j)
      r[j] = __float_as_uint(ex2_approx(fmaf(__uint_as_float(r[j]), LOG2E, d.arg0)));
  } else {
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      const float pj = ex2_approx(fmaf(__uint_as_float(r[j]), LOG2E, d.neg_lse2));
      if constexpr (PMAX) pm[j & 1] = fmaxf(pm[j & 1], pj);
      r[j] = __float_as_uint(fmaf(d.pcoef, pj, -d.eps_v));
    }
  }
  const bool mine = off >= 0 && off < 64;
  if (__any_sync(0xffffffffu, mine)) {
    const int offi = mine ? (int)off : -1;
#pragma unroll
    for (int j = 0; j < 64; ++j)
      r[j] = (j == offi) ? __float_as_uint(__uint_as_float(r[j]) - d.tgt) : r[j];
  }
#pragma unroll
  for (int j = 0; j < 32; ++j)
    w[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
  return fmaxf(pm[0], pm[1]);
}

// One warp writes its 32 rows x 128 bytes (one row per lane) through a
// swizzled staging buffer and lane 0 stores (or reduce-adds) the box at
// (c0, row0) by TMA.  Each warp alternates its two buffers by a running count
// of its stores (not by the slice index: a clipped tile can end on either
// buffer), so the buffer written now was last read by the store before the
// latest one, and waiting until at most one store is still reading suffices.
__device__ __forceinline__ void staged_store(uint32_t buf, uint8_t* staging, int lane,
                                             const uint32_t* w, const CUtensorMap* out, int c0,
                                             int row0, bool reduce_add) {
  if (lane == 0) bulk_wait_group_read<1>();
  __syncwarp();
  staging_write_row(buf, lane, w);
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
    const void* src = staging + (buf - smem_u32(staging));
    if (reduce_add)
      tma_reduce_add_2d(out, src, c0, row0);
    else
      tma_store_2d(out, src, c0, row0);
    bulk_commit_group();
  }
}

// QUAD launches: unit u goes to pair (u mod #pairs) as for pairs, and units
// 2v, 2v+1 -- taken by the two pairs of one 4-CTA group in the same round --
// share an operand: with SHARE_B the same column group g and row blocks
// 2m, 2m+1 (row-block pairs walked like row blocks, bands halved); otherwise
// the same row block and column groups 2h, 2h+1 (group length 1).  The host
// only launches QUAD when these pairings cover the grid exactly.
template <bool SHARE_B>
__device__ __forceinline__ void unit_coords_quad(const GemmParams& p, int u, int& mb, int& nb0,
                                                 int& nb1, int& g) {
  const int i = u & 1;
  const int v = u >> 1;
  if constexpr (SHARE_B) {
    const int mh = p.m_blocks >> 1;
    int mbh;
    if (p.m_fastest) {
      const int band_h = p.m_band >> 1;
      if (band_h > 0 && band_h < mh) {
        const int band_units = band_h * p.n_groups;
        const int band = v / band_units;
        const int ub = v - band * band_units;
        const int m0 = band * band_h;
        const int mn = min(band_h, mh - m0);
        mbh = m0 + ub % mn;
        g = ub / mn;
      } else {
        mbh = v % mh;
        g = v / mh;
      }
    } else {
      g = v % p.n_groups;
      mbh = v / p.n_groups;
    }
    mb = 2 * mbh + i;
  } else {
    const int gh = p.n_groups >> 1;
    g = 2 * (v % gh) + i;
    mb = v / gh;
  }
  nb0 = g * p.group_len;
  nb1 = min(nb0 + p.group_len, p.n_blocks);
  if (!dbg_ok(mb >= 0 && mb < p.m_blocks && g >= 0 && g < p.n_groups && nb0 < p.n_blocks,
              p.err_word)) {
    mb = 0;
    g = 0;
    nb0 = nb1 = 0;
  }
}

// One CTA's 128-row half of an operand for one k-block, as two 64-row boxes
// (8 KB each): K-major boxes are 64 rows x 64 k, MN-major boxes 64 MN x 64 k.
// With `shared` and multicast the CTA loads only box `pic` and multicasts it
// to itself and its counterpart in the other pair; otherwise both boxes.
template <bool MN>
__device__ __forceinline__ void load_half_quad(uint8_t* dst, const CUtensorMap* map, uint32_t bar,
                                               int row0, int kb, bool shared, bool mcast,
                                               uint32_t pic, uint16_t mask) {
  if (shared && mcast) {
    const int r = row0 + (int)pic * 64;
    uint8_t* d = dst + pic * MN_BOX_BYTES;
    if constexpr (MN)
      tma_load_2d_pair_mcast(d, map, bar, r, kb * BK, mask);
    else
      tma_load_2d_pair_mcast(d, map, bar, kb * BK, r, mask);
  } else {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if constexpr (MN)
        tma_load_2d_pair(dst + i * MN_BOX_BYTES, map, bar, row0 + i * 64, kb * BK);
      else
        tma_load_2d_pair(dst + i * MN_BOX_BYTES, map, bar, kb * BK, row0 + i * 64);
    }
  }
}

// CL: 1 single-CTA tiles, 2 CTA pairs, 4 CTA pairs with 4-CTA clusters
// preferred (QUAD; EXT must be false).
template <Epi EPI, bool A_MN, bool B_MN, int STAGES, int CL, bool EXT, bool SHARE_B = false>
__device__ __forceinline__ void gemm_body(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                          const CUtensorMap& tmOut, const GemmParams& p) {
  constexpr bool PAIR = CL >= 2;
  constexpr bool QUAD = CL == 4;
  static_assert(!(QUAD && EXT), "4-CTA clusters run only the plain kernels");
  using Cfg = TileCfg<PAIR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  constexpr int kStaging = (EPI == Epi::kLse) ? 0 : STAGING_BYTES;
  uint8_t* staging = smem + STAGES * Cfg::STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + kStaging);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* stage_meta = abort_flag + 1;  // filtered launches: k-block index | last-of-tile flag
  uint8_t* tile_keep = reinterpret_cast<uint8_t*>(stage_meta + STAGES_META);  // FILTER_MAX_KB

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = PAIR ? cluster_ctarank() : 0u;  // rank in the cluster
  const uint32_t rank = crank & 1u;   // rank in the pair: 0 = leader (issues the MMAs)
  const uint32_t lrank = crank & ~1u;  // cluster rank of this pair's leader
  // QUAD: multicast only inside a 4-CTA cluster; pic = this pair's place in it
  const bool mcast = QUAD && cluster_nctarank() == 4u;
  const uint32_t pic = mcast ? (crank >> 1) : 0u;
  const uint16_t mc_mask = (uint16_t)((1u << crank) | (1u << (crank ^ 2u)));
  const uint16_t pair_mask = (uint16_t)(0x3u << lrank);
  const int pair_id = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int num_pairs = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      // with multicast both pairs' MMAs read into this CTA's stages
      mbar_init(&empty[s], mcast ? 2 : 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], PAIR ? 2 * NUM_EPI_WARPS : NUM_EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    if (EPI != Epi::kLse) prefetch_tensormap(&tmOut);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR) {
    cluster_sync_all();  // the peer's barriers exist before any remote arrive
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtx ctx{abort_flag, p.err_word, p.timeout_ns};
  const int num_kb_all = (p.k_size + BK - 1) / BK;
  const int num_kb = EXT ? kblock_count(p, num_kb_all) : num_kb_all;
  const UnitSpace us = EXT ? unit_space(p) : UnitSpace{p.m_blocks, p.num_units};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      uint64_t keep = 0;
      bool keep_a = false, keep_b = false;
      if constexpr (EXT) {
        keep = l2_policy_evict_last(p.l2_keep_frac);
        keep_a = p.l2_keep_frac > 0.f && !p.l2_keep_b;
        keep_b = p.l2_keep_frac > 0.f && p.l2_keep_b;
      }
      for (int u = pair_id; u < us.num_units && ok; u += num_pairs) {
        int mb, nb0, nb1, g;
        if constexpr (QUAD)
          unit_coords_quad<SHARE_B>(p, u, mb, nb0, nb1, g);
        else
          unit_coords<EXT>(p, us, u, mb, nb0, nb1, g);
        const int a_row = mb * Cfg::TILE_M + (int)rank * BM;
        for (int nb = nb0; nb < nb1 && ok; ++nb) {
          const int b_row = nb * BN + (int)rank * Cfg::B_ROWS;
          // filtered launches: the last kept k-block of the tile ends it
          int last_kept = num_kb - 1;
          if constexpr (EXT) {
            if (p.fmask) last_kept = load_tile_keep(p, mb, num_kb, tile_keep);
          }
          for (int ki = 0; ki < num_kb; ++ki) {
            int kb = ki;
            if constexpr (EXT) {
              kb = kblock_at(p, ki);
              if (p.fmask && ki > last_kept) break;
              if (p.fmask && !tile_keep[ki]) continue;
            }
            const int s = it % STAGES;
            const uint32_t r = it / STAGES;
            if (!mbar_wait(&empty[s], (r & 1u) ^ 1u, ctx)) {
              ok = false;
              break;
            }
            if constexpr (EXT) {
              if (p.fmask && rank == 0) stage_meta[s] = kb | (ki == last_kept ? (1 << 30) : 0);
            }
            uint8_t* a_dst = stages + s * Cfg::STAGE;
            uint8_t* b_dst = a_dst + Cfg::A_STAGE;
            if constexpr (QUAD) {
              // The pair's bytes -- its own loads and the pieces the other
              // pair multicasts into it -- complete on the leader's barrier.
              const uint32_t bar = mapa_shared(smem_u32(&full[s]), lrank);
              if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * Cfg::STAGE);
              load_half_quad<A_MN>(a_dst, &tmA, bar, a_row, kb, !SHARE_B, mcast, pic, mc_mask);
              load_half_quad<B_MN>(b_dst, &tmB, bar, b_row, kb, SHARE_B, mcast, pic, mc_mask);
            } else if constexpr (PAIR) {
              // Both CTAs' loads complete on the leader's full barrier, which
              // only the leader arms with the pair's byte count.
              const uint32_t bar = mapa_shared(smem_u32(&full[s]), lrank);
              if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * Cfg::STAGE);
              if constexpr (!EXT) {
                if constexpr (!A_MN) {
                  tma_load_2d_pair(a_dst, &tmA, bar, kb * BK, a_row);
                } else {
#pragma unroll
                  for (int i = 0; i < BM / 64; ++i)
                    tma_load_2d_pair(a_dst + i * MN_BOX_BYTES, &tmA, bar, a_row + i * 64, kb * BK);
                }
                if constexpr (!B_MN) {
                  tma_load_2d_pair(b_dst, &tmB, bar, kb * BK, b_row);
                } else {
#pragma unroll
                  for (int i = 0; i < Cfg::B_ROWS / 64; ++i)
                    tma_load_2d_pair(b_dst + i * MN_BOX_BYTES, &tmB, bar, b_row + i * 64,
                                     kb * BK);
                }
              } else {
                auto ld = [&](void* dst, const CUtensorMap* m, int x, int y, bool hint) {
                  if (hint)
                    tma_load_2d_pair_hint(dst, m, bar, x, y, keep);
                  else
                    tma_load_2d_pair(dst, m, bar, x, y);
                };
                if constexpr (!A_MN) {
                  ld(a_dst, &tmA, kb * BK, a_row, keep_a);
                } else {
#pragma unroll
                  for (int i = 0; i < BM / 64; ++i)
                    ld(a_dst + i * MN_BOX_BYTES, &tmA, a_row + i * 64, kb * BK, keep_a);
                }
                if constexpr (!B_MN) {
                  ld(b_dst, &tmB, kb * BK, b_row, keep_b);
                } else {
#pragma unroll
                  for (int i = 0; i < Cfg::B_ROWS / 64; ++i)
                    ld(b_dst + i * MN_BOX_BYTES, &tmB, b_row + i * 64, kb * BK, keep_b);
                }
              }
            } else {
              mbar_arrive_expect_tx(&full[s], Cfg::STAGE);
              if constexpr (!EXT) {
                if constexpr (!A_MN) {
                  tma_load_2d(a_dst, &tmA, &full[s], kb * BK, a_row);
                } else {
#pragma unroll
                  for (int i = 0; i < BM / 64; ++i)
                    tma_load_2d(a_dst + i * MN_BOX_BYTES, &tmA, &full[s], a_row + i * 64, kb * BK);
                }
                if constexpr (!B_MN) {
                  tma_load_2d(b_dst, &tmB, &full[s], kb * BK, b_row);
                } else {
#pragma unroll
                  for (int i = 0; i < Cfg::B_ROWS / 64; ++i)
                    tma_load_2d(b_dst + i * MN_BOX_BYTES, &tmB, &full[s], b_row + i * 64,
                                kb * BK);
                }
              } else {
                auto ld = [&](void* dst, const CUtensorMap* m, int x, int y, bool hint) {
                  if (hint)
                    tma_load_2d_hint(dst, m, &full[s], x, y, keep);
                  else
                    tma_load_2d(dst, m, &full[s], x, y);
                };
                if constexpr (!A_MN) {
                  ld(a_dst, &tmA, kb * BK, a_row, keep_a);
                } else {
#pragma unroll
                  for (int i = 0; i < BM / 64; ++i)
                    ld(a_dst + i * MN_BOX_BYTES, &tmA, a_row + i * 64, kb * BK, keep_a);
                }
                if constexpr (!B_MN) {
                  ld(b_dst, &tmB, kb * BK, b_row, keep_b);
                } else {
#pragma unroll
                  for (int i = 0; i < Cfg::B_ROWS / 64; ++i)
                    ld(b_dst + i * MN_BOX_BYTES, &tmB, b_row + i * 64, kb * BK, keep_b);
                }
              }
            }
            ++it;
          }
        }
      }
      if (!ok && rank == 0) {
        // Drain: the loads of the last (up to) STAGES issued iterations may
        // still be landing in shared memory.
        const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
        for (uint32_t j = first; j < it; ++j)
          mbar_wait_drain(&full[j % STAGES], (j / STAGES) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = make_idesc(A_MN, B_MN, Cfg::TILE_M, BN);
      // MN-major operand blocks are 64 elements wide; LBO = distance between them.
      constexpr uint32_t kMnLbo = MN_BOX_BYTES;
      uint32_t it = 0, tile = 0;
      bool ok = true;
      for (int u = pair_id; u < us.num_units && ok; u += num_pairs) {
        int mb, nb0, nb1, g;
        if constexpr (QUAD)
          unit_coords_quad<SHARE_B>(p, u, mb, nb0, nb1, g);
        else
          unit_coords<EXT>(p, us, u, mb, nb0, nb1, g);
        for (int nb = nb0; nb < nb1 && ok; ++nb) {
          const uint32_t acc = tile & 1u;
          const uint32_t ra = tile >> 1;
          if (!mbar_wait(&tempty[acc], (ra & 1u) ^ 1u, ctx)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * BN;
          for (int ki = 0; ki < num_kb; ++ki) {
            const int s = it % STAGES;
            const uint32_t r = it / STAGES;
            if (!mbar_wait(&full[s], r & 1u, ctx)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // filtered launches: the producer tells which stage ends the tile
            bool last_stage = false;
            if constexpr (EXT) last_stage = p.fmask && (stage_meta[s] & (1 << 30));
            const uint32_t a_addr = smem_u32(stages + s * Cfg::STAGE);
            const uint32_t b_addr = a_addr + Cfg::A_STAGE;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = A_MN ? smem_desc_sw128(a_addr + kk * 2048, kMnLbo, 1024)
                                       : smem_desc_sw128(a_addr + kk * 32, 16, 1024);
              const uint64_t bd = B_MN ? smem_desc_sw128(b_addr + kk * 2048, kMnLbo, 1024)
                                       : smem_desc_sw128(b_addr + kk * 32, 16, 1024);
              if constexpr (PAIR)
                mma_issue_pair(d_tmem, ad, bd, idesc, (ki | kk) != 0 ? 1u : 0u);
              else
                mma_issue(d_tmem, ad, bd, idesc, (ki | kk) != 0 ? 1u : 0u);
            }
            if constexpr (PAIR)
              mma_commit_pair_multicast(&empty[s], mcast ? (uint16_t)0xF : pair_mask);
            else
              mma_commit(&empty[s]);
            ++it;
            if (last_stage) break;
          }
          if (!ok) break;
          if constexpr (PAIR)
            mma_commit_pair_multicast(&tfull[acc], pair_mask);
          else
            mma_commit(&tfull[acc]);
          ++tile;
        }
      }
      // Every MMA this thread issued must finish before TMEM is released.
      if constexpr (PAIR)
        mma_commit_pair_multicast(mma_done, (uint16_t)(1u << lrank));
      else
        mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;              // TMEM lane quadrant of this warp
    const int row_in_tile = (int)rank * BM + q * 32 + lane;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t stag0 = smem_u32(staging) + (warp - 2) * 2 * STAGING_BUF_BYTES;
    uint32_t tile = 0;
    uint32_t nstore = 0;  // this warp's staged stores so far: buffer nstore & 1
    bool ok = true;
    float c_scale = 0.f;
    if constexpr (EPI == Epi::kDz) c_scale = *p.scale;

    for (int u = pair_id; u < us.num_units && ok; u += num_pairs) {
      int mb, nb0, nb1, g;
      if constexpr (QUAD)
        unit_coords_quad<SHARE_B>(p, u, mb, nb0, nb1, g);
      else
        unit_coords<EXT>(p, us, u, mb, nb0, nb1, g);
      const int row = mb * Cfg::TILE_M + row_in_tile;
      const int store_row0 = mb * Cfg::TILE_M + (int)rank * BM + q * 32;
      const bool row_ok = row < p.m_size;

      // Per-row state for kLse (natural-log max is m2 / log2(e)).
      float m2 = -INFINITY, ssum = 0.f, zy = 0.f, zsum = 0.f;
      long long label = 0;
      if constexpr (EPI != Epi::kStore)
        label = row_ok ? (long long)p.labels[row] : (long long)p.ignore_index;
      // A label outside [0, V) that is not ignore_index counts as ignored, as
      // in the forward's merge (which records FLCE_ERR_LABEL for it).
      const bool valid =
          row_ok && label != p.ignore_index && label >= 0 && label < (long long)p.vocab;
      const long long lab_rel = label - p.col_base;

      DzRow dzr{};
      if constexpr (EPI == Epi::kDz)
        dzr = dz_row(valid, row_ok ? p.lse[row] : 0.f, c_scale, p.smoothing, p.z_loss, p.vocab);

      for (int nb = nb0; nb < nb1; ++nb) {
        const uint32_t acc = tile & 1u;
        const uint32_t ra = tile >> 1;
        if (!warp_wait(&tfull[acc], ra & 1u, ctx, lane)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = lane_base + acc * BN;

        if constexpr (EPI == Epi::kLse) {
          // 64-column slices.  The epilogue runs beside the next tile's MMAs
          // and competes with them for the SM, so it is kept lean: a tile
          // wholly inside the vocabulary skips the per-column range check,
          // the exponent arguments take one packed FMA per two columns, the
          // max and sum run as four independent chains (the sums in two
          // packed adds), and the target-logit gather only runs for a
          // slice that holds some lane's target (a warp vote).
          const int tile_c0 = nb * BN;
          const bool full_tile = tile_c0 + BN <= p.col_limit;  // warp-uniform
#pragma unroll 1
          for (int sl = 0; sl < BN / 64; ++sl) {
            const int c0 = tile_c0 + sl * 64;
            const int nvalid = p.col_limit - c0;  // warp-uniform
            if (nvalid <= 0) break;
            uint32_t r[64];
            tmem_ld_32x32b_x64(taddr + sl * 64, r);
            tmem_ld_wait_regs64(r);
            if (p.smoothing != 0.f) {
              float zs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int j = 0; j < 64; ++j)
                zs[j & 3] += (full_tile || j < nvalid) ? __uint_as_float(r[j]) : 0.f;
              zsum += (zs[0] + zs[1]) + (zs[2] + zs[3]);
            }
            // target logit: a select chain (no dynamic register indexing)
            const long long off = lab_rel - c0;
            const bool mine = off >= 0 && off < 64 && off < nvalid;
            if (__any_sync(0xffffffffu, mine)) {
              const int offi = mine ? (int)off : -1;
#pragma unroll
              for (int j = 0; j < 64; ++j) zy = (j == offi) ? __uint_as_float(r[j]) : zy;
            }
            if (!full_tile) {
#pragma unroll
              for (int j = 0; j < 64; ++j)
                if (j >= nvalid) r[j] = __float_as_uint(-INFINITY);
            }
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int j = 0; j < 64; j += 2)
              mx[(j >> 1) & 3] =
                  fmax3(mx[(j >> 1) & 3], __uint_as_float(r[j]), __uint_as_float(r[j + 1]));
            // running max in units of log2 (scaling by log2(e) > 0 keeps the order)
            const float cm2 = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * LOG2E;
            if (cm2 > m2) {
              ssum *= ex2_approx(m2 - cm2);
              m2 = cm2;
            }
            // sum chains j mod 4, packed two per f32x2 register (each lane
            // rounds like the scalar FMA and add: same bits)
            uint64_t ps01 = 0ull, ps23 = 0ull;
            const uint64_t l2e = pack_f32x2(LOG2E, LOG2E), nm2 = pack_f32x2(-m2, -m2);
#pragma unroll
            for (int j = 0; j < 64; j += 2) {
              float a0, a1;
              unpack_f32x2(fma_f32x2(pack_u32x2(r[j], r[j + 1]), l2e, nm2), a0, a1);
              const uint64_t e = pack_f32x2(ex2_approx(a0), ex2_approx(a1));
              if ((j & 3) == 0)
                ps01 = add_f32x2(ps01, e);
              else
                ps23 = add_f32x2(ps23, e);
            }
            float p0, p1, p2, p3;
            unpack_f32x2(ps01, p0, p1);
            unpack_f32x2(ps23, p2, p3);
            ssum += (p0 + p1) + (p2 + p3);
          }
        } else if constexpr (EPI == Epi::kDz) {
#pragma unroll 1
          for (int sl = 0; sl < BN / 64; ++sl) {
            const int c0 = nb * BN + sl * 64;
            if (c0 >= p.col_limit) break;  // warp-uniform; the store would be clipped anyway
            const long long off = lab_rel - c0;
            uint32_t w[32];
            const float pmax = dz_slice<EXT>(taddr + sl * 64, dzr, off, w);
            if (EXT && p.mask_x_out) {
              // this 32-token x 64-column block is kept if a valid row has a
              // probability >= the threshold or its target in it
              const bool keep_row = valid && (pmax >= p.filter_thr || (off >= 0 && off < 64));
              if (__ballot_sync(0xffffffffu, keep_row) != 0u && lane == 0) {
                const long long ix = (long long)(store_row0 / p.mask_tile) * p.mask_x_ld + c0 / 64;
                const long long iw = (long long)(c0 / p.mask_tile) * p.mask_w_ld + store_row0 / 64;
                if (dbg_ok(c0 / 64 < p.mask_x_ld && ix < p.mask_x_bytes, p.err_word))
                  p.mask_x_out[ix] = 1;
                if (dbg_ok(store_row0 / 64 < p.mask_w_ld && iw < p.mask_w_bytes, p.err_word))
                  p.mask_w_out[iw] = 1;
              }
            }
            staged_store(stag0 + (nstore++ & 1u) * STAGING_BUF_BYTES, staging, lane, w, &tmOut,
                         c0, store_row0, false);
          }
        } else {  // kStore
#pragma unroll 1
          for (int sl = 0; sl < BN / 32; ++sl) {
            const int c0 = nb * BN + sl * 32;
            if (c0 >= p.n_size) break;  // warp-uniform
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + sl * 32, r);
            tmem_ld_wait_regs(r);
            if (EXT && num_kb == 0) {  // every token block skipped: the product is zero
#pragma unroll
              for (int j = 0; j < 32; ++j) r[j] = 0u;
            }
            staged_store(stag0 + (nstore++ & 1u) * STAGING_BUF_BYTES, staging, lane, r, &tmOut,
                         c0, store_row0, p.reduce_add != 0);
          }
        }

        // Release the accumulator buffer to the MMA warp (the leader's barrier).
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), lrank));
          else
            mbar_arrive(&tempty[acc]);
        }
        ++tile;
      }

      if constexpr (EPI == Epi::kLse) {
        if (ok && dbg_ok(g < p.n_groups && row < p.m_pad, p.err_word))
          p.partials[(size_t)g * p.m_pad + row] = make_float4(m2, ssum, zy, zsum);
      }
    }
    if constexpr (EPI != Epi::kLse) {
      if (lane == 0) bulk_wait_group<0>();
      __syncwarp();
    }
  }

  __syncthreads();
  if constexpr (PAIR) {
    if (*abort_flag) {
      // After an abort the peer's loads into this CTA may still be landing
      // (they signal the leader's barrier, which this CTA cannot wait on).
      const uint64_t t0 = global_timer_ns();
      while (global_timer_ns() - t0 < 200000ull) {
      }
    }
    tc_fence_before();
    cluster_sync_all();  // all pair MMAs and remote arrivals are done
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
  } else {
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem_base, TMEM_COLS);
    }
  }
}

template <Epi EPI, bool A_MN, bool B_MN, int STAGES, bool EXT = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmOut, const GemmParams p) {
  gemm_body<EPI, A_MN, B_MN, STAGES, 1, EXT>(tmA, tmB, tmOut, p);
}

template <Epi EPI, bool A_MN, bool B_MN, int STAGES, bool EXT = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmOut, const GemmParams p) {
  gemm_body<EPI, A_MN, B_MN, STAGES, 2, EXT>(tmA, tmB, tmOut, p);
}

// CTA pairs without compile-time cluster dimensions: launched with 2-CTA
// clusters required and 4-CTA clusters preferred (QUAD above).
template <Epi EPI, bool A_MN, bool B_MN, int STAGES, bool SHARE_B>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_quad_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmOut, const GemmParams p) {
  gemm_body<EPI, A_MN, B_MN, STAGES, 4, false, SHARE_B>(tmA, tmB, tmOut, p);
}

}  // namespace flce
