// Merged backward launch: the weight- and input-gradient GEMMs of one
// vocabulary chunk and the dZ recompute of the next chunk in one persistent
// CTA-pair kernel.
//
// Why: run as three launches per chunk, each GEMM ends on a partial wave (at
// the Llama-3 shape the dW and dX launches have 13.5 and 6.7 waves of
// 256 x 256 tiles over 76 CTA pairs, so ~4% of each launch runs on part of the
// GPU), and every launch pays its own pipeline fill and drain.  Here the tiles
// of all three GEMMs ("Backward Hidden and Weight Accumulation" for chunk c,
// "Mathematical Mechanics ...", step 3 for chunk c+1) form one list, ordered
// by k-loop length (longest first).  The first `static_tiles` tiles go round
// robin (pair p takes p, p + P, ...), so all pairs walk neighbouring tiles in
// step and share their operands in L2; the last few rounds are handed out
// dynamically from a global counter as pairs free up, so one launch ends
// within about one short tile of perfect balance.  (Handing out every tile
// dynamically balanced as well but ran the tiles ~3% slower on a GB300.)
//
//   kind  D                 A (MMA view)        B (MMA view)       epilogue
//   dW    dW[v0:v0+w, :]    dZ_c^T (MN-major)   X (MN-major)       fp32 store / reduce-add
//   dX    dX_acc            dZ_c (K-major)      W_c (MN-major)     fp32 store / reduce-add
//   dZ    dZ_{c+1}          X (K-major)         W_{c+1} (K-major)  dZ (bf16), written into
//                                                                  the other dZ buffer
//
// Each output tile is still computed by exactly one pair over the same
// ascending k-blocks with the same MMA shape as in the separate launches, so
// the results are bit-identical to them and deterministic.
//
// Dynamic hand-out inside a pair: the leader's producer thread takes a tile
// index with atomicAdd, writes it into a ring of SCHED_SLOTS slots in both
// CTAs' shared memory and arrives (release, cluster scope) on each CTA's
// sched_full barrier of that slot.  The readers -- the peer's producer, the leader's MMA
// thread and the eight epilogue warps of the pair -- read the index after an
// acquire-scope wait and arrive on the leader's sched_empty barrier; the
// leader reuses the slot once all ten have read it.  An index >= the tile
// count ends every role's loop.  Every wait is bounded (see mbar_wait).
#pragma once
#include "gemm_core.cuh"

namespace flce {

enum FusedKind : int { kFusedDw = 0, kFusedDx = 1, kFusedDz = 2 };
constexpr int FUSED_MAX_SEGS = 3;
constexpr int SCHED_SLOTS = 4;
constexpr int FUSED_BARRIER_BYTES = 512;
constexpr int SCHED_READERS = 1 + 1 + 2 * NUM_EPI_WARPS;  // peer producer, MMA, epilogue warps
constexpr int DYNAMIC_ROUNDS = 3;  // rounds of tiles (one per pair) at the end handed out dynamically

// One segment of the tile list: all tiles of one GEMM.
struct FusedSeg {
  int kind;        // FusedKind
  int first;       // index of the segment's first tile in the launch's list
  int num_tiles;   // m_blocks * n_blocks
  int m_size;      // rows of D
  int n_size;      // columns of D (store clipping)
  int k_size;      // contraction length
  int m_blocks;    // ceil(m_size / 256)
  int n_blocks;    // ceil(n_size / 256)
  int m_fastest;   // 1: consecutive tiles walk row blocks; 0: walk column blocks
  int m_band;      // m_fastest: row blocks walked in bands of this many (0 = all)
  int n_band;      // !m_fastest: column blocks walked in bands of this many (0 = all)
  int reduce_add;  // dW / dX: 1 = TMA reduce-add onto the output, 0 = overwrite
};

struct FusedParams {
  FusedSeg seg[FUSED_MAX_SEGS];  // in list order (ascending `first`)
  int n_seg;
  int total_tiles;
  int static_tiles;              // tiles [0, static_tiles) go round robin; a multiple of the pairs
  int* tile_counter;             // global; 0 before the launch (counts the dynamic tiles)
  // dZ epilogue (chunk c+1)
  const int64_t* labels;
  long long ignore_index;
  int vocab;                     // V of the softmax
  int col_base;                  // vocabulary index of the chunk's column 0
  int col_limit;                 // chunk width
  float smoothing;
  float z_loss;
  const float* lse;
  const float* scale;            // device scalar c = grad / N_valid
  int* err_word;
  unsigned long long timeout_ns;
};

// Tensor maps, indexed by FusedKind.
struct FusedMaps {
  CUtensorMap a[3];
  CUtensorMap b[3];
  CUtensorMap out[3];
};

template <int STAGES>
constexpr int fused_smem_bytes() {
  return STAGES * TileCfg<true>::STAGE + STAGING_BYTES + FUSED_BARRIER_BYTES + 1024;
}

struct FusedTile {
  int kind, mb, nb, num_kb, seg;
};

__device__ __forceinline__ FusedTile fused_tile(const FusedParams& p, int t) {
  int si = 0;
  while (si + 1 < p.n_seg && t >= p.seg[si + 1].first) ++si;
  const FusedSeg& s = p.seg[si];
  int l = t - s.first;
  if (!dbg_ok(l >= 0 && l < s.num_tiles, p.err_word)) l = 0;
  int mb, nb;
  if (s.m_fastest) {
    if (s.m_band > 0 && s.m_band < s.m_blocks) {
      const int band_units = s.m_band * s.n_blocks;
      const int band = l / band_units;
      const int ub = l - band * band_units;
      const int mb0 = band * s.m_band;
      const int mbn = min(s.m_band, s.m_blocks - mb0);
      mb = mb0 + ub % mbn;
      nb = ub / mbn;
    } else {
      mb = l % s.m_blocks;
      nb = l / s.m_blocks;
    }
  } else if (s.n_band > 0 && s.n_band < s.n_blocks) {
    const int band_units = s.n_band * s.m_blocks;
    const int band = l / band_units;
    const int ub = l - band * band_units;
    const int nb0 = band * s.n_band;
    const int nbn = min(s.n_band, s.n_blocks - nb0);
    nb = nb0 + ub % nbn;
    mb = ub / nbn;
  } else {
    nb = l % s.n_blocks;
    mb = l / s.n_blocks;
  }
  // debug build: a tile outside its GEMM's grid is replaced by tile (0, 0)
  if (!dbg_ok(mb >= 0 && mb < s.m_blocks && nb >= 0 && nb < s.n_blocks, p.err_word)) {
    mb = 0;
    nb = 0;
  }
  return {s.kind, mb, nb, (s.k_size + BK - 1) / BK, si};
}

// Producer side of one tile: the k-block loads of A and B (this CTA's halves)
// into the stage ring.  The operand layouts are template arguments, so each
// kind's k-loop is compiled like the separate kernels' loops.
template <bool A_MN, bool B_MN, int STAGES>
__device__ __forceinline__ bool fused_load_tile(const CUtensorMap* ma, const CUtensorMap* mbm,
                                                int a_row, int b_row, int num_kb,
                                                uint8_t* stages, uint64_t* full,
                                                uint64_t* empty, uint32_t rank, uint32_t& it,
                                                const WaitCtx& ctx) {
  using Cfg = TileCfg<true>;
  for (int kb = 0; kb < num_kb; ++kb) {
    const int s = it % STAGES;
    const uint32_t r = it / STAGES;
    if (!mbar_wait(&empty[s], (r & 1u) ^ 1u, ctx)) return false;
    uint8_t* a_dst = stages + s * Cfg::STAGE;
    uint8_t* b_dst = a_dst + Cfg::A_STAGE;
    // Both CTAs' loads complete on the leader's full barrier, which only the
    // leader arms with the pair's byte count.
    const uint32_t bar = mapa_shared(smem_u32(&full[s]), 0);
    if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * Cfg::STAGE);
    if constexpr (!A_MN) {
      tma_load_2d_pair(a_dst, ma, bar, kb * BK, a_row);
    } else {
#pragma unroll
      for (int i = 0; i < BM / 64; ++i)
        tma_load_2d_pair(a_dst + i * MN_BOX_BYTES, ma, bar, a_row + i * 64, kb * BK);
    }
    if constexpr (!B_MN) {
      tma_load_2d_pair(b_dst, mbm, bar, kb * BK, b_row);
    } else {
#pragma unroll
      for (int i = 0; i < Cfg::B_ROWS / 64; ++i)
        tma_load_2d_pair(b_dst + i * MN_BOX_BYTES, mbm, bar, b_row + i * 64, kb * BK);
    }
    ++it;
  }
  return true;
}

// MMA side of one tile (leader CTA, one thread): num_kb k-blocks of
// 256 x 256 x 64 into the accumulator at d_tmem.
template <bool A_MN, bool B_MN, int STAGES>
__device__ __forceinline__ bool fused_mma_tile(uint32_t d_tmem, int num_kb, uint8_t* stages,
                                               uint64_t* full, uint64_t* empty, uint32_t& it,
                                               const WaitCtx& ctx) {
  using Cfg = TileCfg<true>;
  constexpr uint32_t idesc = make_idesc(A_MN, B_MN, Cfg::TILE_M, BN);
  for (int kb = 0; kb < num_kb; ++kb) {
    const int s = it % STAGES;
    const uint32_t r = it / STAGES;
    if (!mbar_wait(&full[s], r & 1u, ctx)) return false;
    tc_fence_after();
    const uint32_t a_addr = smem_u32(stages + s * Cfg::STAGE);
    const uint32_t b_addr = a_addr + Cfg::A_STAGE;
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      // MN-major operand blocks are 64 elements wide, MN_BOX_BYTES apart; one
      // 16-deep k step is 2048 bytes into them (K-major: 32 bytes).
      const uint64_t ad = A_MN ? smem_desc_sw128(a_addr + kk * 2048, MN_BOX_BYTES, 1024)
                               : smem_desc_sw128(a_addr + kk * 32, 16, 1024);
      const uint64_t bd = B_MN ? smem_desc_sw128(b_addr + kk * 2048, MN_BOX_BYTES, 1024)
                               : smem_desc_sw128(b_addr + kk * 32, 16, 1024);
      mma_issue_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
    }
    mma_commit_pair_multicast(&empty[s], 0x3);
    ++it;
  }
  return true;
}

template <int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    bwd_fused_kernel(const __grid_constant__ FusedMaps maps,
                     const __grid_constant__ FusedParams p) {
  using Cfg = TileCfg<true>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  uint8_t* staging = smem + STAGES * Cfg::STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + STAGING_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint64_t* sfull = mma_done + 1;
  uint64_t* sempty = sfull + SCHED_SLOTS;  // used on the leader
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sempty + SCHED_SLOTS);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  volatile int* sched = abort_flag + 1;  // SCHED_SLOTS tile indices

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 = leader (issues the MMAs, hands out tiles)

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * NUM_EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    for (int s = 0; s < SCHED_SLOTS; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], SCHED_READERS);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane < 9) {
    const CUtensorMap* m =
        lane < 3 ? &maps.a[lane] : (lane < 6 ? &maps.b[lane - 3] : &maps.out[lane - 6]);
    prefetch_tensormap(m);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // the peer's barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtx ctx{abort_flag, p.err_word, p.timeout_ns};

  const int pair_id = (int)(blockIdx.x >> 1);
  const int num_pairs = (int)(gridDim.x >> 1);
  const uint32_t static_rounds = (uint32_t)(p.static_tiles / num_pairs);

  // The i-th tile of this pair, for the readers (every role but the leader's
  // producer): round robin in the static part, else the published index of
  // dynamic slot i - static_rounds.  Returns false on a timeout.
  auto next_tile = [&](uint32_t i, int& t) -> bool {
    if (i < static_rounds) {
      t = pair_id + (int)i * num_pairs;
      return true;
    }
    const uint32_t j = i - static_rounds;
    const uint32_t slot = j % SCHED_SLOTS;
    if (!mbar_wait_cluster(&sfull[slot], (j / SCHED_SLOTS) & 1u, ctx)) return false;
    t = sched[slot];
    mbar_arrive_cluster(mapa_shared(smem_u32(&sempty[slot]), 0));
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (uint32_t i = 0; ok; ++i) {
        int t;
        if (rank == 0 && i >= static_rounds) {
          // take the next dynamic tile and publish it into slot j (both CTAs)
          const uint32_t j = i - static_rounds;
          const uint32_t slot = j % SCHED_SLOTS;
          if (!mbar_wait_cluster(&sempty[slot], ((j / SCHED_SLOTS) & 1u) ^ 1u, ctx)) {
            ok = false;
            break;
          }
          t = p.static_tiles + atomicAdd(p.tile_counter, 1);
          sched[slot] = t;
          st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(&sched[slot])), 1),
                                (uint32_t)t);
          mbar_arrive_cluster(mapa_shared(smem_u32(&sfull[slot]), 0));
          mbar_arrive_cluster(mapa_shared(smem_u32(&sfull[slot]), 1));
        } else if (!next_tile(i, t)) {
          ok = false;
          break;
        }
        if (t >= p.total_tiles) break;
        const FusedTile ft = fused_tile(p, t);
        const CUtensorMap* ma = &maps.a[ft.kind];
        const CUtensorMap* mbm = &maps.b[ft.kind];
        const int a_row = ft.mb * Cfg::TILE_M + (int)rank * BM;
        const int b_row = ft.nb * BN + (int)rank * Cfg::B_ROWS;
        if (ft.kind == kFusedDw)
          ok = fused_load_tile<true, true, STAGES>(ma, mbm, a_row, b_row, ft.num_kb, stages, full,
                                                   empty, rank, it, ctx);
        else if (ft.kind == kFusedDx)
          ok = fused_load_tile<false, true, STAGES>(ma, mbm, a_row, b_row, ft.num_kb, stages,
                                                    full, empty, rank, it, ctx);
        else
          ok = fused_load_tile<false, false, STAGES>(ma, mbm, a_row, b_row, ft.num_kb, stages,
                                                     full, empty, rank, it, ctx);
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
      uint32_t it = 0, tile = 0;
      for (uint32_t i = 0;; ++i) {
        int t;
        if (!next_tile(i, t)) break;
        if (t >= p.total_tiles) break;
        const FusedTile ft = fused_tile(p, t);
        const uint32_t acc = tile & 1u;
        const uint32_t ra = tile >> 1;
        if (!mbar_wait(&tempty[acc], (ra & 1u) ^ 1u, ctx)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok;
        if (ft.kind == kFusedDw)
          ok = fused_mma_tile<true, true, STAGES>(d_tmem, ft.num_kb, stages, full, empty, it, ctx);
        else if (ft.kind == kFusedDx)
          ok = fused_mma_tile<false, true, STAGES>(d_tmem, ft.num_kb, stages, full, empty, it,
                                                   ctx);
        else
          ok = fused_mma_tile<false, false, STAGES>(d_tmem, ft.num_kb, stages, full, empty, it,
                                                    ctx);
        if (!ok) break;
        mma_commit_pair_multicast(&tfull[acc], 0x3);
        ++tile;
      }
      // Every MMA this thread issued must finish before TMEM is released.
      mma_commit_pair_multicast(mma_done, 0x1);
      mbar_wait_drain(mma_done, 0, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant of this warp
    const int row_in_tile = (int)rank * BM + q * 32 + lane;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t stag0 = smem_u32(staging) + (warp - 2) * 2 * STAGING_BUF_BYTES;
    const float c_scale = *p.scale;
    uint32_t tile = 0;
    uint32_t nstore = 0;  // this warp's staged stores so far: buffer nstore & 1
    for (uint32_t i = 0;; ++i) {
      int t = 0;
      bool got = true;
      if (lane == 0) got = next_tile(i, t);
      got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
      t = __shfl_sync(0xffffffffu, t, 0);
      if (!got || t >= p.total_tiles) break;
      const FusedTile ft = fused_tile(p, t);
      const FusedSeg& sg = p.seg[ft.seg];
      const int store_row0 = ft.mb * Cfg::TILE_M + (int)rank * BM + q * 32;

      const uint32_t acc = tile & 1u;
      const uint32_t ra = tile >> 1;
      if (!warp_wait(&tfull[acc], ra & 1u, ctx, lane)) break;
      tc_fence_after();
      const uint32_t taddr = lane_base + acc * BN;

      if (ft.kind == kFusedDz) {
        const int row = ft.mb * Cfg::TILE_M + row_in_tile;
        const bool row_ok = row < sg.m_size;
        const long long label = row_ok ? (long long)p.labels[row] : (long long)p.ignore_index;
        // out-of-range labels count as ignored (see the dZ epilogue of gemm_core.cuh)
        const bool valid =
            row_ok && label != p.ignore_index && label >= 0 && label < (long long)p.vocab;
        const long long lab_rel = label - p.col_base;
        const DzRow dzr =
            dz_row(valid, row_ok ? p.lse[row] : 0.f, c_scale, p.smoothing, p.z_loss, p.vocab);
#pragma unroll 1
        for (int sl = 0; sl < BN / 64; ++sl) {
          const int c0 = ft.nb * BN + sl * 64;
          if (c0 >= p.col_limit) break;  // warp-uniform; the store would be clipped anyway
          uint32_t w[32];
          dz_slice<false>(taddr + sl * 64, dzr, lab_rel - c0, w);
          staged_store(stag0 + (nstore++ & 1u) * STAGING_BUF_BYTES, staging, lane, w,
                       &maps.out[kFusedDz], c0, store_row0, false);
        }
      } else {
        const CUtensorMap* out = &maps.out[ft.kind];
#pragma unroll 1
        for (int sl = 0; sl < BN / 32; ++sl) {
          const int c0 = ft.nb * BN + sl * 32;
          if (c0 >= sg.n_size) break;  // warp-uniform
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + sl * 32, r);
          tmem_ld_wait_regs(r);
          staged_store(stag0 + (nstore++ & 1u) * STAGING_BUF_BYTES, staging, lane, r, out, c0,
                       store_row0, sg.reduce_add != 0);
        }
      }

      // Release the accumulator buffer to the MMA thread (the leader's barrier).
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
      ++tile;
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  __syncthreads();
  if (*abort_flag) {
    // After an abort the peer's loads into this CTA may still be landing
    // (they signal the leader's barrier, which this CTA cannot wait on).
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) {
    }
  }
  tc_fence_before();
  cluster_sync_all();  // all pair MMAs, remote arrivals and remote stores are done
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace flce
