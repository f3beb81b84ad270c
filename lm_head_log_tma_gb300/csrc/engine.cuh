// Persistent, warp-specialised tcgen05 GEMM engine for sm_103a.
//
//   warp 0 (one lane)  : TMA producer, fills a ring of shared-memory stages
//   warp 1 (one lane)  : MMA issuer, tcgen05.mma into one of P::kAccBufs TMEM
//                        accumulators (128 lanes x BN fp32 columns each), or,
//                        with P::kSubs == 2, into one accumulator made of two
//                        column halves ("subs") that share the A operand
//   warp 2             : TMEM allocation / release
//   warps 4..11        : epilogue; warp w reads TMEM lanes 32*(w%4)..+31 and
//                        column half (w-4)/4 of the accumulator
//
// Pair mode (P::kPair == 2, launched as clusters of 2 CTAs): one tile is
// 256 rows; each CTA loads its own 128 rows of A and its half of the B rows
// into its own shared memory, and holds its 128 rows of the accumulator in
// its own TMEM.  The leader CTA (rank 0) issues cta_group::2 MMAs over both
// CTAs' operands.  TMA completions of both CTAs are counted on the leader's
// "full" barriers; the leader's commits release both CTAs' stages and
// accumulators (multicast); both CTAs' epilogues report a drained
// accumulator on the leader's "empty" barrier.
//
// Split accumulator (P::kSubs == 2): the epilogue drains sub 0, releases
// it, then drains sub 1.  The MMA issuer starts the next tile on sub 0 as soon
// as sub 0 is free and holds back sub 1's MMAs, keeping their stages, until
// sub 1 is free too (at most kStages k-blocks behind); so the tensor pipe
// idles only while half of the accumulator is read out, and one A tile feeds
// twice the columns of a double-buffered accumulator of the same TMEM size.
//
// A policy class supplies the tile schedule, the TMA loads of one k-block,
// the shared-memory descriptors of one K=16 step and the epilogue.  Every
// wait is bounded (see mbar_wait); when one role gives up, the others stop at
// their next wait, in-flight copies and MMAs are drained, TMEM is released
// and the kernel returns with RLLOSS_DEV_ETIMEOUT in the status word.
#pragma once
#include "ptx.cuh"

namespace rl {

constexpr int kEngineThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;

struct TileInfo {
  int m0;        // first row of the accumulator tile (A rows; 256 per tile in pair mode)
  int n0;        // first column of the accumulator (B rows)
  int kb_begin;  // k-block range
  int kb_end;
  int unit;      // policy-defined work-unit id
  int seg;       // policy-defined segment id
  bool first;    // first tile of its unit
  bool last;     // last tile of its unit
  int aux = 0;   // policy-defined (dX/dW: k-blocks per product term; forward: vocabulary segments)
  int slot = 0;  // forward: slot of the row tile in the launch's tile order
  int wide = 0;  // dX/dW: 1 when the tile's second sub is widened (set by the schedule)
};

// Wait that ignores the abort flag; used only to drain in-flight work.
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

__device__ __forceinline__ void spin_ns(uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < ns) {
  }
}

template <class P>
__host__ __device__ constexpr int engine_smem_bytes() {
  return 1024 /*alignment slack*/ + P::kStages * (P::kABytes + P::kBBytes) + 1024 /*barriers*/ +
         P::kExtraSmem;
}

// MMA issuer for a split accumulator (see the header).  Sub s lives at TMEM
// column s * P::kBN.  Returns false if a wait gave up.
template <class P>
__device__ bool mma_split_subs(const typename P::Params& prm, uint8_t* smem, uint64_t* full, uint64_t* empty,
                               uint64_t* tfull, uint64_t* tempty, uint32_t tmem, const AbortCtl& ac) {
  constexpr bool kPair = P::kCluster == 2;
  constexpr int S = P::kStages;
  constexpr int SB = P::kABytes + P::kBBytes;
  int stage = 0;
  uint32_t ph = 0;
  uint32_t aph = 0;
  auto release = [&](int s) {
    if constexpr (kPair)
      umma_commit_pair_mc(&empty[s], 0x3);
    else
      umma_commit(&empty[s]);
  };
  // Sub-1 MMAs of k-blocks j0..j1-1 of the tile, held in stages from s0.
  auto catch_up = [&](const TileInfo& t, int s0, int j0, int j1) {
    int s = s0;
    for (int j = j0; j < j1; ++j) {
      const uint32_t sa = smem_u32(smem + s * SB);
#pragma unroll
      for (int k = 0; k < P::kK16; ++k) P::mma(prm, tmem + uint32_t(P::kBN), sa, k, t, 1, (j > 0 || k > 0) ? 1u : 0u);
      release(s);
      if (++s == S) s = 0;
    }
  };
  bool ok = true;
  P::for_each_tile(prm, [&](const TileInfo& t) -> bool {
    if (!mbar_wait(&tempty[0], aph ^ 1u, ac)) { ok = false; return false; }
    tc_fence_after();
    bool ready1 = false;
    int lag = 0;
    const int s0 = stage;
    for (int kb = t.kb_begin; kb < t.kb_end; ++kb) {
      if (!mbar_wait(&full[stage], ph, ac)) { ok = false; return false; }
      tc_fence_after();
      const uint32_t sa = smem_u32(smem + stage * SB);
      const int j = kb - t.kb_begin;
#pragma unroll
      for (int k = 0; k < P::kK16; ++k) P::mma(prm, tmem, sa, k, t, 0, (j > 0 || k > 0) ? 1u : 0u);
      if (!ready1) {
        if (lag + 1 == S) {
          // Every stage is held for sub 1: wait for it to be drained.
          if (!mbar_wait(&tempty[1], aph ^ 1u, ac)) { ok = false; return false; }
          ready1 = true;
        } else {
          ready1 = mbar_try_wait(smem_u32(&tempty[1]), aph ^ 1u);
        }
        if (ready1) {
          tc_fence_after();
          catch_up(t, s0, 0, lag);
          lag = 0;
        }
      }
      if (ready1) {
#pragma unroll
        for (int k = 0; k < P::kK16; ++k) P::mma(prm, tmem + uint32_t(P::kBN), sa, k, t, 1, (j > 0 || k > 0) ? 1u : 0u);
        release(stage);
      } else {
        ++lag;
      }
      if (++stage == S) {
        stage = 0;
        ph ^= 1u;
      }
    }
    if (!ready1) {
      if (!mbar_wait(&tempty[1], aph ^ 1u, ac)) { ok = false; return false; }
      tc_fence_after();
      catch_up(t, s0, 0, lag);
    }
    if constexpr (kPair)
      umma_commit_pair_mc(&tfull[0], uint16_t(0x3u << (cluster_ctarank() & ~1u)));
    else
      umma_commit(&tfull[0]);
    aph ^= 1u;
    return true;
  });
  return ok;
}

template <class P>
__global__ void __launch_bounds__(kEngineThreads, 1) tc_engine_kernel(const __grid_constant__ typename P::Params prm) {
  static_assert(P::kAccBufs * P::kBN <= int(kTmemCols), "accumulators exceed TMEM");
  static_assert(P::kSubs == 1 || (P::kSubs == 2 && P::kAccBufs == 1), "a split accumulator is single-buffered");
  static_assert(P::kCluster == 1 || P::kCluster == 2, "single CTAs or CTA pairs");
  constexpr bool kPair = P::kCluster == 2;
  // Work sizes read on the device (rows left for this launch) are the same for
  // every CTA: a launch with nothing to do returns before any setup.
  if (!P::has_work(prm)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int S = P::kStages;
  constexpr int SB = P::kABytes + P::kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * SB);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = bars + 2 * S + 2;
  uint64_t* drain = bars + 2 * S + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  int* abort_i = reinterpret_cast<int*>(tmem_slot + 1);
  uint8_t* extra = smem + S * SB + 1024;   // 1024-aligned policy scratch

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const uint32_t leader = rank & ~1u;             // pair leader (issues the MMAs)
  const bool is_leader = (rank & 1u) == 0u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kEpiWarps * (kPair ? 2 : 1));
    }
    mbar_init(drain, 1);
    *abort_i = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    if constexpr (kPair) {
      tmem_alloc_pair(tmem_slot, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
  }
  P::cta_setup(prm, extra);
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const AbortCtl ac{abort_i, prm.status, prm.limit_ns};
  bool aborted = false;

  if (warp == 0) {
    if (lane == 0) {
      P::prefetch(prm);
      int stage = 0;
      uint32_t ph = 0;
      int issued = 0;
      P::for_each_tile(prm, [&](const TileInfo& t) -> bool {
        for (int kb = t.kb_begin; kb < t.kb_end; ++kb) {
          if (!mbar_wait(&empty[stage], ph ^ 1u, ac)) { aborted = true; return false; }
          const uint32_t fb = smem_u32(&full[stage]);
          if (is_leader) mbar_expect_tx(&full[stage], (kPair ? 2 : 1) * P::tx_bytes(prm, t));
          P::load(prm, smem + stage * SB, kPair ? mapa_shared(fb, leader) : fb, t, kb, rank);
          ++issued;
          if (++stage == S) {
            stage = 0;
            ph ^= 1u;
          }
        }
        return true;
      });
      if (aborted) {
        // Let every copy this thread started land before the CTA can exit.
        if (is_leader) {
          for (int j = 0; j < S && j < issued; ++j) {
            if (--stage < 0) {
              stage = S - 1;
              ph ^= 1u;
            }
            mbar_wait_drain(&full[stage], ph, 20000000ull);
          }
        } else {
          spin_ns(2000000ull);   // the peer's copies are counted on the leader's barriers
        }
      }
    }
  } else if (warp == 1) {
    if constexpr (P::kSubs == 2) {
      if (lane == 0 && is_leader) aborted = !mma_split_subs<P>(prm, smem, full, empty, tfull, tempty, tmem, ac);
      if (aborted) {
        if constexpr (kPair)
          umma_commit_pair(drain);
        else
          umma_commit(drain);
        mbar_wait_drain(drain, 0, 20000000ull);
      }
    } else if (lane == 0 && is_leader) {
      int stage = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t aph = 0;
      P::for_each_tile(prm, [&](const TileInfo& t) -> bool {
        if (!mbar_wait(&tempty[acc], aph ^ 1u, ac)) { aborted = true; return false; }
        tc_fence_after();
        const uint32_t d = tmem + uint32_t(acc * P::kBN);
        for (int kb = t.kb_begin; kb < t.kb_end; ++kb) {
          if (!mbar_wait(&full[stage], ph, ac)) { aborted = true; return false; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * SB);
#pragma unroll
          for (int k = 0; k < P::kK16; ++k) P::mma(prm, d, sa, k, t, (kb > t.kb_begin || k > 0) ? 1u : 0u);
          if constexpr (kPair)
            umma_commit_pair_mc(&empty[stage], 0x3);
          else
            umma_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if constexpr (kPair)
          umma_commit_pair_mc(&tfull[acc], uint16_t(0x3u << leader));
        else
          umma_commit(&tfull[acc]);
        if (++acc == P::kAccBufs) {
          acc = 0;
          aph ^= 1u;
        }
        return true;
      });
      if (aborted) {
        if constexpr (kPair)
          umma_commit_pair(drain);
        else
          umma_commit(drain);
        mbar_wait_drain(drain, 0, 20000000ull);
      }
    }
  } else if (warp >= kEpiWarp0) {
    const int q = warp & 3;
    const int half = (warp - kEpiWarp0) >> 2;
    int acc = 0;
    uint32_t aph = 0;
    typename P::EpiState st;
    if constexpr (P::kSubs == 2) {
      P::for_each_tile(prm, [&](const TileInfo& t) -> bool {
        const bool got = mbar_wait(&tfull[0], aph, ac);
        if (!__all_sync(0xffffffffu, got)) return false;
        tc_fence_after();
#pragma unroll 1
        for (int sub = 0; sub < 2; ++sub) {
          P::epilogue(prm, st, t, tmem + uint32_t(sub * P::kBN) + (uint32_t(q * 32) << 16), q, half, lane, extra,
                      rank, sub);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (kPair)
              mbar_arrive_remote(mapa_shared(smem_u32(&tempty[sub]), leader));
            else
              mbar_arrive(&tempty[sub]);
          }
        }
        aph ^= 1u;
        return true;
      });
    } else
    P::for_each_tile(prm, [&](const TileInfo& t) -> bool {
      const bool got = mbar_wait(&tfull[acc], aph, ac);
      if (!__all_sync(0xffffffffu, got)) return false;
      tc_fence_after();
      P::epilogue(prm, st, t, tmem + uint32_t(acc * P::kBN) + (uint32_t(q * 32) << 16), q, half, lane, extra, rank);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kPair)
          mbar_arrive_remote(mapa_shared(smem_u32(&tempty[acc]), leader));
        else
          mbar_arrive(&tempty[acc]);
      }
      if (++acc == P::kAccBufs) {
        acc = 0;
        aph ^= 1u;
      }
      return true;
    });
    P::epilogue_finish(prm, lane);
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();
  tc_fence_after();
  if (warp == 2) {
    if constexpr (kPair)
      tmem_dealloc_pair(tmem, kTmemCols);
    else
      tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace rl
