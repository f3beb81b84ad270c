// Tensor-core kernels of the fused LM-head path.
//
//  fwd   : S = X W^T tile by tile (256 tokens x 256 vocab on a CTA pair, or
//          128 x 256 on one CTA; K = H), epilogue folds each tile into
//          per-row streaming log-softmax state (reference max,
//          sum 2^(t-m), sum 2^(t-m)(t-m), target logit) — "support
//          top_entropy_quantile in fused linear GRPO loss", Details (second
//          online accumulator next to the running max and sum).
//  merge : combines the partial row states of the vocabulary segments into
//          lse, logp and entropy per token.
//  dl    : recomputes S for a chunk of rows and writes
//          G = dL/dl = (c/tau)(onehot(y) - p) as bf16 (p = softmax(S/tau)),
//          keeping each row's target-entry rounding error in fp32, the
//          db column partials when there is a bias.
//  gemmH : D[row][h] = sum_k A[row][k] B[h][k] on CTA pairs, 256 rows x 448 h
//          per tile (two 224-h halves sharing each A tile): dX = G W
//          (k = vocab; the target-entry error times W[target] added back,
//          rows of the compacted backward added in place into dX) and
//          dW = G^T X (k = tokens) in one grouped launch.
#include <cuda_runtime.h>

#include "engine.cuh"
#include "merge_row.cuh"
#include "kernels.h"

namespace rl {

// One 32-row x 32-column bf16 box (this lane's 64-byte row w) leaves through
// a per-warp staging buffer (two alternate, 64-byte swizzle) and a TMA store
// to columns x.., rows y.. of map m.
constexpr int kBf16BoxBytes = 32 * 64;
// zero_col in [0, 32): that element of this lane's row is written as 0.
__device__ __forceinline__ void store_bf16_box(const CUtensorMap* m, int* status, uint8_t* wbuf, int& nbuf,
                                               int lane, const uint32_t (&w)[16], int x, int y,
                                               unsigned zero_col = ~0u) {
  uint8_t* buf = wbuf + (nbuf & 1) * kBf16BoxBytes;
  if (lane == 0) tma_store_wait_read<1>();
  __syncwarp();
  const int sw = (lane >> 1) & 3;
  uint4* row = reinterpret_cast<uint4*>(buf + lane * 64);
#pragma unroll
  for (int c = 0; c < 4; ++c) row[c ^ sw] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  if (zero_col < 32u)
    *reinterpret_cast<uint16_t*>(buf + lane * 64 + ((int(zero_col >> 3) ^ sw) << 4) + (zero_col & 7u) * 2) = 0;
  fence_proxy_async();
  __syncwarp();
  if (lane == 0) {
    if (tma_x_ok<2>(x, status)) tma_store_2d(m, buf, x, y);
    tma_store_commit();
  }
  ++nbuf;
}

// A 32-row x 64-column bf16 box (128-byte rows, 128-byte swizzle: 16-byte
// chunk k of row r sits at chunk k ^ (r % 8)), filled from two 32-column halves
// and stored with one TMA store; one such buffer per warp.  stage_half writes
// this lane's 32 columns as half h; zero_col in [0, 32) writes that column of
// the half as 0.  Before half 0 the previous box's store must have finished
// reading the buffer.
constexpr int kBf16Box64Bytes = 32 * 128;
__device__ __forceinline__ void stage_half(uint8_t* buf, int lane, const uint32_t (&w)[16], int h,
                                           unsigned zero_col) {
  if (h == 0) {
    if (lane == 0) tma_store_wait_read<0>();
    __syncwarp();
  }
  uint4* row = reinterpret_cast<uint4*>(buf + lane * 128);
  const int sw = lane & 7;
#pragma unroll
  for (int c = 0; c < 4; ++c) row[(4 * h + c) ^ sw] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  if (zero_col < 32u)
    *reinterpret_cast<uint16_t*>(buf + lane * 128 + (((4 * h + int(zero_col >> 3)) ^ sw) << 4) +
                                 (zero_col & 7u) * 2) = 0;
}
__device__ __forceinline__ void store_box64(const CUtensorMap* m, int* status, uint8_t* buf, int lane, int x, int y) {
  fence_proxy_async();
  __syncwarp();
  if (lane == 0) {
    if (tma_x_ok<2>(x, status)) tma_store_2d(m, buf, x, y);
    tma_store_commit();
  }
}

// =============================================================== forward
// CL = 1: 128-row tiles on one CTA; CL = 2: 256-row tiles over a CTA pair
// (cta_group::2).  F8: e4m3 operands (forward-only scoring) with per-row
// scales of X and W applied in the epilogue; a 128-byte box row is then 128
// elements and each MMA step covers K = 32.  KBX: 128-byte boxes per operand
// in a pipeline stage (2 for pair tiles with one K segment: half as many,
// twice as deep stages, which halves the per-stage barrier round trips the
// MMA issuer waits on — measured 9% on the bf16 forward).  ST: the tiles of
// the first FwdParams::pu_tiles row-tile slots also write every logit's
// unnormalised probability 2^t as bf16 (stored probabilities, for a backward
// that needs no recompute; bf16 CTA pairs without bias).
template <int CL, bool F8 = false, int KBX = 1, bool ST = false>
struct FwdPolicy {
  static constexpr int kCluster = CL;
  static constexpr int PAIR = CL >= 2 ? 2 : 1;
  static constexpr int kRows = 128 * CL;             // accumulator rows per tile (whole cluster)
  static constexpr int kStages = (PAIR == 2 ? 6 : 4) / KBX;
  static constexpr int kSubs = 1;
  static constexpr int kBN = 256;
  static constexpr int kK16 = 4 * KBX;
  static constexpr int kBox = 128 * 128;                    // one 128-row x 128-byte operand box
  static constexpr int kABytes = kBox * KBX;
  static constexpr int kBBytes = (256 / PAIR) * 128 * KBX;   // this CTA's share of the B rows
  static constexpr int kColBytes = 2 * 128 * 4;   // per epilogue warp: its 128 columns' W scales and biases
  // ST: one 32 x 64 staging box per epilogue warp instead (no bias, no scales)
  static constexpr int kExtraSmem = ST ? kEpiWarps * 2 * kBf16BoxBytes : kEpiWarps * kColBytes;
  static_assert(!ST || (CL == 2 && !F8), "stored probabilities: bf16 CTA-pair forward");
  static constexpr uint32_t kIdesc = F8 ? idesc_e4m3(kRows, 256) : idesc_bf16(kRows, 256, 0, 0);
  static constexpr int kKB = (F8 ? 128 : 64) * KBX;   // K elements per k-block
  using Params = FwdParams;

  struct EpiState {
    float mref, s_hi, s_lo, w_hi, w_lo, zy;
    int found, y;
    float xs;     // F8: this row's X scale
    // Per-column vectors (W scales, bias) of this warp's 128 columns, loaded
    // one tile ahead so their L2 latency hides behind the current tile.
    float4 pw, pb;
    int pre_n0 = -1;       // tile whose columns pw / pb hold
    int R = -1, P = 0;     // launch shape (for the next tile's columns)
    int nbuf = 0;          // ST: staging boxes used so far (two alternate)
  };

  // Row tiles and vocabulary segments of this launch: all R tiles with the
  // host's P, or the listed tiles with P chosen here for their count.
  __device__ static void shape(const Params& p, int& R, int& P) {
    if (p.tiles) {
      R = *p.ntiles;
      P = choose_segments(R, p.Vt, int(gridDim.x) / CL, p.pcap);
    } else {
      R = p.R;
      P = p.P;
    }
  }
  __device__ static bool has_work(const Params&) { return true; }   // writes P_out even without tiles
  __device__ static void cta_setup(const Params& p, uint8_t*) {
    if (p.P_out && blockIdx.x == 0 && threadIdx.x == 0) {
      int R, P;
      shape(p, R, P);
      *p.P_out = P;
    }
  }
  __device__ static void prefetch(const Params& p) {
    tma_prefetch_desc(&p.tmA);
    tma_prefetch_desc(&p.tmB);
    if constexpr (ST) tma_prefetch_desc(&p.tmPu);
  }

  // Units u = seg * R + r (row tile r, vocabulary segment seg), dealt
  // round-robin to the CTAs so that CTAs running at the same time share the
  // same W tiles (L2 reuse) while each keeps its own rows.
  template <class F>
  __device__ static void for_each_tile(const Params& p, F&& f) {
    int R, P;
    shape(p, R, P);
    const int units = R * P;
    const int kbs = p.nseg * p.kb_per_seg;
    const int g0 = blockIdx.x / CL, gn = gridDim.x / CL;
    for (int u = g0; u < units; u += gn) {
      const int seg = u / R;
      const int ri = u - seg * R;
      const int r = p.tiles ? p.tiles[ri] : ri;
      const int j0 = int((long long)seg * p.Vt / P);
      const int j1 = int((long long)(seg + 1) * p.Vt / P);
      for (int j = j0; j < j1; ++j) {
        TileInfo t{r * kRows, j * 256, 0, kbs, u, seg, j == j0, j == j1 - 1, P};
        t.slot = ri;
        if (!f(t)) return;
      }
    }
  }

  __device__ static void load(const Params& p, uint8_t* st, uint32_t bar, const TileInfo& t, int kb, uint32_t rank) {
    const int s = kb / p.kb_per_seg;
    const int kk = (kb - s * p.kb_per_seg) * kKB;
    if constexpr (CL == 2) {
      constexpr int kBoxK = kKB / KBX;   // K elements of one 128-byte box row
#pragma unroll
      for (int x = 0; x < KBX; ++x) {
        constexpr int EB = F8 ? 1 : 2;
        if (tma_x_ok<EB>(p.seg_a[s] + kk + kBoxK * x, p.status))
          tma_load_2d_pair(&p.tmA, bar, st + x * kBox, p.seg_a[s] + kk + kBoxK * x, t.m0 + 128 * int(rank));
        if (tma_x_ok<EB>(p.seg_b[s] + kk + kBoxK * x, p.status))
          tma_load_2d_pair(&p.tmB, bar, st + kABytes + x * kBox, p.seg_b[s] + kk + kBoxK * x, t.n0 + 128 * int(rank));
      }
    } else {
      static_assert(KBX == 1, "single-CTA tiles keep one box per operand");
      if (tma_x_ok<F8 ? 1 : 2>(p.seg_a[s] + kk, p.status)) tma_load_2d(&p.tmA, bar, st, p.seg_a[s] + kk, t.m0);
      if (tma_x_ok<F8 ? 1 : 2>(p.seg_b[s] + kk, p.status)) tma_load_2d(&p.tmB, bar, st + kABytes, p.seg_b[s] + kk, t.n0);
    }
  }
  // MMA step k (32 bytes of K each) of the stage: box k / 4, byte offset 32 (k % 4).
  __device__ static uint64_t adesc(uint32_t sa, int k, const TileInfo&) {
    return sdesc_sw128(sa + (k >> 2) * kBox + (k & 3) * 32, 16, 1024);
  }
  __device__ static uint64_t bdesc(uint32_t sa, int k, const TileInfo&) {
    return sdesc_sw128(sa + kABytes + (k >> 2) * kBox + (k & 3) * 32, 16, 1024);
  }
  __device__ static uint32_t idesc(const TileInfo&) { return kIdesc; }
  static constexpr int kAccBufs = 2;
  __device__ static uint32_t tx_bytes(const Params&, const TileInfo&) { return kABytes + kBBytes; }
  __device__ static void mma(const Params&, uint32_t d, uint32_t sa, int k, const TileInfo& t, uint32_t accum) {
    if constexpr (F8) {
      if constexpr (PAIR == 2)
        umma_e4m3_pair(d, adesc(sa, k, t), bdesc(sa, k, t), kIdesc, accum);
      else
        umma_e4m3(d, adesc(sa, k, t), bdesc(sa, k, t), kIdesc, accum);
    } else if constexpr (PAIR == 2) {
      umma_bf16_pair(d, adesc(sa, k, t), bdesc(sa, k, t), kIdesc, accum);
    } else {
      umma_bf16(d, adesc(sa, k, t), bdesc(sa, k, t), kIdesc, accum);
    }
  }

  // First column of the tile this CTA's epilogue handles after t (-1: none).
  __device__ static int next_tile_n0(const Params& p, EpiState& e, const TileInfo& t) {
    if (!t.last) return t.n0 + 256;
    if (e.R < 0) shape(p, e.R, e.P);
    const int u = t.unit + int(gridDim.x) / CL;
    if (u >= e.R * e.P) return -1;
    return int((long long)(u / e.R) * p.Vt / e.P) * 256;
  }
  // This lane's 4 of the warp's 128 column scales / biases of the tile at n0
  // (the vectors are padded to whole 256-column tiles).
  __device__ static void fetch_cols(const Params& p, EpiState& e, int n0, int half, int lane) {
    const int c = n0 + half * 128 + 4 * lane;
    if constexpr (F8) e.pw = __ldg(reinterpret_cast<const float4*>(p.ws2 + c));
    if (p.bias2) e.pb = __ldg(reinterpret_cast<const float4*>(p.bias2 + c));
  }

  __device__ static void epilogue(const Params& p, EpiState& e, const TileInfo& t, uint32_t taddr, int q, int half,
                                  int lane, uint8_t* extra, uint32_t rank) {
    const int row = t.m0 + 128 * int(rank) + q * 32 + lane;
    float* cols = reinterpret_cast<float*>(extra + (q + 4 * half) * kColBytes);   // [128 scales][128 biases]
    // ST: this warp's two staging boxes; the tile's rows go to rows slot * 256 + .. of the buffer
    uint8_t* wbuf = extra + (q + 4 * half) * 2 * kBf16BoxBytes;
    const bool st_tile = ST && t.slot < p.pu_tiles;
    const int pu_y0 = t.slot * kRows + 128 * int(rank) + q * 32;
    if (!ST && (F8 || p.bias2)) {
      if (e.pre_n0 != t.n0) fetch_cols(p, e, t.n0, half, lane);
      __syncwarp();
      if constexpr (F8) reinterpret_cast<float4*>(cols)[lane] = e.pw;
      if (p.bias2) reinterpret_cast<float4*>(cols + 128)[lane] = e.pb;
      __syncwarp();
      e.pre_n0 = next_tile_n0(p, e, t);
      if (e.pre_n0 >= 0) fetch_cols(p, e, e.pre_n0, half, lane);
    }
    if (t.first) {
      e.mref = -INFINITY;
      e.s_hi = e.s_lo = e.w_hi = e.w_lo = 0.f;
      e.zy = 0.f;
      e.found = 0;
      // target column within this vocabulary (shard); -1 when it lies outside
      const long long yl = row < p.N ? p.targets[row] - p.v_begin : -1;
      e.y = (yl >= 0 && yl < p.V) ? int(yl) : -1;
      if constexpr (F8) e.xs = row < p.N ? p.xs[row] : 0.f;
    }
    const float sc = p.scale2;
    // This warp's 32-column chunks that hold vocabulary columns; the TMEM load
    // of chunk ch+1 is in flight while chunk ch is processed.
    const int cbase = t.n0 + half * 128;
    const int nch = min(4, max(0, (p.V - cbase + 31) / 32));
    uint32_t r[32];
    if (nch > 0) {
      tmem_ld32_issue(taddr + uint32_t(half * 128), r);
      tmem_ld32_wait(r);
    }
#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
      const int c0 = cbase + ch * 32;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
      if (ch + 1 < nch) tmem_ld32_issue(taddr + uint32_t(half * 128 + (ch + 1) * 32), r);
      if constexpr (F8) {
        // logit * log2(e)/tau = acc * xs[row] * (ws[col] * log2(e)/tau) (+ b * log2(e)/tau)
        const float4* w4 = reinterpret_cast<const float4*>(cols + ch * 32);
        const float4* b4 = reinterpret_cast<const float4*>(cols + 128 + ch * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 w = w4[i];
          const float4 b = p.bias2 ? b4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
          v[4 * i + 0] = fmaf(v[4 * i + 0] * e.xs, w.x, b.x);
          v[4 * i + 1] = fmaf(v[4 * i + 1] * e.xs, w.y, b.y);
          v[4 * i + 2] = fmaf(v[4 * i + 2] * e.xs, w.z, b.z);
          v[4 * i + 3] = fmaf(v[4 * i + 3] * e.xs, w.w, b.w);
        }
      } else if (p.bias2) {
        // ST keeps no column vectors in shared memory: the bias comes from L1/L2
        const float4* b4 = ST ? reinterpret_cast<const float4*>(p.bias2 + c0)
                              : reinterpret_cast<const float4*>(cols + 128 + ch * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 b = ST ? __ldg(b4 + i) : b4[i];
          v[4 * i + 0] = fmaf(v[4 * i + 0], sc, b.x);
          v[4 * i + 1] = fmaf(v[4 * i + 1], sc, b.y);
          v[4 * i + 2] = fmaf(v[4 * i + 2], sc, b.z);
          v[4 * i + 3] = fmaf(v[4 * i + 3], sc, b.w);
        }
      }
      // Without bias or e4m3 scales v is still the raw logit; its scale to
      // log2 units folds into the FFMA that forms t - m below (mul = sc).
      const float mul = (F8 || p.bias2) ? 1.f : sc;
      const bool tail = c0 + 32 > p.V;   // columns past V: out of the max, weight 0
      if (tail) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c0 + i >= p.V) v[i] = -INFINITY;
      }
      float mx = v[0];
#pragma unroll
      for (int i = 1; i < 32; ++i) mx = fmaxf(mx, v[i]);
      mx *= mul;   // mul > 0
      // Reference max kept on an integer grid in log2 units; move it only
      // when a logit would exceed it by more than 2^16, so rescaling is rare
      // and exact (a power of two).  (Every 2^(t - m) then stays <= 2^16, which
      // also bounds the stored 2^t below, 2^(16 + 100), for any row.)
      if (mx > e.mref + 16.f) {
        const float nref = ceilf(mx);
        if (e.mref == -INFINITY) {
          e.mref = nref;
        } else {
          const float dd = e.mref - nref;     // negative integer
          const int di = int(dd);
          e.w_hi = ldexpf(e.w_hi + dd * e.s_hi, di);
          e.w_lo = ldexpf(e.w_lo + dd * e.s_lo, di);
          e.s_hi = ldexpf(e.s_hi, di);
          e.s_lo = ldexpf(e.s_lo, di);
          e.mref = nref;
        }
      }
      // ST: 2^t = 2^(t - m) 2^m exactly (m an integer); m is capped at 100, past
      // which the backward recomputes the row anyway (its stored values stay
      // finite, below 2^116), and 2^m below 2^-126 is taken as 0 (such a
      // column's p is below 2^-46 in any row the stored path keeps)
      float psc = 0.f;
      if constexpr (ST) {
        const float mr = fminf(e.mref, 100.f);
        psc = mr >= -126.f ? __int_as_float((int(mr) + 127) << 23) : 0.f;
      }
      uint32_t pk[ST ? 16 : 1];
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, w0 = 0.f, w1 = 0.f, w2 = 0.f, w3 = 0.f;
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float nm = -e.mref;
        float d0 = fmaf(v[i], mul, nm), d1 = fmaf(v[i + 1], mul, nm), d2 = fmaf(v[i + 2], mul, nm),
              d3 = fmaf(v[i + 3], mul, nm);
        if (tail) {   // -inf -> a finite large negative: 2^d = 0 and 0 * d = 0
          d0 = fmaxf(d0, -1.0e30f); d1 = fmaxf(d1, -1.0e30f); d2 = fmaxf(d2, -1.0e30f); d3 = fmaxf(d3, -1.0e30f);
        }
        const float x0 = ex2_approx(d0), x1 = ex2_approx(d1), x2 = ex2_approx(d2), x3 = ex2_approx(d3);
        s0 += x0; s1 += x1; s2 += x2; s3 += x3;
        w0 = fmaf(x0, d0, w0); w1 = fmaf(x1, d1, w1); w2 = fmaf(x2, d2, w2); w3 = fmaf(x3, d3, w3);
        if constexpr (ST) {
          pk[i / 2] = pack_bf16x2(x0 * psc, x1 * psc);
          pk[i / 2 + 1] = pack_bf16x2(x2 * psc, x3 * psc);
        }
      }
      two_sum_acc(e.s_hi, e.s_lo, (s0 + s1) + (s2 + s3));
      two_sum_acc(e.w_hi, e.w_lo, (w0 + w1) + (w2 + w3));
      const unsigned ty = unsigned(e.y - c0);
      if (ty < 32u) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (unsigned(i) == ty) e.zy = v[i] * mul;
        e.found = 1;
      }
      if constexpr (ST) {
        // warp-uniform; one 32 x 32 box per chunk through two alternate staging
        // buffers (columns past V are dropped by the store); the target entry
        // is written as 0 (the backward sets it)
        if (st_tile) store_bf16_box(&p.tmPu, p.status, wbuf, e.nbuf, lane, pk, c0, pu_y0, ty);
      }
      if (ch + 1 < nch) tmem_ld32_wait(r);
    }
    if (t.last && row < p.N && RL_DCHECK(t.seg < t.aux && t.aux <= p.pcap, p.status)) {
      float4* dst = p.partial + (size_t(row) * (2 * t.aux) + size_t(t.seg) * 2 + half) * 2;
      dst[0] = make_float4(e.mref, e.s_hi, e.s_lo, e.w_hi);
      dst[1] = make_float4(e.w_lo, e.zy, e.found ? 1.f : 0.f, 0.f);
    }
  }
  __device__ static void epilogue_finish(const Params&, int lane) {
    if constexpr (ST) {
      if (lane == 0) tma_store_wait_all<0>();
      __syncwarp();
    }
  }
};

// kMergeLanes lanes per row: see merge_row.cuh.
__global__ void fwd_merge_kernel(MergeParams p) {
  const int r = int((blockIdx.x * (long long)blockDim.x + threadIdx.x) / kMergeLanes);
  const bool live = r < p.N && row_has_forward(p, r);
  merge_row(p, live ? r : -1, threadIdx.x % kMergeLanes);
}

// One merged state slot per row, written in the partial-slot format
// (M, s_hi, s_lo, w_hi), (w_lo, t_target, found, 0).
__global__ void shard_state_kernel(MergeParams p, float4* state) {
  const int r = int((blockIdx.x * (long long)blockDim.x + threadIdx.x) / kMergeLanes);
  const int sub = threadIdx.x % kMergeLanes;
  const bool live = r < p.N;
  const RowSums m = merge_slots(p, live ? r : -1, sub);
  if (!live || sub != 0) return;
  state[2 * size_t(r)] = make_float4(m.M, m.shi, m.slo, m.whi);
  state[2 * size_t(r) + 1] = make_float4(m.wlo, m.who ? m.zy : 0.f, m.who ? 1.f : 0.f, 0.f);
}

__global__ void backward_rows_in_kernel(const float* lse, const float* dlogp, int N, double inv_tau, float* lse2,
                                        float* coef) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  lse2[n] = float(double(lse[n]) * 1.4426950408889634);
  coef[n] = float(double(dlogp[n]) * inv_tau);
}

// =============================================================== dlogits
// Column sums of a 32 x 32 block held one row per lane (v[j] = column j):
// a butterfly in which each step halves the columns a lane keeps and adds the
// partner's half, so lane l ends with column l's sum in v[0] (fixed order).
template <int OFF>
__device__ __forceinline__ void colsum_step(float (&v)[32], int lane) {
  const bool upper = (lane & OFF) != 0;
#pragma unroll
  for (int i = 0; i < OFF; ++i) {
    const float send = upper ? v[i] : v[i + OFF];
    const float keep = upper ? v[i + OFF] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
  }
}
__device__ __forceinline__ float warp_column_sum(float (&v)[32], int lane) {
  colsum_step<16>(v, lane);
  colsum_step<8>(v, lane);
  colsum_step<4>(v, lane);
  colsum_step<2>(v, lane);
  colsum_step<1>(v, lane);
  return v[0];
}

template <int CL, int KBX = 1>   // KBX: as for FwdPolicy
struct DlPolicy {
  static constexpr int kCluster = CL;
  static constexpr int PAIR = CL >= 2 ? 2 : 1;
  static constexpr int kRows = 128 * CL;
  static constexpr int kStages = (PAIR == 2 ? 6 : 4) / KBX;
  static constexpr int kSubs = 1;
  static constexpr int kBN = 256;
  static constexpr int kK16 = 4 * KBX;
  static constexpr int kBox = 128 * 128;                    // one 128-row x 128-byte operand box
  static constexpr int kABytes = kBox * KBX;
  static constexpr int kBBytes = (256 / PAIR) * 128 * KBX;
  static constexpr int kStageBuf = kBf16BoxBytes;  // one 32-row x 32-column bf16 box, 64-byte swizzle
  static constexpr int kExtraSmem = kEpiWarps * 2 * kStageBuf;
  static_assert(2 * kStageBuf == kBf16Box64Bytes, "a warp's two boxes hold one 32 x 64 bf16 box (bf16 G)");
  static constexpr uint32_t kIdesc = idesc_bf16(kRows, 256, 0, 0);
  using Params = DlParams;
  struct EpiState {
    int nbuf = 0;
    int nc = -1;   // rows of this chunk (read from the device on the first tile)
  };
  __device__ static int chunk_rows(const Params& p) { return min(max(*p.rows_total - p.n0, 0), p.Nc); }
  __device__ static bool has_work(const Params& p) { return chunk_rows(p) > 0; }

  __device__ static void cta_setup(const Params&, uint8_t*) {}
  __device__ static void prefetch(const Params& p) {
    tma_prefetch_desc(&p.tmA);
    tma_prefetch_desc(&p.tmB);
    tma_prefetch_desc(&p.tmG);
  }
  // Tiles u = j * Rc + r: CTAs running together share the W tile j.
  template <class F>
  __device__ static void for_each_tile(const Params& p, F&& f) {
    const int Rc = (chunk_rows(p) + kRows - 1) / kRows;
    const int tiles = Rc * p.Vt;
    const int kbs = p.nseg * p.kb_per_seg;
    const int g0 = blockIdx.x / CL, gn = gridDim.x / CL;
    for (int u = g0; u < tiles; u += gn) {
      const int j = u / Rc;
      const int r = u - j * Rc;
      TileInfo t{r * kRows, j * 256, 0, kbs, u, 0, true, true};
      if (!f(t)) return;
    }
  }
  __device__ static void load(const Params& p, uint8_t* st, uint32_t bar, const TileInfo& t, int kb, uint32_t rank) {
    const int s = kb / p.kb_per_seg;
    const int kk = (kb - s * p.kb_per_seg) * 64 * KBX;
    if constexpr (CL == 2) {
#pragma unroll
      for (int x = 0; x < KBX; ++x) {
        if (tma_x_ok<2>(p.seg_a[s] + kk + 64 * x, p.status))
          tma_load_2d_pair(&p.tmA, bar, st + x * kBox, p.seg_a[s] + kk + 64 * x, p.a_row0 + t.m0 + 128 * int(rank));
        if (tma_x_ok<2>(p.seg_b[s] + kk + 64 * x, p.status))
          tma_load_2d_pair(&p.tmB, bar, st + kABytes + x * kBox, p.seg_b[s] + kk + 64 * x, t.n0 + 128 * int(rank));
      }
    } else {
      static_assert(KBX == 1, "single-CTA tiles keep one box per operand");
      if (tma_x_ok<2>(p.seg_a[s] + kk, p.status)) tma_load_2d(&p.tmA, bar, st, p.seg_a[s] + kk, p.a_row0 + t.m0);
      if (tma_x_ok<2>(p.seg_b[s] + kk, p.status)) tma_load_2d(&p.tmB, bar, st + kABytes, p.seg_b[s] + kk, t.n0);
    }
  }
  __device__ static uint64_t adesc(uint32_t sa, int k, const TileInfo&) {
    return sdesc_sw128(sa + (k >> 2) * kBox + (k & 3) * 32, 16, 1024);
  }
  __device__ static uint64_t bdesc(uint32_t sa, int k, const TileInfo&) {
    return sdesc_sw128(sa + kABytes + (k >> 2) * kBox + (k & 3) * 32, 16, 1024);
  }
  __device__ static uint32_t idesc(const TileInfo&) { return kIdesc; }
  static constexpr int kAccBufs = 2;
  __device__ static uint32_t tx_bytes(const Params&, const TileInfo&) { return kABytes + kBBytes; }
  __device__ static void mma(const Params&, uint32_t d, uint32_t sa, int k, const TileInfo& t, uint32_t accum) {
    if constexpr (PAIR == 2)
      umma_bf16_pair(d, adesc(sa, k, t), bdesc(sa, k, t), kIdesc, accum);
    else
      umma_bf16(d, adesc(sa, k, t), bdesc(sa, k, t), kIdesc, accum);
  }

  // Write one 32x32 bf16 box (this lane's 64-byte row) through shared memory
  // with a TMA store; two staging buffers per warp alternate.
  __device__ static void store_box(const Params& p, EpiState& e, uint8_t* wbuf, int lane, const uint32_t (&w)[16],
                                   int x, int y) {
    store_bf16_box(&p.tmG, p.status, wbuf, e.nbuf, lane, w, x, y);
  }

  __device__ static void epilogue(const Params& p, EpiState& e, const TileInfo& t, uint32_t taddr, int q, int half,
                                  int lane, uint8_t* extra, uint32_t rank) {
    uint8_t* wbuf = extra + (q + 4 * half) * 2 * kStageBuf;
    const int r0 = t.m0 + 128 * int(rank) + q * 32;   // first row of this warp within the chunk
    const int rl = r0 + lane;
    if (e.nc < 0) e.nc = chunk_rows(p);
    const bool valid = rl < e.nc;
    const int row = p.n0 + rl;
    const float lse2 = valid ? p.lse2[row] : 0.f;
    const float cf = valid ? p.coef[row] : 0.f;
    const long long yl = valid ? p.targets[row] - p.v_begin : -1;
    const int y = (yl >= 0 && yl < p.V) ? int(yl) : -1;   // target column within this vocabulary (shard)
    const float sc = p.scale2;
#pragma unroll 1
    for (int ch = 0; ch < 4; ++ch) {
      const int c0 = t.n0 + half * 128 + ch * 32;
      if (c0 >= p.Vp) break;
      float v[32];
      tmem_ld32(taddr + uint32_t(half * 128 + ch * 32), v);
      if (p.bias2) {
        const float4* b4 = reinterpret_cast<const float4*>(p.bias2 + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 b = __ldg(b4 + i);
          v[4 * i + 0] = fmaf(v[4 * i + 0], sc, b.x - lse2);
          v[4 * i + 1] = fmaf(v[4 * i + 1], sc, b.y - lse2);
          v[4 * i + 2] = fmaf(v[4 * i + 2], sc, b.z - lse2);
          v[4 * i + 3] = fmaf(v[4 * i + 3], sc, b.w - lse2);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = fmaf(v[i], sc, -lse2);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = -cf * ex2_approx(v[i]);
      const unsigned ty = unsigned(y - c0);
      if (ty < 32u) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (unsigned(i) == ty) v[i] += cf;
      }
      if (c0 + 32 > p.V) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c0 + i >= p.V) v[i] = 0.f;
      }
      if (p.err && ty < 32u) {
        // The target entry c (1 - p_y) / tau carries a row's dX; its bf16
        // rounding error (one relative error for every row of a sequence
        // with the same c) is kept in fp32 and added back in the dX epilogue.
        float vt = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (unsigned(i) == ty) vt = v[i];
        p.err[row] = vt - __bfloat162float(__float2bfloat16_rn(vt));
      }
      uint32_t hi[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) hi[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
      const int y0 = r0;
      if (!p.lo_off) {
        // bf16 G: chunks pair up into 64-column boxes (tmG: box 64 x 32, 128-byte
        // swizzle); a lone last chunk's partner columns lie past V and are dropped
        stage_half(wbuf, lane, hi, ch & 1, ~0u);
        if ((ch & 1) || ch == 3 || c0 + 32 >= p.Vp) store_box64(&p.tmG, p.status, wbuf, lane, c0 - (ch & 1) * 32, y0);
      } else {
        store_box(p, e, wbuf, lane, hi, c0, y0);
      }
      if (p.lo_off) {
        uint32_t lo[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const __nv_bfloat162 h2 = *reinterpret_cast<const __nv_bfloat162*>(&hi[i]);
          lo[i] = pack_bf16x2(v[2 * i] - __low2float(h2), v[2 * i + 1] - __high2float(h2));
        }
        store_box(p, e, wbuf, lane, lo, c0 + p.lo_off, y0);
      }
      if (p.dbp) {
        // db partial: this warp's 32 rows summed per column (fp32 G, before
        // the bf16 rounding), one row of the [rows/32][V] partial buffer
        const float cs = warp_column_sum(v, lane);
        if (c0 + lane < p.V && RL_DCHECK((r0 >> 5) < (p.Nc + 255) / 256 * 8, p.status))
          p.dbp[size_t(r0 >> 5) * p.V + c0 + lane] = cs;
      }
    }
  }
  __device__ static void epilogue_finish(const Params&, int lane) {
    if (lane == 0) tma_store_wait_all<0>();
    __syncwarp();
  }
};

// =============================================================== gemmH
// D[row][h] on CTA pairs: TMEM lane = output row (128 per CTA), columns = h.
// A tile is 256 rows x 448 h, held as one split accumulator of two 224-h
// subs (TMEM columns 0.. and 256..): each k-block's A tile (G rows) feeds
// both, so an A byte carries 448 columns of work.  Output rows leave through
// shared memory as 32x32 fp32 boxes with TMA stores (or TMA reduce-adds when
// accumulating); the dX rows of the compacted backward are instead added from
// registers straight into dX at their original rows (HParams::dx_idx).  One
// launch runs up to two such problems (dX and dW of a chunk) with a balanced
// static schedule; see for_each_tile.
struct HPolicy {
  static constexpr int kCluster = 2;
  static constexpr int kStages = 4;
  static constexpr int kSubs = 2;
  static constexpr int kBN = 256;                 // TMEM column offset of sub 1
  static constexpr int kAccBufs = 1;
  static constexpr int kNS = 224;                 // h per sub (112 per CTA)
  static constexpr int kNH = 2 * kNS;             // h per tile
  static constexpr int kK16 = 4;
  static constexpr int kABytes = 128 * 64 * 2;    // 128 rows x 64 k
  static constexpr int kBSub = 128 * 64 * 2;      // per sub: two 64-h runs (112 h used)
  static constexpr int kBBytes = 2 * kBSub;
  static constexpr int kBoxBytes = 32 * 32 * 4;
  static constexpr int kExtraSmem = kEpiWarps * kBoxBytes;
  using Params = HParams;
  struct EpiState {};

  __device__ static void cta_setup(const Params&, uint8_t*) {}
  __device__ static void prefetch(const Params& p) {
    for (int q = 0; q < p.nprob; ++q) {
      tma_prefetch_desc(&p.tmA[q]);
      tma_prefetch_desc(&p.tmB[q]);
      tma_prefetch_desc(&p.tmB48[q]);
      tma_prefetch_desc(&p.tmO[q]);
    }
  }
  // The chunk's row count is read on the device: problem 0 (dX) gets its
  // row tiles from it, problem 1 (dW) its k-blocks per term.
  __device__ static void chunk_problems(const Params& p, HProblem (&pr)[2]) {
    const int nc = min(max(*p.rows_total - p.n0, 0), p.nc_max);
    pr[0] = p.pr[0];
    pr[1] = p.pr[1];
    pr[0].Mt = (nc + 255) / 256;
    if (p.nprob > 1) {
      pr[1].kb_per_seg = (nc + 63) / 64;
      if (nc == 0 && pr[1].reduce) pr[1].Mt = 0;   // nothing to add
    }
  }
  // Unit u of problem q: order 0 numbers (k part, h tile, row tile) with the
  // row tile fastest; order 1 numbers (row tile, h tile) with h fastest.
  // A problem with ksplit 2 cuts the k range in two halves, one unit each.
  __device__ static TileInfo tile_of(const Params& p, const HProblem& pr, int q, int u) {
    const int per = pr.Mt * pr.Ht;
    const int part = u / per;
    const int v = u - part * per;
    int i, j;
    if (pr.order == 0) {
      j = v / pr.Mt;
      i = v - j * pr.Mt;
    } else {
      i = v / pr.Ht;
      j = v - i * pr.Ht;
    }
    const int kbt = p.nseg * pr.kb_per_seg;
    const int cut = pr.ksplit == 2 ? kbt / 2 : kbt;
    TileInfo t{i * 256, j * kNH, part == 0 ? 0 : cut, part == 0 ? cut : kbt, u, q, true, true, pr.kb_per_seg};
    t.wide = (pr.wide && j == pr.Ht - 1) ? 1 : 0;
    return t;
  }
  __device__ static int units(const HProblem& pr) { return pr.Mt * pr.Ht * pr.ksplit; }
  __device__ static bool has_work(const Params& p) {
    HProblem pr[2];
    chunk_problems(p, pr);
    return units(pr[0]) > 0 || (p.nprob > 1 && units(pr[1]) > 0);
  }
  // Pair g of gn: problem 0 units g, g+gn, ...; then problem 1 units.  Pairs
  // that got fewer problem-0 units ("early" pairs) first take problem-1 units
  // [0, F*d) round-robin among themselves, d = problem-0 unit length in
  // problem-1 units (by cost); the rest go round-robin over all pairs.  Consecutive
  // units run at the same time, so operand tiles they share stay in L2.
  template <class F>
  __device__ static void for_each_tile(const Params& p, F&& f) {
    HProblem pr[2];
    chunk_problems(p, pr);
    const int g = blockIdx.x >> 1, gn = gridDim.x >> 1;
    const int T0 = units(pr[0]);
    for (int u = g; u < T0; u += gn)
      if (!f(tile_of(p, pr[0], 0, u))) return;
    if (p.nprob < 2) return;
    const int T1 = units(pr[1]);
    // A problem-1 (dW) unit costs its k-blocks plus the drain of its accumulator
    // (two 224-column subs stored from TMEM with no next k-loop to hide behind),
    // measured as about kDrainKb k-blocks: d problem-1 units match one problem-0
    // unit (kDrainKb = 6 against 0: the B=1, T=4096 dX/dW launch 1.095 -> 1.055 ms;
    // 4 and 8 bracket it).
    constexpr int kDrainKb = 6;
    const int kx = p.nseg * pr[0].kb_per_seg / pr[0].ksplit, kw = p.nseg * pr[1].kb_per_seg;
    const int d_tiles = kw > 0 ? max(1, (kx + (kw + kDrainKb) / 2) / (kw + kDrainKb)) : 1;
    const int r = T0 % gn;
    const int early = (r == 0) ? 0 : gn - r;
    const int ph1 = min(T1, early * d_tiles);
    if (early > 0 && g >= r)
      for (int u = g - r; u < ph1; u += early)
        if (!f(tile_of(p, pr[1], 1, u))) return;
    for (int u = ph1 + g; u < T1; u += gn)
      if (!f(tile_of(p, pr[1], 1, u))) return;
  }
  // Columns of sub `sub` of tile t: 224, or 240 for the widened last sub.
  __device__ static int sub_n(const TileInfo& t, int sub) { return (t.wide && sub == 1) ? kNS + 16 : kNS; }
  // One k-block: this CTA's 128 A rows and, for each sub, its half of the B
  // rows: a 64-h run and the next 48 (a 48-wide box lands where the first 48
  // columns of a 64-wide one would, the rest of that run untouched and unread),
  // or two 64-h runs for the 120 of a widened sub.
  __device__ static void load(const Params& p, uint8_t* st, uint32_t bar, const TileInfo& t, int kb, uint32_t rank) {
    const int q = t.seg;
    const HProblem& pr = p.pr[q];
    const int s = kb / t.aux;
    const int kk = (kb - s * t.aux) * 64;
    const int r = t.m0 + 128 * int(rank);
    if (pr.a_mn) {   // dW: k = A rows (positions) kk..kk+63, this CTA's 128 columns
      const int pk = pr.a_outer0 + kk;
      const int y = p.row_map ? __ldg(p.row_map + (pk >> 7)) + (pk & 127) : pk;
      if (tma_x_ok<2>(p.seg_a[s] + r, p.status)) tma_load_2d_pair(&p.tmA[q], bar, st, p.seg_a[s] + r, y);
      if (tma_x_ok<2>(p.seg_a[s] + r + 64, p.status))
        tma_load_2d_pair(&p.tmA[q], bar, st + 8192, p.seg_a[s] + r + 64, y);
    } else {         // dX: this CTA's 128 A rows (positions r..r+127), k = columns kk..kk+63
      const int y = p.row_map ? __ldg(p.row_map + (r >> 7)) : r;
      if (tma_x_ok<2>(p.seg_a[s] + kk, p.status)) tma_load_2d_pair(&p.tmA[q], bar, st, p.seg_a[s] + kk, y);
    }
#pragma unroll
    for (int sub = 0; sub < 2; ++sub) {
      const int h = p.seg_b[s] + t.n0 + kNS * sub + (sub_n(t, sub) / 2) * int(rank);
      uint8_t* b = st + kABytes + sub * kBSub;
      if (tma_x_ok<2>(h, p.status)) tma_load_2d_pair(&p.tmB[q], bar, b, h, pr.b_outer0 + kk);
      const CUtensorMap* m2 = sub_n(t, sub) == kNS ? &p.tmB48[q] : &p.tmB[q];
      if (tma_x_ok<2>(h + 64, p.status)) tma_load_2d_pair(m2, bar, b + 8192, h + 64, pr.b_outer0 + kk);
    }
  }
  // Bytes one CTA's copies of a sub's B rows bring: 64 + 48 columns, or 64 + 64
  // in a widened sub.
  __device__ static uint32_t b_sub_bytes(const TileInfo& t, int sub) {
    return sub_n(t, sub) == kNS ? 8192u + 6144u : 16384u;
  }
  __device__ static uint64_t adesc(uint32_t sa, int k, const TileInfo& t) {
    return t.seg == 1 ? sdesc_sw128(sa + k * 2048, 8192, 1024) : sdesc_sw128(sa + k * 32, 16, 1024);
  }
  __device__ static uint64_t bdesc(uint32_t sa, int k, int sub) {
    return sdesc_sw128(sa + kABytes + sub * kBSub + k * 2048, 8192, 1024);
  }
  __device__ static uint32_t idesc(const TileInfo& t, int sub) {
    if (sub_n(t, sub) == kNS) return t.seg == 1 ? idesc_bf16(256, kNS, 1, 1) : idesc_bf16(256, kNS, 0, 1);
    return t.seg == 1 ? idesc_bf16(256, kNS + 16, 1, 1) : idesc_bf16(256, kNS + 16, 0, 1);
  }
  __device__ static uint32_t tx_bytes(const Params&, const TileInfo& t) {
    return kABytes + b_sub_bytes(t, 0) + b_sub_bytes(t, 1);
  }
  __device__ static void mma(const Params&, uint32_t d, uint32_t sa, int k, const TileInfo& t, int sub,
                             uint32_t accum) {
    umma_bf16_pair(d, adesc(sa, k, t), bdesc(sa, k, sub), idesc(t, sub), accum);
  }

  // v[i] += err * W[target][x0 + i] for the valid columns (bf16 W row, 16-byte aligned).
  __device__ static void add_target_row(float (&v)[32], const __nv_bfloat16* wrow, float err, int x0, int Hout) {
    if (x0 + 32 <= Hout) {
      const uint4* w4 = reinterpret_cast<const uint4*>(wrow + x0);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 u = __ldg(w4 + k);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&w[j]);
          v[8 * k + 2 * j] = fmaf(err, __low2float(b2), v[8 * k + 2 * j]);
          v[8 * k + 2 * j + 1] = fmaf(err, __high2float(b2), v[8 * k + 2 * j + 1]);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (x0 + i < Hout) v[i] = fmaf(err, __bfloat162float(wrow[x0 + i]), v[i]);
    }
  }

  // Sub `sub` of the accumulator: warp (q, half) writes TMEM lanes 32q..+31,
  // 32-column chunks 0-3 (half 0) or 4-6 (half 1).
  __device__ static void epilogue(const Params& p, EpiState&, const TileInfo& t, uint32_t taddr, int q, int half,
                                  int lane, uint8_t* extra, uint32_t rank, int sub) {
    const HProblem& pr = p.pr[t.seg];
    const CUtensorMap* om = &p.tmO[t.seg];
    uint8_t* buf = extra + (q + 4 * half) * kBoxBytes;
    const int y0 = t.m0 + 128 * int(rank) + q * 32;
    const int c_begin = half ? 4 : 0, c_end = half ? (sub_n(t, sub) > kNS ? 8 : 7) : 4;
    const bool no_k = t.kb_end <= t.kb_begin;   // empty sum (a chunk without rows): store zeros
    // dX rows: the target-entry correction err * W[target] on the first k part
    const __nv_bfloat16* wrow = nullptr;
    float ferr = 0.f;
    if (t.seg == 0 && p.dx_err && t.kb_begin == 0 && !no_k) {
      const int nc = min(max(*p.rows_total - p.n0, 0), p.nc_max);
      const int y = y0 + lane;
      if (y < nc) {
        ferr = p.dx_err[p.n0 + y];
        const long long tr = p.dx_tgt[p.n0 + y] - p.dx_wbegin;
        if (ferr != 0.f && tr >= 0 && tr < p.dx_wrows) wrow = p.dx_w + size_t(tr) * p.dx_wld;
      }
    }
    if (t.seg == 0 && p.dx_idx) {
      // dX rows of the compacted backward, added at their original rows.
      const int nc = min(max(*p.rows_total - p.n0, 0), p.nc_max);
      const int y = y0 + lane;
      const int drow = (y < nc && !no_k) ? p.dx_idx[p.n0 + y] : -1;
      float* dst = (drow >= 0 && RL_DCHECK(drow < p.dx_nrows, p.status)) ? p.dx_out + size_t(drow) * p.dx_ld
                                                                          : nullptr;
      const float ks = (p.dx_scale && dst) ? p.dx_scale[p.n0 + y] : 1.f;
#pragma unroll 1
      for (int c = c_begin; c < c_end; ++c) {
        const int x0 = t.n0 + sub * kNS + c * 32;
        if (x0 >= pr.Hout) break;
        float v[32];
        tmem_ld32(taddr + uint32_t(c * 32), v);   // warp-collective: every lane loads
        if (!dst) continue;
        if (p.dx_scale) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= ks;
        }
        if (wrow) add_target_row(v, wrow, ferr, x0, pr.Hout);
        if (p.dx_vec && x0 + 32 <= pr.Hout) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            atomicAdd(reinterpret_cast<float4*>(dst + x0 + 4 * k),
                      make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (x0 + i < pr.Hout) atomicAdd(dst + x0 + i, v[i]);
        }
      }
      return;
    }
#pragma unroll 1
    for (int c = c_begin; c < c_end; ++c) {
      const int x0 = t.n0 + sub * kNS + c * 32;
      if (pr.xcol_out != nullptr && pr.xcol >= x0 && pr.xcol < x0 + 32) {
        // the routed column (db through dW's GEMM), one value per output row,
        // read on its own (warp-uniform column)
        const float xv = no_k ? 0.f : tmem_ld1(taddr + uint32_t(c * 32 + (pr.xcol - x0)));
        const int r = y0 + lane;
        if (r < pr.xrows) pr.xcol_out[r] = pr.reduce ? pr.xcol_out[r] + xv : xv;
      }
      if (x0 >= pr.Hout) break;
      float v[32];
      if (no_k) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      } else {
        tmem_ld32(taddr + uint32_t(c * 32), v);
      }
      if (wrow) add_target_row(v, wrow, ferr, x0, pr.Hout);
      if (lane == 0) tma_store_wait_read<0>();
      __syncwarp();
      float4* row = reinterpret_cast<float4*>(buf + lane * 128);
#pragma unroll
      for (int k = 0; k < 8; ++k) row[k ^ (lane & 7)] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        if (!tma_x_ok<4>(x0, p.status)) {
        } else if (pr.reduce) {
          tma_reduce_add_2d(om, buf, x0, y0);
        } else {
          tma_store_2d(om, buf, x0, y0);
        }
        tma_store_commit();
      }
    }
  }
  __device__ static void epilogue_finish(const Params&, int lane) {
    if (lane == 0) tma_store_wait_all<0>();
    __syncwarp();
  }
};

// =============================================================== small kernels
__global__ void bias2_kernel(const void* b, int is_fp32, int V, int Vpad, float scale2, float* out) {
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= Vpad) return;
  float x = 0.f;
  if (v < V) x = is_fp32 ? static_cast<const float*>(b)[v] : __bfloat162float(static_cast<const __nv_bfloat16*>(b)[v]);
  out[v] = v < V ? x * scale2 : 0.f;
}

// fp32 -> three bf16 terms hi + mid + lo (each the rounding of what is left),
// laid out [rows, 3*Cp] with each term in its own Cp-wide column block.
__global__ void split3_kernel(const float* src, long long rows, int cols, int Cp, __nv_bfloat16* out) {
  const long long n = rows * Cp;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long r = idx / Cp;
    const int c = int(idx - r * Cp);
    const float x = c < cols ? src[r * cols + c] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    __nv_bfloat16* o = out + r * 3 * Cp + c;
    o[0] = hi;
    o[Cp] = mid;
    o[2 * Cp] = lo;
  }
}

// db (+)= the sum, in row-block order, of the recompute's per-32-row column
// partials over the chunk's rows.
__global__ void db_reduce_kernel(const float* part, const int* rows_total, int n0, int Nc, int V, float* db,
                                 int accumulate) {
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= V) return;
  const int nc = min(max(*rows_total - n0, 0), Nc);
  const int nblk = (nc + 31) / 32;
  float a = 0.f;
  for (int k = 0; k < nblk; ++k) a += part[size_t(k) * V + v];
  db[v] = accumulate ? db[v] + a : a;
}

__global__ void selftest_wait_kernel(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const AbortCtl ac{&abort_flag, status, limit_ns};
    mbar_wait(&bar, 0, ac);   // nothing arrives: runs out after limit_ns
  }
}

// =============================================================== launchers
// Per device: set the shared-memory attribute once and find how many
// clusters (CTAs for kCluster == 1) of this kernel can be resident at once.
template <class P>
static int engine_resident(cudaError_t* err) {
  constexpr int smem = engine_smem_bytes<P>();
  static_assert(smem <= 232448, "shared memory budget");
  static int cached[64] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return 0;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  *err = cudaFuncSetAttribute(tc_engine_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (*err != cudaSuccess) return 0;
  int n = 0;
  if (P::kCluster == 1) {
    int per_sm = 0, sms = 0;
    *err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc_engine_kernel<P>, kEngineThreads, smem);
    if (*err == cudaSuccess) *err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    n = per_sm * sms;
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(P::kCluster), 1, 1);
    cfg.blockDim = dim3(kEngineThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = P::kCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    *err = cudaOccupancyMaxActiveClusters(&n, tc_engine_kernel<P>, &cfg);
  }
  if (*err != cudaSuccess) return 0;
  if (n < 1) {
    *err = cudaErrorInvalidConfiguration;
    return 0;
  }
  if (dev < 64) cached[dev] = n;
  return n;
}

// Launch ``units`` independent work units' worth of persistent clusters.
template <class P>
static cudaError_t launch_engine(const typename P::Params& prm, int units, cudaStream_t st) {
  constexpr int smem = engine_smem_bytes<P>();
  cudaError_t err = cudaSuccess;
  const int resident = engine_resident<P>(&err);
  if (err != cudaSuccess) return err;
  const int grid = P::kCluster * (units < resident ? (units < 1 ? 1 : units) : resident);
  if (P::kCluster == 1) {
    tc_engine_kernel<P><<<grid, kEngineThreads, smem, st>>>(prm);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid), 1, 1);
  cfg.blockDim = dim3(kEngineThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = P::kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_engine_kernel<P>, prm);
}

int fwd_resident_clusters(int cluster) {
  cudaError_t e;
  return cluster == 2 ? engine_resident<FwdPolicy<2, false, 2>>(&e) : engine_resident<FwdPolicy<1>>(&e);
}
int gemmH_resident_clusters() {
  cudaError_t e;
  return engine_resident<HPolicy>(&e);
}
cudaError_t launch_fwd(const FwdParams& p, int units, int cluster, int kbx, cudaStream_t st) {
  if (p.xs) return launch_engine<FwdPolicy<2, true, 2>>(p, units, st);   // e4m3 operands: CTA pairs only
  if (p.pu_tiles > 0) {
    if (cluster != 2 || kbx != 2 || p.nseg != 1) return cudaErrorInvalidValue;
    return launch_engine<FwdPolicy<2, false, 2, true>>(p, units, st);
  }
  if (cluster == 1) return launch_engine<FwdPolicy<1>>(p, units, st);
  return kbx == 2 ? launch_engine<FwdPolicy<2, false, 2>>(p, units, st) : launch_engine<FwdPolicy<2>>(p, units, st);
}
cudaError_t launch_dl(const DlParams& p, int units, int cluster, int kbx, cudaStream_t st) {
  if (cluster == 1) return launch_engine<DlPolicy<1>>(p, units, st);
  return kbx == 2 ? launch_engine<DlPolicy<2, 2>>(p, units, st) : launch_engine<DlPolicy<2>>(p, units, st);
}
cudaError_t launch_gemmH(const HParams& p, int units, cudaStream_t st) { return launch_engine<HPolicy>(p, units, st); }
cudaError_t launch_merge(const MergeParams& p, cudaStream_t st) {
  constexpr int rows = 256 / kMergeLanes;   // rows per 256-thread block
  fwd_merge_kernel<<<(p.N + rows - 1) / rows, 256, 0, st>>>(p);
  return cudaGetLastError();
}
cudaError_t launch_shard_state(const MergeParams& p, float4* state, cudaStream_t st) {
  constexpr int rows = 256 / kMergeLanes;
  shard_state_kernel<<<(p.N + rows - 1) / rows, 256, 0, st>>>(p, state);
  return cudaGetLastError();
}
cudaError_t launch_backward_rows_in(const float* lse, const float* dlogp, int N, double inv_tau, float* lse2,
                                   float* coef, cudaStream_t st) {
  backward_rows_in_kernel<<<(N + 255) / 256, 256, 0, st>>>(lse, dlogp, N, inv_tau, lse2, coef);
  return cudaGetLastError();
}
cudaError_t launch_bias2(const void* b, int is_fp32, int V, int Vpad, float scale2, float* out, cudaStream_t st) {
  bias2_kernel<<<(Vpad + 255) / 256, 256, 0, st>>>(b, is_fp32, V, Vpad, scale2, out);
  return cudaGetLastError();
}
cudaError_t launch_split3(const float* src, long long rows, int cols, int Cp, __nv_bfloat16* out, cudaStream_t st) {
  const long long n = rows * Cp;
  long long nb = (n + 255) / 256;
  if (nb > 65535LL * 8) nb = 65535LL * 8;
  const int blocks = int(nb < 1 ? 1 : nb);
  split3_kernel<<<blocks, 256, 0, st>>>(src, rows, cols, Cp, out);
  return cudaGetLastError();
}
// Rows of the partial buffer: the recompute's tiles cover the chunk in whole
// 256-row tiles, and each 32 rows of a tile write one partial row.
int db_part_rows(int Nc) { return (Nc + 255) / 256 * 8; }
cudaError_t launch_db_reduce(const float* part, const int* rows_total, int n0, int Nc, int V, float* db, int accumulate,
                             cudaStream_t st) {
  db_reduce_kernel<<<(V + 255) / 256, 256, 0, st>>>(part, rows_total, n0, Nc, V, db, accumulate);
  return cudaGetLastError();
}
cudaError_t launch_selftest_wait(int* status, unsigned long long limit_ns, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace rl
