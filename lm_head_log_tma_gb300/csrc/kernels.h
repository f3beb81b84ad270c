// Kernel parameter blocks and launchers shared by the host API and the CUDA
// translation units of the library.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace rl {

constexpr int kMaxSeg = 6;

// Vocabulary segments of the forward: for R row tiles, Vt vocabulary tiles and
// G clusters, the P <= pcap that minimises (waves of R*P units) x (tiles per
// segment).  The host plan and the forward kernel (for a row count known only
// on the device) use this same rule.
__host__ __device__ inline int choose_segments(int R, int Vt, int G, int pcap) {
  int best = 1;
  long long best_t = -1;
  for (int P = 1; P <= pcap && P <= Vt; ++P) {
    const long long waves = ((long long)R * P + G - 1) / G;
    const long long t = waves * ((Vt + P - 1) / P);
    if (best_t < 0 || t < best_t) {
      best_t = t;
      best = P;
    }
  }
  return best;
}

struct FwdParams {
  CUtensorMap tmA;            // X (or its 3-term bf16 split, or e4m3): inner K, outer rows; box 128 B x 128
  CUtensorMap tmB;            // W (or split, or e4m3): inner K, outer vocab; box 128 B x 256 (128 per CTA of a pair)
  int nseg, kb_per_seg;       // K = nseg * kb_per_seg * (64 bf16 or 128 e4m3 elements)
  int seg_a[kMaxSeg], seg_b[kMaxSeg];  // K offsets of each product term
  int N, V, R, Vt, P;         // rows, vocab, row tiles (128 or 256 rows), vocab tiles (256), vocab segments
  // Optional: only the row tiles in tiles[0 .. *ntiles) (ascending) are computed, and
  // the segment count is chosen on the device for them (<= pcap; written to *P_out).
  const int* tiles;
  const int* ntiles;
  int pcap;
  int* P_out;
  float scale2;               // log2(e) / temperature
  const float* bias2;         // [Vt*256] b * scale2, zero padded; null without bias
  const float* xs;            // e4m3 operands: [N] per-row X scales, else null
  const float* ws2;           // e4m3 operands: [Vt*256] per-row W scales * scale2, zero padded
  const int64_t* targets;
  long long v_begin;          // vocabulary id of column 0 (a shard of a larger vocabulary), else 0
  float4* partial;            // [N][2P][2]
  // Optional stored probabilities (pu_tiles > 0, bf16 CTA-pair forward only):
  // for the row tiles in the first pu_tiles slots of the launch's tile order
  // (slot i = the i-th listed tile, or tile i without a list), every
  // computed logit's unnormalised probability 2^t (t = logit log2(e) / tau,
  // so p = 2^(t - lse2)) is written as bf16 to row (slot * 256 + row in
  // tile) of the buffer tmPu maps; the target column is written as 0.
  CUtensorMap tmPu;           // inner V columns, outer pu_tiles * 256 rows; box 32 x 32, 64-byte swizzle
  int pu_tiles;
  int* status;
  unsigned long long limit_ns;
};

struct MergeParams {
  const float4* partial;
  int N, V, slots;            // slots = 2P
  int slot_stride;            // 0: partial is [N][slots][2]; else [slots][slot_stride][2] (gathered shard states)
  const int* P_dev;           // if set, slots = 2 * *P_dev (segments chosen on the device)
  const uint8_t* tile_active; // if set, rows of row tiles (1 << tile_shift rows) with a 0 flag
  int tile_shift;             //   had no forward: they are skipped (all their rows are masked)
  const int64_t* targets;
  float* lse2;                // [N] lse in log2 units
  double* logp64;             // [N]
  float* ent32;               // [N]
  float* out_logp;            // optional
  float* out_ent;             // optional
  float* out_lse;             // optional, natural-log units
  int* status;
};

struct DlParams {
  CUtensorMap tmA, tmB;
  CUtensorMap tmG;            // G chunk buffer: inner columns, outer chunk rows; bf16 G: box 64 x 32,
                              // 128-byte swizzle; fp32 mode (hi and lo terms): box 32 x 32, 64-byte swizzle
  int nseg, kb_per_seg;
  int seg_a[kMaxSeg], seg_b[kMaxSeg];
  int n0, Nc, Rc, V, Vp, Vt;  // chunk start row, rows in chunk (upper bound), row tiles (128 or 256 rows), vocab, padded vocab, vocab tiles
  int a_row0;                 // row of tmA holding the chunk's first row (n0, or 0 for a chunk-sized X buffer)
  const int* rows_total;      // device: rows of the backward operands (chunk rows = clamp(*rows_total - n0, 0, Nc))
  float scale2;
  const float* bias2;
  const int64_t* targets;
  long long v_begin;          // as in FwdParams
  const float* lse2;
  const float* coef;          // dL/dlogp / temperature
  __nv_bfloat16* dl;          // [Nc, ld] chunk buffer (hi terms)
  int ld;                     // row stride in elements
  int lo_off;                 // element offset of the lo terms (fp32 mode), else 0
  float* dbp;                 // bias: [rows/32][V] column sums of G per 32 chunk rows, else null
  // Optional (bf16 G): per row (same index as coef) the fp32 value of the
  // row's target entry of G minus its bf16 rounding.  Rows without a target
  // among these columns are not written (the caller zeroes them).
  float* err;
  int* status;
  unsigned long long limit_ns;
};

// Output D[row][h] = sum_k A[row][k] B[h][k] on CTA pairs: 256 output rows
// by 224 h per tile.  dX: rows = tokens of the chunk, k = vocabulary,
// A = G (K-major), B = W.  dW: rows = vocabulary, k = tokens of the chunk,
// A = G read MN-major, B = X.  B is always read MN-major (h contiguous).
struct HProblem {
  int kb_per_seg;             // k-blocks per product term
  int a_outer0, b_outer0;     // outer (k) coordinate origins of MN-major operands
  int Mt, Ht;                 // 256-row tiles, 448-column h tiles
  int Hout;                   // valid h
  int order;                  // tile numbering: 0 = h tile major, 1 = row tile major
  int a_mn;                   // A operand: 0 = K-major (dX form), 1 = MN-major (dW form)
  int reduce;                 // 0: store, 1: add into the output
  int ksplit;                 // 1, or 2: each tile's k range in two units that both add
                              // into a zeroed output (two addends: the sum is order-free)
  // Optional output column routed elsewhere (xcol_out set): column xcol (>= Hout
  // allowed) of output row r < xrows goes to xcol_out[r] (added when reduce;
  // one tile writes each row).
  // wide = 1: the last h tile's second sub is 240 columns (xcol = Ht * 448).
  int xcol, xrows, wide;
  float* xcol_out;
};
struct HParams {
  CUtensorMap tmA[2];         // K-major: inner k, box 64 x 128 | MN-major: inner row, box 64 x 64
  // Optional (both problems' A operand rows by position): position p is A row
  // row_map[p / 128] + p % 128 (blocks of 128 positions map to 128 consecutive
  // rows), so one box of 128 (dX) or 64 (dW k-block) positions is one plain
  // tile.  row_map covers every block a tile can reach.
  const int* row_map;
  CUtensorMap tmB[2];         // inner h, outer k, box 64 x 64
  CUtensorMap tmB48[2];       // the same maps with box 48 x 64: the last 48 columns of a CTA's
                              // 112 of a sub, placed as in a 64-column box (the rest untouched)
  CUtensorMap tmO[2];         // fp32 output: inner h, outer rows, box 32 x 32, 128-byte swizzle
  HProblem pr[2];             // problem 0 must be the K-major one (a_mn = 0) when both run
  int nprob;                  // 1 or 2
  // Rows of the chunk, read on the device: nc = clamp(*rows_total - n0, 0, nc_max).
  // Problem 0 (dX) has ceil(nc/256) row tiles; problem 1 (dW) ceil(nc/64) k-blocks per term.
  const int* rows_total;
  int n0, nc_max;
  int nseg;
  int seg_a[kMaxSeg], seg_b[kMaxSeg];  // inner-coordinate offsets of each product term
  // Optional (problem 0 of the compacted backward): output row r of the chunk
  // is added straight into dx_out[dx_idx[n0 + r]][...] (row stride dx_ld),
  // with float4 atomic adds when dx_vec, else scalar ones, instead of going
  // through tmO[0].  dx_out must hold zeros there, and at most two additions
  // reach an element (ksplit <= 2), so the sum does not depend on their order.
  const int* dx_idx;
  float* dx_out;
  int dx_nrows;               // rows of dx_out (checked in debug builds)
  int dx_ld;
  int dx_vec;
  // Optional (problem 0): the recompute's target-entry rounding errors
  // (dx_err, indexed like the chunk's rows, n0 + row) are added back in fp32
  // as err * W[target - w_begin] on the first k part, so the dominant
  // c (onehot - p) W term of each dX row carries no bf16 rounding.
  const float* dx_err;
  // Optional (problem 0 with dx_idx): each row's accumulator is first scaled
  // by dx_scale[n0 + row] (the stored-probability backward's -c 2^-lse2 / tau).
  const float* dx_scale;
  const int64_t* dx_tgt;
  const __nv_bfloat16* dx_w;  // bf16 W [dx_wrows, dx_wld]
  long long dx_wbegin;
  int dx_wrows, dx_wld;
  int* status;
  unsigned long long limit_ns;
};

struct LossParams {
  int B, T, loss_type;
  double eps_low, eps_high;   // GMPO log-space bounds, fp32 values widened
  double clip_lo, clip_hi;    // GSPO ratio bounds, fp32 values of 1-eps_low, 1+eps_high
  double beta, inv_tau;
  const void* logp;           // fp64 [N] when logp_is_f64, else fp32
  int logp_is_f64;
  const float* old_logp;
  const float* ref_logp;
  const float* adv;           // [B], or [N] when adv_per_token
  int adv_per_token;
  const uint8_t* mask;
  const uint8_t* emask;       // entropy mask, or null (= mask)
  const double* k3;           // K3 state (threshold at k3[0]) or null
  double* seqres;             // [B][8]
  double* part;               // [B][slices][5] partial sums
  unsigned int* seq_ticket;   // [B], zero on entry
  unsigned int* ticket;       // zero on entry
  int slices;                 // blocks per sequence
  int coef_slices;            // blocks per sequence of the coefficient kernel (0: by T alone)
  float* coef;                // optional: c / tau
  float* dlogp;               // optional: c
  float* out_loss;            // null: write out_sums only
  float* out_metrics;
  // Batch size of the GMPO mean and the GSPO clip fraction: B on one device,
  // every rank's sequences together when the batch is split over ranks.
  double Bg;
  double* out_sums;           // optional: the 8 additive batch sums (see fold_batch)
  int* status;
};

// Persistent launches: ``units`` = independent work units; the grid is the
// number of clusters that can be resident at once (or fewer).  cluster = 1
// or 2 CTAs per 128 * cluster-row tile.
int fwd_resident_clusters(int cluster);
int gemmH_resident_clusters();
// kbx: 128-byte boxes per operand per pipeline stage (2: pair tiles with one K segment)
cudaError_t launch_fwd(const FwdParams& p, int units, int cluster, int kbx, cudaStream_t st);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t st);
// One state slot per row ([N][2] float4, the partial-slot layout) from the
// forward's 2P partial slots of each row: the vocabulary shard's mergeable
// softmax state.
cudaError_t launch_shard_state(const MergeParams& p, float4* state, cudaStream_t st);
// Backward row inputs from the caller's units: lse2[n] = lse[n] log2(e) (the
// kernels' log2 units) and coef[n] = dlogp[n] / temperature.
cudaError_t launch_backward_rows_in(const float* lse, const float* dlogp, int N, double inv_tau, float* lse2,
                                   float* coef, cudaStream_t st);
cudaError_t launch_dl(const DlParams& p, int units, int cluster, int kbx, cudaStream_t st);
cudaError_t launch_gemmH(const HParams& p, int units, cudaStream_t st);
cudaError_t launch_bias2(const void* b, int is_fp32, int V, int Vpad, float scale2, float* out, cudaStream_t st);
cudaError_t launch_split3(const float* src, long long rows, int cols, int Cp, __nv_bfloat16* out, cudaStream_t st);
// Backward row compaction (rows whose coefficient c_n is 0 add nothing to
// dX, dW, db).  Arrays are indexed by compacted row; rows from the total up
// to the next multiple of 256 are zero-filled (target -1).
struct CompactParams {
  int N, Kx, Ncap;            // rows, bf16 row width of X operand, rows allocated (multiple of 256)
  const float* coef;          // [N] c_n / temperature
  const float* lse2;          // [N]
  const int64_t* targets;     // [N]
  const __nv_bfloat16* x;     // [N, Kx] X operand (bf16, or the fp32 split terms)
  int* blk_cnt;               // [compact_groups(N)] scratch
  int* blk_off;               // [compact_groups(N)] scratch
  unsigned int* ticket;       // zeroed before the launch
  int* total;                 // out: compacted rows
  int* idx;                   // [Ncap] compacted row -> original row
  float* coefc;               // [Ncap]
  float* lse2c;               // [Ncap]
  int64_t* tgtc;              // [Ncap]
  __nv_bfloat16* xc;          // optional: [Ncap, Kx] the kept X rows by position (null: not copied)
  float* errc;                // optional: [Ncap] zeroed for kept rows and the tile tail
  int* status;                // device status word (index checks of debug builds)
  float* dx_zero;             // optional: [N, H] gradient buffer the gather sets to zero
  int H;
  int dx_vec;                 // dx_zero is 16-byte aligned and H % 4 == 0
  const uint8_t* done;        // optional: [N] rows already handled (1): not kept here
};

// Backward rows of the stored-probability path: buffer row j holds row n of
// the forward's slot j / 256 (see FwdParams::tmPu).  A row with c != 0 whose
// lse2 lies in [kStoredLse2Min, kStoredLse2Max] is kept; kept rows are numbered
// in buffer order (position p) and get
//   k2 = -(c/tau) 2^-lse2 (so G = k2 pu off the target, as pu = 2^t),
//   k1 = (c/tau)(1 - p_y), the target entry of G,
//   the target entry of pu set to bf16(k1 / k2) and err = k1 - k2 bf16(k1 / k2),
//   rows[p] = j, idx[p] = n, xs[p] = bf16(k2 X[n]) (with xcol set, also k2 in
//   column H), done[n] = 1.
// Positions from the kept count up to the next multiple of 256 get rows = 0,
// idx = -1 and zeros.  Other rows go to the recompute.
constexpr float kStoredLse2Min = -80.f;
constexpr float kStoredLse2Max = 96.f;
struct StoredParams {
  int N, H, V, rows_cap;      // rows_cap = stored tiles * 256 (host upper bound)
  int R;                      // row tiles of the forward without a tile list
  const int* tiles;           // the forward's tile list, or null (slot = tile)
  const int* ntiles;
  int pu_tiles;
  const float* coef;          // [N] c / tau
  const float* lse2;          // [N]
  const double* logp64;       // [N]
  const int64_t* targets;     // [N]
  const __nv_bfloat16* x;     // [N, H]
  __nv_bfloat16* pu;          // [rows_cap, pu_ld]
  int pu_ld;
  __nv_bfloat16* xs;          // [rows_cap, xs_ld] by position
  int xs_ld, xcol;            // row stride of xs (elements); xcol: H (bias: db through dW's GEMM) or -1
  int* rows;                  // [rows_cap / 128 + 1] buffer row of each block of 128 positions
  int* idx;                   // [rows_cap] original row by position, -1 where not kept
  float* k2;                  // [rows_cap]
  float* err;                 // [rows_cap]
  int64_t* tgt;               // [rows_cap]
  int* blk_cnt;               // [rows_cap / 32] scratch
  int* blk_off;               // [rows_cap / 32] scratch
  unsigned int* ticket;       // zeroed before the launch
  uint8_t* done;              // [N], zeroed before the launch
  int* kept;                  // out: kept rows
  int* positions;             // out: positions (rows of the taken 128-row blocks)
};
cudaError_t launch_stored_rows(const StoredParams& p, cudaStream_t st);
// Row counters of a call run in groups of sequences: acc[k] += *c[k] (after a
// group), or *c[k] = acc[k] (after the last).
cudaError_t launch_counters(int* const (&c)[4], int* acc, bool write_back, cudaStream_t st);
int compact_groups(int N);   // 32-row groups
// Row tiles of tile_rows rows holding a row with mask != 0: flags[R], their
// ascending list and count (ticket zeroed before the launch).
cudaError_t launch_tile_scan(const uint8_t* mask, int N, int tile_rows, uint8_t* flags, int* list, int* count,
                             unsigned int* ticket, cudaStream_t st);
cudaError_t launch_compact(const CompactParams& p, cudaStream_t st);
cudaError_t launch_set_total(int* total, int N, cudaStream_t st);
// out[j] = X row idx[n0 + j] for j < kept = clamp(*total - n0, 0, nc), zero rows
// after them up to a whole 256-row tile, at most `rows` (a chunk's X operand rows
// of the recompute, which reads whole tiles of its kept rows).
cudaError_t launch_gather_chunk_rows(const __nv_bfloat16* x, int Kx, const int* idx, const int* total, int n0, int nc,
                                     int rows, __nv_bfloat16* out, cudaStream_t st);
// dst[idx[n0 + j]][:] (+)= src[j][:] for j < clamp(*total - n0, 0, nc_max); H % 4 == 0.
cudaError_t launch_scatter_rows(const float* src, const int* idx, const int* total, int n0, int nc_max, int H,
                                float* dst, bool accumulate, cudaStream_t st);

// db (+)= the recompute's per-32-row column partials of the chunk (DlParams::dbp,
// db_part_rows(Nc) rows of V floats), summed over clamp(*rows_total - n0, 0, Nc) rows.
int db_part_rows(int Nc);
cudaError_t launch_db_reduce(const float* part, const int* rows_total, int n0, int Nc, int V, float* db, int accumulate,
                             cudaStream_t st);
cudaError_t launch_selftest_wait(int* status, unsigned long long limit_ns, cudaStream_t st);

// entropy quantile (K3): a 256-byte state block followed by 4 passes x 2 x 256
// uint32 histogram bins
constexpr int kK3Bytes = 256 + 4 * 512 * 4;
cudaError_t launch_entropy_mask(const float* ent, const uint8_t* mask, long long N, double q, void* k3_ws,
                                uint8_t* emask, cudaStream_t st);
cudaError_t launch_loss(const LossParams& p, cudaStream_t st);
// The entropy quantile split into its passes, for batches whose tokens are
// spread over ranks: pass `pass` histogram of the active keys under the
// state's prefixes (counts [kSelectCounts], zeroed here first); the select
// step from (all ranks' summed) counts; the mask from the final state.
constexpr int kSelectPasses = 4;
constexpr int kSelectCounts = 512;
constexpr int kSelectStateBytes = 256;
cudaError_t launch_entropy_hist(const float* ent, const uint8_t* mask, long long N, int pass, const void* state,
                                uint32_t* counts, cudaStream_t st);
cudaError_t launch_entropy_select(int pass, const uint32_t* counts, double q, void* state, cudaStream_t st);
cudaError_t launch_entropy_apply(const float* ent, const uint8_t* mask, long long N, const void* state,
                                 uint8_t* emask, cudaStream_t st);
int loss_slices(int B, int T, int sms);
int fused_loss_slices(int T);
int coef_slices(int B, int T, int sms);
cudaError_t launch_merge_loss(const MergeParams& mp, const LossParams& p, cudaStream_t st);
// Loss and metrics (p.out_loss, p.out_metrics) from the batch sums of ngroups
// groups of sequences ([ngroups][8] doubles, as written through out_sums),
// added in group order; p.Bg is the whole batch's sequence count.
cudaError_t launch_fold_sums(const double* sums, int ngroups, const LossParams& p, cudaStream_t st);

}  // namespace rl
