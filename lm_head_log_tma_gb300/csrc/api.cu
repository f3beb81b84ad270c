// Host side of the C ABI declared in include/rlloss.h: validation, the
// work plan (tiles, vocabulary segments, backward chunks), the workspace
// layout, TMA tensor maps and the launch sequence on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <vector>
#include <cstdint>
#include <cstring>

#include "kernels.h"
#include "status.h"

namespace {

using namespace rl;

constexpr unsigned long long kWaitLimitNs = 4000000000ull;  // 4 s per wait
// Status region (first 256 bytes of every workspace): [0] device status word,
// [4] loss-stage batch ticket, [8] compaction ticket, [12] backward rows,
// [16] tile-scan ticket, [20] forward row tiles, [24] forward vocabulary segments,
// [28] stored-probability kept rows, [32] its ticket, [36] its positions.
constexpr size_t kBackwardRowsOffset = 12;
constexpr size_t kTileTicketOffset = 16, kFwdTilesOffset = 20, kFwdSegmentsOffset = 24;
constexpr size_t kStoredRowsOffset = 28;   // kept rows of the stored-probability backward
constexpr size_t kStoredTicketOffset = 32;
constexpr size_t kStoredPositionsOffset = 36;   // rows it ran over (taken 128-row blocks)
constexpr size_t kPartialCapBytes = size_t(64) << 20;

inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }
inline long long rup(long long a, long long b) { return cdiv(a, b) * b; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 152;
  }
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();
    return 152;
  }
  return sms;
}

bool finite(float x) { return std::isfinite(x); }

// Resident-cluster count from the runtime, or a fallback when no device is
// usable (host-only sizing).
int resident_or(int n, int fallback) {
  if (n > 0) return n;
  cudaGetLastError();
  return std::max(1, fallback);
}

int validate_common(const rlloss_cfg* c) {
  if (!c) return RLLOSS_EINVAL;
  if (c->B < 1 || c->T < 1) return RLLOSS_EINVAL;
  if ((long long)c->B * c->T > (1ll << 31) - 1) return RLLOSS_EINVAL;
  if (c->loss_type != RLLOSS_GMPO && c->loss_type != RLLOSS_GSPO_TOKEN) return RLLOSS_EINVAL;
  if (c->is_level != RLLOSS_IS_TOKEN && c->is_level != RLLOSS_IS_SEQUENCE) return RLLOSS_EINVAL;
  if (c->loss_type == RLLOSS_GMPO && c->is_level == RLLOSS_IS_SEQUENCE) return RLLOSS_EINVAL;
  if (!finite(c->eps_low) || !finite(c->eps_high) || c->eps_low < 0.f || c->eps_high < 0.f) return RLLOSS_EINVAL;
  if (!finite(c->beta)) return RLLOSS_EINVAL;
  const float q = c->top_entropy_quantile;
  if (!(q >= 0.f && q <= 1.f)) return RLLOSS_EINVAL;
  if (c->flags & ~(RLLOSS_FLAG_FORCE_ENTROPY_PATH | RLLOSS_FLAG_SINGLE_CTA_TILES | RLLOSS_FLAG_ADV_PER_TOKEN |
                   RLLOSS_FLAG_ALL_ROWS | RLLOSS_FLAG_ACCUMULATE | RLLOSS_FLAG_RECOMPUTE))
    return RLLOSS_EINVAL;
  if ((c->flags & RLLOSS_FLAG_ADV_PER_TOKEN) && c->loss_type != RLLOSS_GSPO_TOKEN) return RLLOSS_EUNSUPPORTED;
  if (c->loss_type == RLLOSS_GSPO_TOKEN) {
    if (c->beta != 0.f) return RLLOSS_EUNSUPPORTED;
    if (q < 1.f || (c->flags & RLLOSS_FLAG_FORCE_ENTROPY_PATH)) return RLLOSS_EUNSUPPORTED;
  }
  return RLLOSS_OK;
}

// LM-head part of a configuration (shapes, dtype, temperature, bias).
int validate_head(const rlloss_cfg* c) {
  if (!c) return RLLOSS_EINVAL;
  if (c->B < 1 || c->T < 1) return RLLOSS_EINVAL;
  if ((long long)c->B * c->T > (1ll << 31) - 1) return RLLOSS_EINVAL;
  if (c->flags & ~(RLLOSS_FLAG_FORCE_ENTROPY_PATH | RLLOSS_FLAG_SINGLE_CTA_TILES | RLLOSS_FLAG_ADV_PER_TOKEN |
                   RLLOSS_FLAG_ALL_ROWS | RLLOSS_FLAG_ACCUMULATE | RLLOSS_FLAG_RECOMPUTE))
    return RLLOSS_EINVAL;
  if (c->H < 1 || c->V < 1) return RLLOSS_EINVAL;
  if (c->dtype != RLLOSS_BF16 && c->dtype != RLLOSS_FP32 && c->dtype != RLLOSS_FP8_E4M3) return RLLOSS_EINVAL;
  if (!(c->temperature > 0.f) || !finite(c->temperature)) return RLLOSS_EINVAL;
  if (c->has_bias != 0 && c->has_bias != 1) return RLLOSS_EINVAL;
  if (c->chunk_rows < 0) return RLLOSS_EINVAL;
  if (c->dtype == RLLOSS_BF16 && (c->H % 8) != 0) return RLLOSS_EUNSUPPORTED;  // TMA row stride: 16 bytes
  if (c->dtype == RLLOSS_FP8_E4M3) {
    if ((c->H % 16) != 0) return RLLOSS_EUNSUPPORTED;                          // TMA row stride: 16 bytes
    if (c->flags & RLLOSS_FLAG_SINGLE_CTA_TILES) return RLLOSS_EUNSUPPORTED;
  }
  if ((c->H % 4) != 0) return RLLOSS_EUNSUPPORTED;                            // fp32 dX / dW rows: 16 bytes
  if (c->H > 65536 || c->V > (1 << 30)) return RLLOSS_EUNSUPPORTED;
  return RLLOSS_OK;
}

int validate_full(const rlloss_cfg* c) {
  int e = validate_common(c);
  if (e) return e;
  e = validate_head(c);
  if (e) return e;
  if (c->dtype == RLLOSS_FP8_E4M3) return RLLOSS_EUNSUPPORTED;   // e4m3: forward-only scoring
  return RLLOSS_OK;
}

bool entropy_path(const rlloss_cfg* c) {
  return c->top_entropy_quantile < 1.f || (c->flags & RLLOSS_FLAG_FORCE_ENTROPY_PATH);
}

struct Plan {
  int B, T, N, H, V, sms;
  int pair, rows_tile;      // CTAs per LM-head tile (1 or 2) and rows per tile
  int fwd_clusters, h_pairs;  // resident clusters of the forward and dX/dW kernels
  bool fp32, f8, bias, ent;
  bool fused_loss;          // row merge and loss stage in one launch (no entropy mask)
  bool compact;             // backward over the rows with c_n != 0 only
  int R, Vt, P, pcap, Hp, Vp;
  int kb_fwd, nseg_fwd;     // forward K: nseg_fwd * kb_fwd k-blocks
  int kbx;                  // 128-byte boxes per operand per stage of the forward and recompute
  int kb_dl;                // recompute K-blocks per product term
  int Kx;                   // row width (elements) of the bf16 X / W operand arrays
  int Nc, nchunks, ld_dl;
  // workspace offsets
  int slices;
  size_t o_tickets, o_part;
  size_t o_status, o_partial, o_lse2, o_logp64, o_ent, o_coef, o_emask, o_k3, o_seq, o_bias2, o_dl, o_x3, o_w3,
      o_dbpart, o_ws2, o_tflags, o_tlist, o_blk, o_cidx, o_xc, o_coefc, o_lse2c, o_tgtc, o_dxc, o_err, total;
  int Ncap;                 // rows of the compacted arrays (N rounded up to 256)
  // Stored probabilities: the forward writes 2^t for the row tiles of its
  // first pu_tiles slots into the chunk buffer, and the backward of their
  // rows needs no recompute (bf16 CTA pairs, no bias, no ACCUMULATE).
  bool stored;
  int pu_tiles;
  int xs_ld;                // row stride (elements) of the stored path's scaled X rows
  size_t o_done;
  int seq_group, ngroups;   // sequences per group of a grouped call (0: one pass), groups
  size_t o_sums;            // grouped call: [ngroups][8] batch sums, then 4 int row counters
};

// Largest vocabulary-segment count whose partial states fit the cap (<= 64).
int segment_cap(long long N) {
  long long c = (long long)(kPartialCapBytes / (size_t(N) * 2 * 32));
  if (c > 64) c = 64;
  return c < 1 ? 1 : int(c);
}

// kShardLoss: loss stage over row states gathered from vocabulary shards (row
// buffers, no LM head); kBackwardOnly: the backward of one vocabulary shard
// from given lse and dL/dlogp (LM-head operands and backward buffers only).
enum PlanMode { kFull, kLossOnly, kForwardOnly, kShardLoss, kBackwardOnly };

Plan make_plan(const rlloss_cfg* c, PlanMode mode) {
  const bool head = mode != kLossOnly && mode != kShardLoss;        // LM-head operands
  const bool fwd = head && mode != kBackwardOnly;                   // LM-head forward kernels
  const bool loss = mode != kForwardOnly && mode != kBackwardOnly;  // loss stage
  const bool bwd = mode == kFull || mode == kBackwardOnly;          // backward chunks
  Plan p{};
  p.B = c->B;
  p.T = c->T;
  p.N = c->B * c->T;
  p.sms = device_sms();
  p.ent = entropy_path(c);
  p.fused_loss = mode == kFull && !p.ent;
  // ---- LM-head parameters
  if (head) {
    p.H = c->H;
    p.V = c->V;
    p.fp32 = c->dtype == RLLOSS_FP32;
    p.f8 = c->dtype == RLLOSS_FP8_E4M3;
    p.bias = c->has_bias != 0;
    p.pair = (c->flags & RLLOSS_FLAG_SINGLE_CTA_TILES) ? 1 : 2;
    p.rows_tile = 128 * p.pair;
    p.R = int(cdiv(p.N, p.rows_tile));
    p.Vt = int(cdiv(p.V, 256));
    p.fwd_clusters = resident_or(fwd_resident_clusters(p.pair), p.sms / p.pair);
    p.Hp = int(rup(p.H, 64));
    p.Vp = int(rup(p.V, 64));
    // Stages hold two 128-byte boxes per operand with CTA pairs and one K
    // segment (bf16, e4m3), one box otherwise (fp32 split terms: K segments
    // of Hp elements; single-CTA tiles).
    p.kbx = (p.pair == 2 && !p.fp32) ? 2 : 1;
    if (p.fp32) {
      p.nseg_fwd = 6;
      p.kb_fwd = p.Hp / 64;
      p.Kx = 3 * p.Hp;
    } else if (p.f8) {
      p.nseg_fwd = 1;
      p.kb_fwd = int(cdiv(p.H, 128 * p.kbx));   // 128 e4m3 elements per 128-byte box row
      p.Kx = p.H;
    } else {
      p.nseg_fwd = 1;
      p.kb_fwd = int(cdiv(p.H, 64 * p.kbx));
      p.Kx = p.H;
    }
    p.kb_dl = p.fp32 ? p.Hp / 64 : int(cdiv(p.H, 64 * p.kbx));
  }
  // ---- backward parameters: chunk buffer, stored probabilities, sequence groups
  if (bwd) {
    p.h_pairs = resident_or(gemmH_resident_clusters(), p.sms / 2);
    // Default chunk: a whole number of dX units per pair of SMs (one or two
    // waves of 256-row x 448-h tiles, each in two k halves).
    const int hts = int(cdiv(p.H, 448));
    const int per_wave = 256 * std::max(1, p.h_pairs / (2 * hts));
    const int base_chunk = p.N > 2 * per_wave ? 2 * per_wave : per_wave;
    const int want = c->chunk_rows > 0 ? int(rup(c->chunk_rows, 256)) : std::max(base_chunk, 1024);
    p.Nc = int(std::min<long long>(want, rup(p.N, 128)));
    p.nchunks = int(cdiv(p.N, p.Nc));
    p.ld_dl = p.fp32 ? 2 * p.Vp : p.Vp;
    p.compact = !(c->flags & RLLOSS_FLAG_ALL_ROWS);
    p.stored = mode == kFull && !p.fp32 && !p.f8 && p.pair == 2 && p.kbx == 2 && p.compact &&
               !(c->flags & (RLLOSS_FLAG_ACCUMULATE | RLLOSS_FLAG_RECOMPUTE));
    // scaled X rows of the stored path: H columns, plus k2 in column H (and
    // zeros to a 16-byte multiple) with a bias, so dW's GEMM also forms db
    p.xs_ld = p.stored && p.bias ? p.H + 8 : p.Kx;
    p.pu_tiles = p.stored ? int(cdiv(p.Nc, 256)) : 0;
    // Whole sequences per group when the batch runs in groups that each fit the
    // stored-probability buffer (no batch-global entropy threshold couples them;
    // whole 256-row tiles per sequence); 0: one pass over the batch.
    p.seq_group = 0;
    if (p.stored && !p.ent && c->T % 256 == 0 && !(c->flags & RLLOSS_FLAG_ADV_PER_TOKEN)) {
      const int s = p.pu_tiles * 256 / c->T;
      if (s >= 1 && s < c->B) p.seq_group = s;
    }
    p.ngroups = p.seq_group ? int(cdiv(c->B, p.seq_group)) : 1;
    if (p.seq_group) {   // the buffer holds exactly one group (and a recompute chunk never needs more)
      p.Nc = p.seq_group * c->T;
      p.pu_tiles = p.Nc / 256;
      p.nchunks = int(cdiv(p.N, p.Nc));
    }
  }
  // ---- regions.  Per-row regions hold one group's rows when the call runs in
  // groups (the groups reuse them in turn), else the whole batch's.
  const long long Nr = p.seq_group ? (long long)p.seq_group * p.T : p.N;
  const int Rr = head ? int(cdiv(Nr, p.rows_tile)) : 0;
  if (head) {
    p.pcap = segment_cap(Nr);
    p.P = choose_segments(p.R, p.Vt, p.fwd_clusters, p.pcap);
  }
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  p.o_status = take(256);
  if (loss) {
    p.o_tickets = take(size_t(p.B) * 4);
    p.slices = p.fused_loss ? fused_loss_slices(p.T) : loss_slices(p.B, p.T, p.sms);
    p.o_part = take(size_t(p.B) * p.slices * 5 * 8);
  }
  if (head) {
    if (fwd) {
      p.o_partial = take(size_t(Nr) * 2 * p.pcap * 32);   // room for a segment count chosen on the device
      p.o_logp64 = take(size_t(Nr) * 8);
      p.o_ent = take(size_t(Nr) * 4);
    }
    p.o_lse2 = take(size_t(Nr) * 4);
    p.o_bias2 = take(p.bias ? size_t(p.Vt) * 256 * 4 : 0);
    p.o_ws2 = take(p.f8 ? size_t(p.Vt) * 256 * 4 : 0);
    p.o_x3 = take(p.fp32 ? size_t(p.N) * 3 * p.Hp * 2 : 0);
    p.o_w3 = take(p.fp32 ? size_t(p.V) * 3 * p.Hp * 2 : 0);
  }
  if (mode == kShardLoss) {
    p.V = c->V;
    p.o_lse2 = take(size_t(p.N) * 4);
    p.o_logp64 = take(size_t(p.N) * 8);
    p.o_ent = take(size_t(p.N) * 4);
  }
  if (loss) {
    p.o_emask = take(size_t(Nr));
    p.o_k3 = take(kK3Bytes);
    p.o_seq = take(size_t(p.B) * 10 * 8);   // sequence records, 10 doubles each
  }
  if (bwd) {
    p.o_coef = take(size_t(Nr) * 4);
    p.o_dl = take(size_t(std::max(p.Nc, p.pu_tiles * 256)) * p.ld_dl * 2);
    p.o_dbpart = take(p.bias ? size_t(db_part_rows(p.Nc)) * p.V * 4 : 0);
    p.o_done = take(p.stored ? size_t(Nr) : 0);
    p.o_sums = take(p.seq_group ? size_t(p.ngroups) * 8 * 8 + 64 : 0);
    // bf16 G: each backward row's target-entry rounding error (rows or
    // compacted rows, N rounded up to whole 256-row tiles)
    p.o_err = take(p.fp32 ? 0 : size_t(rup(Nr, 256)) * 4);
    p.o_tflags = take(size_t(Rr));
    p.o_tlist = take(size_t(Rr) * 4);
    if (p.compact) {
      p.Ncap = int(rup(Nr, 256));
      p.o_blk = take(size_t(compact_groups(int(std::max<long long>(Nr, (long long)p.pu_tiles * 256)))) * 2 * 4);
      p.o_cidx = take(size_t(p.Ncap) * 4);
      p.o_coefc = take(size_t(p.Ncap) * 4);
      p.o_lse2c = take(size_t(p.Ncap) * 4);
      p.o_tgtc = take(size_t(p.Ncap) * 8);
      // X operand rows of one backward chunk (the recompute gathers each chunk's
      // kept rows before its launch), or the stored path's scaled rows
      p.o_xc = take(size_t(rup(std::max(p.Nc, p.pu_tiles * 256), 256)) * std::max(p.Kx, p.xs_ld) * 2);
      p.o_dxc = take(size_t(p.Nc) * p.H * 4);
    }
  }
  p.total = off;
  return p;
}

// ------------------------------------------------------------------ instrumentation
std::atomic<uint64_t> g_launches{0};

struct PhaseRec {
  int phase;
  int launches;
  cudaEvent_t a, b;
};
struct PhaseTimer {
  std::mutex mu;
  bool on = false;
  std::vector<PhaseRec> recs;
  std::vector<cudaEvent_t> pool;
  cudaEvent_t get() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
};
PhaseTimer g_timer;

// Records an event pair around one phase when timing is on; counts launches.
struct Phase {
  cudaStream_t st;
  int phase;
  int n = 0;
  cudaEvent_t a = nullptr;
  Phase(cudaStream_t s, int ph) : st(s), phase(ph) {
    std::lock_guard<std::mutex> g(g_timer.mu);
    if (g_timer.on) {
      a = g_timer.get();
      cudaEventRecord(a, st);
    }
  }
  void launched(int k = 1) {
    n += k;
    g_launches += uint64_t(k);
  }
  ~Phase() {
    std::lock_guard<std::mutex> g(g_timer.mu);
    if (a) {
      cudaEvent_t b = g_timer.get();
      cudaEventRecord(b, st);
      g_timer.recs.push_back(PhaseRec{phase, n, a, b});
    }
  }
};

// ------------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D bf16 map; OOB reads return 0 and OOB parts of stores are dropped.
bool tmap_bf16_box(CUtensorMap* m, const void* base, long long inner, long long outer, long long row_elems,
                   int box_inner, int box_outer, CUtensorMapSwizzle swz) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
  const cuuint64_t strides[1] = {cuuint64_t(row_elems) * 2};
  const cuuint32_t box[2] = {cuuint32_t(box_inner), cuuint32_t(box_outer)};
  const cuuint32_t es[2] = {1u, 1u};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand map: 128-byte swizzle, box {64, box_outer}.
bool tmap_bf16(CUtensorMap* m, const void* base, long long inner, long long outer, long long row_elems,
               int box_outer) {
  return tmap_bf16_box(m, base, inner, outer, row_elems, 64, box_outer, CU_TENSOR_MAP_SWIZZLE_128B);
}

// 2-D byte (e4m3) operand map: rows of `inner` bytes, box 128 bytes x box_outer,
// 128-byte swizzle (the same shared-memory layout as a 64-wide bf16 box).
bool tmap_u8(CUtensorMap* m, const void* base, long long inner, long long outer, int box_outer) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
  const cuuint64_t strides[1] = {cuuint64_t(inner)};
  const cuuint32_t box[2] = {128u, cuuint32_t(box_outer)};
  const cuuint32_t es[2] = {1u, 1u};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 output map for TMA stores / reduce-adds: box 32 x 32, 128-byte swizzle.
bool tmap_f32_out(CUtensorMap* m, const float* base, long long inner, long long outer) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
  const cuuint64_t strides[1] = {cuuint64_t(inner) * 4};
  const cuuint32_t box[2] = {32u, 32u};
  const cuuint32_t es[2] = {1u, 1u};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? RLLOSS_OK : RLLOSS_ECUDA; }
#define RL_TRY(x)                    \
  do {                               \
    cudaError_t _e = (x);            \
    if (_e != cudaSuccess) return RLLOSS_ECUDA; \
  } while (0)

// K-segments of the dX / dW GEMMs.  bf16: one product.  fp32: G = G_hi + G_lo
// and W (or X) = hi + mid + lo; the products G_hi*hi, G_hi*mid, G_lo*hi.
void set_bwd_segments(HParams& hp, const Plan& p) {
  if (p.fp32) {
    hp.nseg = 3;
    hp.seg_a[0] = 0;    hp.seg_b[0] = 0;
    hp.seg_a[1] = 0;    hp.seg_b[1] = p.Hp;
    hp.seg_a[2] = p.Vp; hp.seg_b[2] = 0;
  } else {
    hp.nseg = 1;
  }
}

LossParams loss_params(const rlloss_cfg* c, const Plan& p, char* ws) {
  LossParams lp{};
  lp.B = c->B;
  lp.T = c->T;
  lp.loss_type = c->loss_type;
  lp.eps_low = double(c->eps_low);
  lp.eps_high = double(c->eps_high);
  lp.clip_lo = double(1.0f - c->eps_low);
  lp.clip_hi = double(1.0f + c->eps_high);
  lp.beta = double(c->beta);
  lp.inv_tau = 1.0 / double(c->temperature > 0.f ? c->temperature : 1.f);
  lp.seqres = reinterpret_cast<double*>(ws + p.o_seq);
  lp.part = reinterpret_cast<double*>(ws + p.o_part);
  lp.seq_ticket = reinterpret_cast<unsigned int*>(ws + p.o_tickets);
  lp.slices = p.slices;
  lp.coef_slices = coef_slices(c->B, c->T, p.sms > 0 ? p.sms : 1);
  lp.ticket = reinterpret_cast<unsigned int*>(ws + p.o_status + 4);
  lp.status = reinterpret_cast<int*>(ws + p.o_status);
  lp.k3 = p.ent ? reinterpret_cast<const double*>(ws + p.o_k3) : nullptr;
  lp.adv_per_token = (c->flags & RLLOSS_FLAG_ADV_PER_TOKEN) ? 1 : 0;
  lp.Bg = double(c->B);
  return lp;
}

// The LM-head forward shared by rlloss_fwd_bwd and rlloss_forward: operand
// preparation (fp32 split, scaled bias), the tensor-core forward, and the
// row merge into lse, logp and entropy.
struct Head {
  const void* Xop = nullptr;
  const void* Wop = nullptr;
  const float* bias2 = nullptr;
  const float* x_scale = nullptr;   // e4m3 operands: per-row scales (set by the caller of run_head)
  const float* w_scale = nullptr;
  int seg_a[kMaxSeg] = {0, 0, 0, 0, 0, 0};
  int seg_b[kMaxSeg] = {0, 0, 0, 0, 0, 0};
  FwdParams fp{};
  MergeParams mp{};
};

#define RL_TRY_RC(x)             \
  do {                           \
    const int _rc = (x);         \
    if (_rc != RLLOSS_OK) return _rc; \
  } while (0)

// Operand preparation of the LM head (fp32 split, scaled bias, e4m3 column
// scales), the K-segments and the forward's tensor maps; launches no GEMM.
int prepare_head(const rlloss_cfg* cfg, const Plan& p, const void* X, const void* W, const void* b, char* ws,
                 cudaStream_t st, Head& h) {
  const float scale2 = float(1.4426950408889634 / double(cfg->temperature));
  // Operand arrays: bf16 inputs are used in place; fp32 inputs are split
  // into three bf16 terms (hi, mid, lo) so the same bf16 tensor-core kernels
  // reach fp32-level accuracy (six of the nine term products are kept).
  h.Xop = X;
  h.Wop = W;
  if (p.fp32) {
    __nv_bfloat16* x3 = reinterpret_cast<__nv_bfloat16*>(ws + p.o_x3);
    __nv_bfloat16* w3 = reinterpret_cast<__nv_bfloat16*>(ws + p.o_w3);
    Phase ph(st, 5);
    RL_TRY(launch_split3(static_cast<const float*>(X), p.N, p.H, p.Hp, x3, st));
    RL_TRY(launch_split3(static_cast<const float*>(W), p.V, p.H, p.Hp, w3, st));
    ph.launched(2);
    h.Xop = x3;
    h.Wop = w3;
  }
  if (p.bias) {
    float* b2 = reinterpret_cast<float*>(ws + p.o_bias2);
    Phase ph(st, 5);
    RL_TRY(launch_bias2(b, (p.fp32 || p.f8) ? 1 : 0, p.V, p.Vt * 256, scale2, b2, st));
    ph.launched();
    h.bias2 = b2;
  }
  float* ws2 = nullptr;
  if (p.f8) {   // w_scale * log2(e) / tau, zero padded (same layout as the scaled bias)
    ws2 = reinterpret_cast<float*>(ws + p.o_ws2);
    Phase ph(st, 5);
    RL_TRY(launch_bias2(h.w_scale, 1, p.V, p.Vt * 256, scale2, ws2, st));
    ph.launched();
  }
  // K-segments of the forward / recompute GEMM: products of the split terms.
  if (p.fp32) {
    const int hp = p.Hp;
    const int sa[6] = {0, 0, hp, 0, hp, 2 * hp};   // hi*hi, hi*mid, mid*hi, hi*lo, mid*mid, lo*hi
    const int sb[6] = {0, hp, 0, 2 * hp, hp, 0};
    std::memcpy(h.seg_a, sa, sizeof(sa));
    std::memcpy(h.seg_b, sb, sizeof(sb));
  }

  FwdParams& fp = h.fp;
  fp.ws2 = ws2;
  if (p.f8) {
    if (!tmap_u8(&fp.tmA, h.Xop, p.Kx, p.N, 128)) return RLLOSS_ECUDA;
    if (!tmap_u8(&fp.tmB, h.Wop, p.Kx, p.V, 128)) return RLLOSS_ECUDA;
    fp.xs = h.x_scale;
  } else {
    if (!tmap_bf16(&fp.tmA, h.Xop, p.Kx, p.N, p.Kx, 128)) return RLLOSS_ECUDA;
    if (!tmap_bf16(&fp.tmB, h.Wop, p.Kx, p.V, p.Kx, p.pair == 1 ? 256 : 128)) return RLLOSS_ECUDA;
  }
  fp.nseg = p.nseg_fwd;
  fp.kb_per_seg = p.kb_fwd;
  std::memcpy(fp.seg_a, h.seg_a, sizeof(h.seg_a));
  std::memcpy(fp.seg_b, h.seg_b, sizeof(h.seg_b));
  fp.N = p.N;
  fp.V = p.V;
  fp.R = p.R;
  fp.Vt = p.Vt;
  fp.P = p.P;
  fp.scale2 = scale2;
  fp.bias2 = h.bias2;
  fp.partial = reinterpret_cast<float4*>(ws + p.o_partial);
  fp.pcap = p.pcap;
  fp.status = reinterpret_cast<int*>(ws + p.o_status);
  fp.limit_ns = kWaitLimitNs;
  return RLLOSS_OK;
}

// With merge == false the row merge is left to the caller (the fused merge +
// loss launch); h.mp is filled either way.
// With skip_mask set, the forward runs only over row tiles that hold a row
// with skip_mask != 0 (the rows of the other tiles get no outputs).
// v_begin: vocabulary id of W's first row when W is a shard of a larger
// vocabulary (targets outside the shard match no column).
// With p.stored the forward also writes the stored probabilities of its first
// p.pu_tiles row-tile slots into the chunk buffer.
int run_head(const rlloss_cfg* cfg, const Plan& p, const void* X, const void* W, const void* b,
             const int64_t* targets, float* out_logp, float* out_entropy, float* out_lse, char* ws,
             cudaStream_t st, Head& h, bool merge = true, const uint8_t* skip_mask = nullptr,
             long long v_begin = 0) {
  int* status = reinterpret_cast<int*>(ws + p.o_status);
  RL_TRY_RC(prepare_head(cfg, p, X, W, b, ws, st, h));
  // ---- forward: tensor-core logits + streamed row state
  FwdParams& fp = h.fp;
  fp.targets = targets;
  fp.v_begin = v_begin;
  if (p.stored) {
    if (!tmap_bf16_box(&fp.tmPu, ws + p.o_dl, p.V, (long long)p.pu_tiles * 256, p.ld_dl, 32, 32,
                       CU_TENSOR_MAP_SWIZZLE_64B))
      return RLLOSS_ECUDA;
    fp.pu_tiles = p.pu_tiles;
  }
  const uint8_t* tflags = nullptr;
  if (skip_mask) {
    tflags = reinterpret_cast<uint8_t*>(ws + p.o_tflags);
    int* tlist = reinterpret_cast<int*>(ws + p.o_tlist);
    int* ntiles = reinterpret_cast<int*>(ws + p.o_status + kFwdTilesOffset);
    Phase ph(st, 5);
    RL_TRY(launch_tile_scan(skip_mask, p.N, p.rows_tile, const_cast<uint8_t*>(tflags), tlist, ntiles,
                            reinterpret_cast<unsigned int*>(ws + p.o_status + kTileTicketOffset), st));
    ph.launched();
    fp.tiles = tlist;
    fp.ntiles = ntiles;
    fp.P_out = reinterpret_cast<int*>(ws + p.o_status + kFwdSegmentsOffset);
  } else {
    RL_TRY(launch_set_total(reinterpret_cast<int*>(ws + p.o_status + kFwdTilesOffset), p.R, st));
    g_launches += 1;
  }
  {
    Phase ph(st, 0);
    RL_TRY(launch_fwd(fp, p.R * p.P, p.pair, p.kbx, st));
    ph.launched();
  }
  MergeParams& mp = h.mp;
  mp.partial = fp.partial;
  mp.N = p.N;
  mp.V = p.V;
  mp.slots = 2 * p.P;
  if (skip_mask) {
    mp.P_dev = fp.P_out;
    mp.tile_active = tflags;
    mp.tile_shift = p.rows_tile == 256 ? 8 : 7;
  }
  mp.targets = targets;
  mp.lse2 = reinterpret_cast<float*>(ws + p.o_lse2);
  mp.logp64 = reinterpret_cast<double*>(ws + p.o_logp64);
  mp.ent32 = reinterpret_cast<float*>(ws + p.o_ent);
  mp.out_logp = out_logp;
  mp.out_ent = out_entropy;
  mp.out_lse = out_lse;
  mp.status = status;
  if (merge) {
    Phase ph(st, 1);
    RL_TRY(launch_merge(mp, st));
    ph.launched();
  }
  return RLLOSS_OK;
}

// The backward from per-row lse (log2 units) and coefficients c_n (G = (c/tau)
// (onehot(y) - p)): row compaction, then per chunk the G recompute and the
// grouped dX / dW GEMMs, and db.  hd holds the prepared operands.
// With add_dw set (a later group of sequences of a grouped call), dW and db
// are added to instead of stored by the stored-probability launch.
int run_backward(const rlloss_cfg* cfg, const Plan& p, const Head& hd, const int64_t* targets, long long v_begin,
                 const float* lse2, const float* coef, float* dX, float* dW, float* db, char* ws, cudaStream_t st,
                 bool add_dw = false) {
  int* status = reinterpret_cast<int*>(ws + p.o_status);
  // ---- backward, one chunk of rows at a time:
  //      G = (c/tau)(onehot - p) as bf16, dX = G W, dW += G^T X, db += sum G.
  // Rows with c_n = 0 add nothing to any of the three; unless the caller asks
  // for the dense backward they are dropped first (ordered compaction), the
  // chunks run over the kept rows, and dX rows are scattered back (the rest
  // of dX is zero).  The kept-row count stays on the device: every backward
  // kernel reads it, and chunks past it do no work.  With ACCUMULATE every
  // output element still receives one addition per chunk (dX rows: one per
  // call), so the sums keep a fixed order.
  const bool acc = (cfg->flags & RLLOSS_FLAG_ACCUMULATE) != 0;
  // Compacted backward without ACCUMULATE: the dX rows of each chunk are added
  // straight into the zeroed dX at their original rows (two k halves, two
  // addends); with ACCUMULATE they go through the chunk buffer and a
  // read-add-write scatter, so each dX element gets one addition per call.
  const bool dx_direct = p.compact && !acc;
  const bool dx_vec = p.H % 4 == 0 && (reinterpret_cast<uintptr_t>(dX) & 15u) == 0;
  float* err = p.fp32 ? nullptr : reinterpret_cast<float*>(ws + p.o_err);
  __nv_bfloat16* dl = reinterpret_cast<__nv_bfloat16*>(ws + p.o_dl);
  const int lo_off = p.fp32 ? p.Vp : 0;
  int* rows_total = reinterpret_cast<int*>(ws + p.o_status + kBackwardRowsOffset);
  const void* Xb = hd.Xop;           // X operand rows of the backward
  const int64_t* tg_b = targets;
  const float* lse2_b = lse2;
  const float* coef_b = coef;
  const int* cidx = nullptr;
  float* dxc = nullptr;
  long long xb_rows = p.N;
  uint8_t* done = nullptr;
  if (p.stored) {
    // ---- rows whose probabilities the forward stored: no recompute.
    //   G = k2 pu off the target and k1 at it (StoredParams), so
    //   dX = k2 (pu W) + err W[target] with pu's target entry bf16(k1 / k2),
    //   dW = pu^T (k2 X), both in one grouped launch over the stored rows.
    done = reinterpret_cast<uint8_t*>(ws + p.o_done);
    int* srows = reinterpret_cast<int*>(ws + p.o_status + kStoredRowsOffset);
    __nv_bfloat16* pu = reinterpret_cast<__nv_bfloat16*>(ws + p.o_dl);
    const int pu_rows = p.pu_tiles * 256;
    StoredParams sp{};
    sp.N = p.N;
    sp.H = p.H;
    sp.V = p.V;
    sp.rows_cap = pu_rows;
    sp.R = p.R;
    sp.tiles = hd.fp.tiles;
    sp.ntiles = hd.fp.ntiles;
    sp.pu_tiles = p.pu_tiles;
    sp.coef = coef;
    sp.lse2 = lse2;
    sp.logp64 = reinterpret_cast<const double*>(ws + p.o_logp64);
    sp.targets = targets;
    sp.x = static_cast<const __nv_bfloat16*>(hd.Xop);
    sp.pu = pu;
    sp.pu_ld = p.ld_dl;
    sp.xs = reinterpret_cast<__nv_bfloat16*>(ws + p.o_xc);
    sp.xs_ld = p.xs_ld;
    sp.xcol = p.bias ? p.H : -1;
    sp.rows = reinterpret_cast<int*>(ws + p.o_lse2c);   // buffer row by position
    sp.idx = reinterpret_cast<int*>(ws + p.o_cidx);
    sp.k2 = reinterpret_cast<float*>(ws + p.o_coefc);
    sp.err = err;
    sp.tgt = reinterpret_cast<int64_t*>(ws + p.o_tgtc);
    sp.blk_cnt = reinterpret_cast<int*>(ws + p.o_blk);
    sp.blk_off = sp.blk_cnt + compact_groups(pu_rows);
    sp.ticket = reinterpret_cast<unsigned int*>(ws + p.o_status + kStoredTicketOffset);
    sp.done = done;
    sp.kept = srows;
    sp.positions = reinterpret_cast<int*>(ws + p.o_status + kStoredPositionsOffset);
    {
      Phase ph(st, 5);
      RL_TRY(cudaMemsetAsync(dX, 0, size_t(p.N) * p.H * 4, st));
      RL_TRY(cudaMemsetAsync(done, 0, size_t(p.N), st));   // rows_valid: zeroed with the status block
      RL_TRY(launch_stored_rows(sp, st));
      ph.launched(2);
    }
    HParams hp{};
    set_bwd_segments(hp, p);
    // both problems read their A rows (the stored probabilities) by position
    hp.row_map = sp.rows;
    if (!tmap_bf16(&hp.tmA[0], pu, p.V, pu_rows, p.ld_dl, 128)) return RLLOSS_ECUDA;
    if (!tmap_bf16(&hp.tmB[0], hd.Wop, p.Kx, p.V, p.Kx, 64)) return RLLOSS_ECUDA;
    if (!tmap_bf16_box(&hp.tmB48[0], hd.Wop, p.Kx, p.V, p.Kx, 48, 64, CU_TENSOR_MAP_SWIZZLE_128B))
      return RLLOSS_ECUDA;
    if (!tmap_f32_out(&hp.tmO[0], dX, p.H, p.N)) return RLLOSS_ECUDA;   // unused: rows go through dx_idx
    if (!tmap_bf16(&hp.tmA[1], pu, p.V, pu_rows, p.ld_dl, 64)) return RLLOSS_ECUDA;
    if (!tmap_bf16(&hp.tmB[1], sp.xs, p.H + (p.bias ? 1 : 0), pu_rows, p.xs_ld, 64)) return RLLOSS_ECUDA;
    if (!tmap_bf16_box(&hp.tmB48[1], sp.xs, p.H + (p.bias ? 1 : 0), pu_rows, p.xs_ld, 48, 64, CU_TENSOR_MAP_SWIZZLE_128B))
      return RLLOSS_ECUDA;
    if (!tmap_f32_out(&hp.tmO[1], dW, p.H, p.V)) return RLLOSS_ECUDA;
    HProblem& px = hp.pr[0];
    px.kb_per_seg = int(cdiv(p.V, 64));
    px.Mt = p.pu_tiles;
    px.Ht = int(cdiv(p.H, 448));
    px.Hout = p.H;
    px.order = 0;
    px.a_mn = 0;
    px.ksplit = px.kb_per_seg >= 2 ? 2 : 1;   // two halves: two addends onto the zeroed dX
    px.reduce = 1;
    HProblem& pw = hp.pr[1];
    pw.kb_per_seg = int(cdiv(pu_rows, 64));
    pw.Mt = int(cdiv(p.V, 256));
    pw.Ht = int(cdiv(p.H, 448));
    pw.Hout = p.H;
    pw.order = 1;
    pw.a_mn = 1;
    pw.reduce = add_dw ? 1 : 0;
    pw.ksplit = 1;
    if (p.bias) {   // db = sum over rows of k2 pu (+ the target entries): X~'s column H
      pw.xcol = p.H;
      pw.xrows = p.V;
      pw.xcol_out = db;
      pw.wide = (p.H % 448 == 0) ? 1 : 0;
    }
    hp.nprob = 2;
    hp.rows_total = sp.positions;   // 0: e.g. a clipped GSPO sequence, nothing to add
    hp.n0 = 0;
    hp.nc_max = pu_rows;
    hp.status = status;
    hp.limit_ns = kWaitLimitNs;
    hp.dx_idx = sp.idx;
    hp.dx_out = dX;
    hp.dx_nrows = p.N;
    hp.dx_ld = p.H;
    hp.dx_vec = dx_vec ? 1 : 0;
    hp.dx_scale = sp.k2;
    hp.dx_err = err;
    hp.dx_tgt = sp.tgt;
    hp.dx_w = static_cast<const __nv_bfloat16*>(hd.Wop);
    hp.dx_wbegin = 0;
    hp.dx_wrows = p.V;
    hp.dx_wld = p.Kx;
    Phase ph(st, 3);
    RL_TRY(launch_gemmH(hp, px.Mt * px.Ht * px.ksplit + pw.Mt * pw.Ht, st));
    ph.launched();
  }
  {
    Phase ph(st, 5);
    if (p.compact) {
      CompactParams cp{};
      cp.N = p.N;
      cp.Kx = p.Kx;
      cp.Ncap = p.Ncap;
      cp.coef = coef;
      cp.lse2 = lse2;
      cp.targets = targets;
      cp.x = static_cast<const __nv_bfloat16*>(hd.Xop);
      cp.blk_cnt = reinterpret_cast<int*>(ws + p.o_blk);
      cp.blk_off = cp.blk_cnt + compact_groups(p.N);
      cp.ticket = reinterpret_cast<unsigned int*>(ws + p.o_status + 8);
      cp.total = rows_total;
      cp.idx = reinterpret_cast<int*>(ws + p.o_cidx);
      cp.coefc = reinterpret_cast<float*>(ws + p.o_coefc);
      cp.lse2c = reinterpret_cast<float*>(ws + p.o_lse2c);
      cp.tgtc = reinterpret_cast<int64_t*>(ws + p.o_tgtc);
      // one chunk: the compaction copies the kept X rows into the chunk's X
      // buffer (every position fits it); several: each chunk gathers its own
      cp.xc = p.nchunks == 1 ? reinterpret_cast<__nv_bfloat16*>(ws + p.o_xc) : nullptr;
      cp.errc = err;
      cp.status = status;
      cp.done = done;
      if (!acc && !p.stored) {   // the gather zeroes dX; the dX/dW launch adds the kept rows into it
        cp.dx_zero = dX;
        cp.H = p.H;
        cp.dx_vec = dx_vec ? 1 : 0;
      }
      RL_TRY(launch_compact(cp, st));
      ph.launched(2);
      Xb = ws + p.o_xc;
      tg_b = cp.tgtc;
      lse2_b = cp.lse2c;
      coef_b = cp.coefc;
      cidx = cp.idx;
      dxc = reinterpret_cast<float*>(ws + p.o_dxc);
      xb_rows = rup(p.Nc, 256);
    } else {
      RL_TRY(launch_set_total(rows_total, p.N, st));
      ph.launched();
      if (err) RL_TRY(cudaMemsetAsync(err, 0, size_t(p.N) * 4, st));
    }
  }
  CUtensorMap tm_xb;
  if (!tmap_bf16(&tm_xb, Xb, p.Kx, xb_rows, p.Kx, 128)) return RLLOSS_ECUDA;
  for (int ch = 0; ch < p.nchunks; ++ch) {
    const int n0 = ch * p.Nc;
    const int nc = std::min(p.Nc, p.N - n0);   // upper bound; the kernels clamp to the kept rows
    const int Rc = int(cdiv(nc, p.rows_tile));

    if (p.compact && p.nchunks > 1) {   // this chunk's kept X rows, zeros after them
      Phase ph(st, 2);
      RL_TRY(launch_gather_chunk_rows(static_cast<const __nv_bfloat16*>(hd.Xop), p.Kx, cidx, rows_total, n0, nc,
                                      int(xb_rows), static_cast<__nv_bfloat16*>(const_cast<void*>(Xb)), st));
      ph.launched();
    }
    DlParams dp{};
    dp.tmA = tm_xb;
    dp.a_row0 = p.compact ? 0 : n0;
    dp.tmB = hd.fp.tmB;
    dp.nseg = hd.fp.nseg;
    dp.kb_per_seg = p.kb_dl;
    std::memcpy(dp.seg_a, hd.seg_a, sizeof(hd.seg_a));
    std::memcpy(dp.seg_b, hd.seg_b, sizeof(hd.seg_b));
    dp.n0 = n0;
    dp.Nc = nc;
    dp.Rc = Rc;
    dp.rows_total = rows_total;
    dp.V = p.V;
    dp.Vp = p.Vp;
    dp.Vt = p.Vt;
    dp.scale2 = hd.fp.scale2;
    dp.bias2 = hd.bias2;
    dp.targets = tg_b;
    dp.v_begin = v_begin;
    dp.lse2 = lse2_b;
    dp.coef = coef_b;
    dp.dl = dl;
    dp.ld = p.ld_dl;
    // bf16 G leaves in 64 x 32 boxes (128-byte swizzle); fp32 mode's hi and lo
    // terms in 32 x 32 boxes (64-byte swizzle)
    if (!(p.fp32 ? tmap_bf16_box(&dp.tmG, dl, 2ll * p.Vp, nc, p.ld_dl, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B)
                 : tmap_bf16_box(&dp.tmG, dl, p.V, nc, p.ld_dl, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B)))
      return RLLOSS_ECUDA;
    dp.lo_off = lo_off;
    dp.dbp = p.bias ? reinterpret_cast<float*>(ws + p.o_dbpart) : nullptr;
    dp.err = err;
    dp.status = status;
    dp.limit_ns = kWaitLimitNs;
    {
      Phase ph(st, 2);
      RL_TRY(launch_dl(dp, Rc * p.Vt, p.pair, p.kbx, st));
      ph.launched();
    }

    // One grouped launch: problem 0 = dX rows of this chunk,
    //   dX[n][h] = sum_v G[n][v] W[v][h];  problem 1 = dW (+)= over this chunk,
    //   dW[v][h] = sum_n G[n][v] X[n][h].
    {
      HParams hp{};
      set_bwd_segments(hp, p);
      float* dx_out = p.compact ? dxc : dX + size_t(n0) * p.H;
      const long long g_inner = p.fp32 ? 2ll * p.Vp : p.V;
      if (!tmap_bf16(&hp.tmA[0], dl, g_inner, nc, p.ld_dl, 128)) return RLLOSS_ECUDA;
      if (!tmap_bf16(&hp.tmB[0], hd.Wop, p.Kx, p.V, p.Kx, 64)) return RLLOSS_ECUDA;
      if (!tmap_bf16_box(&hp.tmB48[0], hd.Wop, p.Kx, p.V, p.Kx, 48, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return RLLOSS_ECUDA;
      if (!tmap_f32_out(&hp.tmO[0], dx_out, p.H, nc)) return RLLOSS_ECUDA;
      if (!tmap_bf16(&hp.tmA[1], dl, g_inner, nc, p.ld_dl, 64)) return RLLOSS_ECUDA;
      if (!tmap_bf16(&hp.tmB[1], Xb, p.Kx, xb_rows, p.Kx, 64)) return RLLOSS_ECUDA;
      if (!tmap_bf16_box(&hp.tmB48[1], Xb, p.Kx, xb_rows, p.Kx, 48, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return RLLOSS_ECUDA;
      if (!tmap_f32_out(&hp.tmO[1], dW, p.H, p.V)) return RLLOSS_ECUDA;
      HProblem& px = hp.pr[0];
      px.kb_per_seg = int(cdiv(p.V, 64));
      px.a_outer0 = 0;
      px.b_outer0 = 0;
      px.Mt = int(cdiv(nc, 256));
      px.Ht = int(cdiv(p.H, 448));
      px.Hout = p.H;
      px.order = 0;
      px.a_mn = 0;
      // Two k halves reduce-added onto a zeroed buffer (two addends: the same
      // sum in either order); accumulating straight into dX takes one
      // unsplit reduce-add instead, since a third addend would make the
      // result depend on the order of the halves.
      const bool dx_in_place_acc = acc && !p.compact;
      px.ksplit = (hp.nseg * px.kb_per_seg >= 2 && !dx_in_place_acc) ? 2 : 1;
      px.reduce = (px.ksplit == 2 || dx_in_place_acc) ? 1 : 0;
      HProblem& pw = hp.pr[1];
      pw.kb_per_seg = int(cdiv(nc, 64));
      pw.a_outer0 = 0;
      pw.b_outer0 = p.compact ? 0 : n0;
      pw.Mt = int(cdiv(p.V, 256));
      pw.Ht = int(cdiv(p.H, 448));
      pw.Hout = p.H;
      pw.order = 1;
      pw.a_mn = 1;
      pw.reduce = (ch > 0 || acc || p.stored) ? 1 : 0;
      pw.ksplit = 1;
      hp.nprob = 2;
      hp.rows_total = rows_total;
      hp.n0 = n0;
      hp.nc_max = nc;
      hp.status = status;
      hp.limit_ns = kWaitLimitNs;
      if (err) {
        hp.dx_err = err;
        hp.dx_tgt = tg_b;
        hp.dx_w = static_cast<const __nv_bfloat16*>(hd.Wop);
        hp.dx_wbegin = v_begin;
        hp.dx_wrows = p.V;
        hp.dx_wld = p.Kx;
      }
      if (dx_direct) {
        hp.dx_idx = cidx;
        hp.dx_out = dX;
        hp.dx_nrows = p.N;
        hp.dx_ld = p.H;
        hp.dx_vec = dx_vec ? 1 : 0;
      }
      Phase ph(st, 3);
      if (px.reduce && !dx_in_place_acc && !dx_direct)
        RL_TRY(cudaMemsetAsync(dx_out, 0, size_t(nc) * p.H * 4, st));
      RL_TRY(launch_gemmH(hp, px.Mt * px.Ht * px.ksplit + pw.Mt * pw.Ht, st));
      ph.launched();
      if (p.compact && !dx_direct) {
        RL_TRY(launch_scatter_rows(dxc, cidx, rows_total, n0, nc, p.H, dX, acc, st));
        ph.launched();
      }
    }
    if (p.bias) {
      Phase ph(st, 5);
      RL_TRY(launch_db_reduce(reinterpret_cast<float*>(ws + p.o_dbpart), rows_total, n0, nc, p.V, db,
                              ch > 0 || acc || p.stored, st));
      ph.launched();
    }
  }
  return RLLOSS_OK;
}

}  // namespace

extern "C" {

size_t rlloss_workspace_bytes(const rlloss_cfg* cfg) {
  if (validate_full(cfg) != RLLOSS_OK) return 0;
  return make_plan(cfg, kFull).total;
}

size_t rlloss_loss_workspace_bytes(const rlloss_cfg* cfg) {
  if (validate_common(cfg) != RLLOSS_OK) return 0;
  return make_plan(cfg, kLossOnly).total;
}

const char* rlloss_status_str(int code) {
  switch (code) {
    case RLLOSS_OK: return "ok";
    case RLLOSS_EINVAL: return "invalid argument";
    case RLLOSS_EUNSUPPORTED: return "unsupported configuration";
    case RLLOSS_EWORKSPACE: return "workspace too small or misaligned";
    case RLLOSS_ECUDA: return "CUDA error";
    case RLLOSS_DEV_ETIMEOUT: return "device: bounded wait ran out";
    case RLLOSS_DEV_ENONFINITE: return "device: non-finite loss";
    case RLLOSS_DEV_EBADTARGET: return "device: target id out of range";
    case RLLOSS_DEV_EEMPTYSEQ: return "device: sequence without active tokens";
    default: return "unknown status";
  }
}

int rlloss_phase_timing(int enable) {
  std::lock_guard<std::mutex> g(g_timer.mu);
  for (PhaseRec& r : g_timer.recs) {
    g_timer.pool.push_back(r.a);
    g_timer.pool.push_back(r.b);
  }
  g_timer.recs.clear();
  g_timer.on = enable != 0;
  return RLLOSS_OK;
}

int rlloss_phase_times(float* ms, int32_t* launches, int nphase) {
  if (!ms || nphase < 1 || nphase > RLLOSS_NPHASES) return RLLOSS_EINVAL;
  std::lock_guard<std::mutex> g(g_timer.mu);
  for (int i = 0; i < nphase; ++i) {
    ms[i] = 0.f;
    if (launches) launches[i] = 0;
  }
  int rc = RLLOSS_OK;
  for (PhaseRec& r : g_timer.recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
      rc = RLLOSS_ECUDA;
    if (r.phase >= 0 && r.phase < nphase) {
      ms[r.phase] += t;
      if (launches) launches[r.phase] += r.launches;
    }
    g_timer.pool.push_back(r.a);
    g_timer.pool.push_back(r.b);
  }
  g_timer.recs.clear();
  return rc;
}

uint64_t rlloss_kernel_launches(void) { return g_launches.load(); }

int rlloss_get_device_status(const void* workspace, int32_t* status) {
  if (!workspace || !status) return RLLOSS_EINVAL;
  return cuda_rc(cudaMemcpy(status, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost));
}

int rlloss_get_forward_tiles(const void* workspace, int32_t* tiles) {
  if (!workspace || !tiles) return RLLOSS_EINVAL;
  return cuda_rc(cudaMemcpy(tiles, static_cast<const char*>(workspace) + kFwdTilesOffset, sizeof(int32_t),
                            cudaMemcpyDeviceToHost));
}

int rlloss_get_backward_rows(const void* workspace, int32_t* rows) {
  if (!workspace || !rows) return RLLOSS_EINVAL;
  return cuda_rc(cudaMemcpy(rows, static_cast<const char*>(workspace) + kBackwardRowsOffset, sizeof(int32_t),
                            cudaMemcpyDeviceToHost));
}

int rlloss_get_stored_rows(const void* workspace, int32_t* rows) {
  if (!workspace || !rows) return RLLOSS_EINVAL;
  return cuda_rc(cudaMemcpy(rows, static_cast<const char*>(workspace) + kStoredRowsOffset, sizeof(int32_t),
                            cudaMemcpyDeviceToHost));
}

int rlloss_get_stored_positions(const void* workspace, int32_t* rows) {
  if (!workspace || !rows) return RLLOSS_EINVAL;
  return cuda_rc(cudaMemcpy(rows, static_cast<const char*>(workspace) + kStoredPositionsOffset, sizeof(int32_t),
                            cudaMemcpyDeviceToHost));
}

int rlloss_selftest_bounded_wait(void* workspace, uint64_t limit_ns, void* stream) {
  if (!workspace || !aligned(workspace, 256)) return RLLOSS_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  RL_TRY(cudaMemsetAsync(workspace, 0, 256, st));
  RL_TRY(launch_selftest_wait(static_cast<int*>(workspace), limit_ns, st));
  g_launches += 1;
  return RLLOSS_OK;
}

size_t rlloss_forward_workspace_bytes(const rlloss_cfg* cfg) {
  if (validate_head(cfg) != RLLOSS_OK) return 0;
  return make_plan(cfg, kForwardOnly).total;
}

int rlloss_forward(const rlloss_cfg* cfg, const void* X, const void* W, const void* b, const int64_t* targets,
                   float* out_logp, float* out_entropy, float* out_lse, void* workspace, size_t workspace_bytes,
                   void* stream) {
  int e = validate_head(cfg);
  if (e) return e;
  if (cfg->dtype == RLLOSS_FP8_E4M3) return RLLOSS_EINVAL;   // needs the scales: rlloss_forward_e4m3
  if (!X || !W || !targets || !workspace) return RLLOSS_EINVAL;
  if (cfg->has_bias && !b) return RLLOSS_EINVAL;
  if (!aligned(X, 16) || !aligned(W, 16)) return RLLOSS_EINVAL;
  const Plan p = make_plan(cfg, kForwardOnly);
  if (!aligned(workspace, 256) || workspace_bytes < p.total) return RLLOSS_EWORKSPACE;
  if (!encode_fn()) return RLLOSS_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  RL_TRY(cudaMemsetAsync(ws + p.o_status, 0, 256, st));
  Head hd;
  return run_head(cfg, p, X, W, b, targets, out_logp, out_entropy, out_lse, ws, st, hd);
}

int rlloss_forward_e4m3(const rlloss_cfg* cfg, const void* X8, const float* x_scale, const void* W8,
                        const float* w_scale, const float* b, const int64_t* targets, float* out_logp,
                        float* out_entropy, float* out_lse, void* workspace, size_t workspace_bytes,
                        void* stream) {
  int e = validate_head(cfg);
  if (e) return e;
  if (cfg->dtype != RLLOSS_FP8_E4M3) return RLLOSS_EINVAL;
  if (!X8 || !W8 || !x_scale || !w_scale || !targets || !workspace) return RLLOSS_EINVAL;
  if (cfg->has_bias && !b) return RLLOSS_EINVAL;
  if (!aligned(X8, 16) || !aligned(W8, 16)) return RLLOSS_EINVAL;
  const Plan p = make_plan(cfg, kForwardOnly);
  if (!aligned(workspace, 256) || workspace_bytes < p.total) return RLLOSS_EWORKSPACE;
  if (!encode_fn()) return RLLOSS_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  RL_TRY(cudaMemsetAsync(ws + p.o_status, 0, 256, st));
  Head hd;
  hd.x_scale = x_scale;
  hd.w_scale = w_scale;
  return run_head(cfg, p, X8, W8, b, targets, out_logp, out_entropy, out_lse, ws, st, hd);
}

int rlloss_loss_from_logp(const rlloss_cfg* cfg, const float* logp, const float* entropy, const float* old_logp,
                          const float* ref_logp, const float* adv, const uint8_t* mask, float* out_loss,
                          float* out_metrics, float* out_dlogp, uint8_t* out_entropy_mask, void* workspace,
                          size_t workspace_bytes, void* stream) {
  int e = validate_common(cfg);
  if (e) return e;
  if (!logp || !old_logp || !adv || !mask || !out_loss || !out_metrics || !workspace) return RLLOSS_EINVAL;
  if (cfg->beta != 0.f && !ref_logp) return RLLOSS_EINVAL;
  const Plan p = make_plan(cfg, kLossOnly);
  if (p.ent && !entropy) return RLLOSS_EINVAL;
  if (!aligned(workspace, 256) || workspace_bytes < p.total) return RLLOSS_EWORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  RL_TRY(cudaMemsetAsync(ws + p.o_status, 0, p.o_tickets + size_t(p.B) * 4 - p.o_status, st));
  uint8_t* emask = reinterpret_cast<uint8_t*>(ws + p.o_emask);
  if (p.ent) {
    RL_TRY(launch_entropy_mask(entropy, mask, p.N, double(cfg->top_entropy_quantile), ws + p.o_k3, emask, st));
    g_launches += 9;
  }
  LossParams lp = loss_params(cfg, p, ws);
  lp.logp = logp;
  lp.logp_is_f64 = 0;
  lp.old_logp = old_logp;
  lp.ref_logp = ref_logp;
  lp.adv = adv;
  lp.mask = mask;
  lp.emask = p.ent ? emask : nullptr;
  lp.dlogp = out_dlogp;
  lp.out_loss = out_loss;
  lp.out_metrics = out_metrics;
  RL_TRY(launch_loss(lp, st));
  g_launches += out_dlogp ? 2 : 1;
  if (out_entropy_mask)
    RL_TRY(cudaMemcpyAsync(out_entropy_mask, p.ent ? emask : mask, size_t(p.N), cudaMemcpyDeviceToDevice, st));
  return RLLOSS_OK;
}

// ---- Batch split over ranks by whole sequences (see rlloss.h).

size_t rlloss_select_state_bytes(void) { return size_t(kSelectStateBytes); }

int rlloss_entropy_hist(const float* entropy, const uint8_t* mask, int64_t N, int32_t pass, const void* select_state,
                        uint32_t* counts, void* stream) {
  if (N < 0 || pass < 0 || pass >= kSelectPasses || !counts) return RLLOSS_EINVAL;
  if (N > 0 && (!entropy || !mask)) return RLLOSS_EINVAL;
  if (pass > 0 && !select_state) return RLLOSS_EINVAL;
  if (select_state && !aligned(select_state, 16)) return RLLOSS_EINVAL;
  RL_TRY(launch_entropy_hist(entropy, mask, N, pass, select_state, counts, static_cast<cudaStream_t>(stream)));
  g_launches += N > 0 ? 1 : 0;
  return RLLOSS_OK;
}

int rlloss_entropy_select(int32_t pass, const uint32_t* counts, float q, void* select_state, void* stream) {
  if (pass < 0 || pass >= kSelectPasses || !counts || !select_state || !aligned(select_state, 16)) return RLLOSS_EINVAL;
  if (!(q >= 0.f && q <= 1.f)) return RLLOSS_EINVAL;
  RL_TRY(launch_entropy_select(pass, counts, double(q), select_state, static_cast<cudaStream_t>(stream)));
  g_launches += 1;
  return RLLOSS_OK;
}

int rlloss_select_threshold(const void* select_state, double* threshold) {
  if (!select_state || !threshold) return RLLOSS_EINVAL;
  return cuda_rc(cudaMemcpy(threshold, select_state, sizeof(double), cudaMemcpyDeviceToHost));
}

int rlloss_loss_from_logp_dp(const rlloss_cfg* cfg, int32_t B_global, const void* select_state, const float* logp,
                             const float* entropy, const float* old_logp, const float* ref_logp, const float* adv,
                             const uint8_t* mask, double* out_sums, float* out_dlogp, uint8_t* out_entropy_mask,
                             void* workspace, size_t workspace_bytes, void* stream) {
  int e = validate_common(cfg);
  if (e) return e;
  if (B_global < cfg->B) return RLLOSS_EINVAL;
  if (!logp || !old_logp || !adv || !mask || !out_sums || !workspace) return RLLOSS_EINVAL;
  if (cfg->beta != 0.f && !ref_logp) return RLLOSS_EINVAL;
  const Plan p = make_plan(cfg, kLossOnly);
  if (p.ent && (!entropy || !select_state || !aligned(select_state, 16))) return RLLOSS_EINVAL;
  if (!aligned(workspace, 256) || workspace_bytes < p.total) return RLLOSS_EWORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  RL_TRY(cudaMemsetAsync(ws + p.o_status, 0, p.o_tickets + size_t(p.B) * 4 - p.o_status, st));
  uint8_t* emask = reinterpret_cast<uint8_t*>(ws + p.o_emask);
  if (p.ent) {   // the batch-global threshold comes from the ranks' joint selection
    RL_TRY(launch_entropy_apply(entropy, mask, p.N, select_state, emask, st));
    g_launches += 1;
  }
  LossParams lp = loss_params(cfg, p, ws);
  lp.k3 = p.ent ? static_cast<const double*>(select_state) : nullptr;
  lp.Bg = double(B_global);
  lp.logp = logp;
  lp.logp_is_f64 = 0;
  lp.old_logp = old_logp;
  lp.ref_logp = ref_logp;
  lp.adv = adv;
  lp.mask = mask;
  lp.emask = p.ent ? emask : nullptr;
  lp.dlogp = out_dlogp;
  lp.out_loss = nullptr;
  lp.out_metrics = nullptr;
  lp.out_sums = out_sums;
  RL_TRY(launch_loss(lp, st));
  g_launches += out_dlogp ? 2 : 1;
  if (out_entropy_mask)
    RL_TRY(cudaMemcpyAsync(out_entropy_mask, p.ent ? emask : mask, size_t(p.N), cudaMemcpyDeviceToDevice, st));
  return RLLOSS_OK;
}

int rlloss_metrics_from_sums(const rlloss_cfg* cfg, int32_t B_global, const double* sums, double threshold,
                             float* out_loss, float* out_metrics) {
  if (!cfg || !sums || !out_loss || !out_metrics || B_global < 1) return RLLOSS_EINVAL;
  if (cfg->loss_type != RLLOSS_GMPO && cfg->loss_type != RLLOSS_GSPO_TOKEN) return RLLOSS_EINVAL;
  const bool gmpo = cfg->loss_type == RLLOSS_GMPO;
  const double Bg = double(B_global);
  const double n_act = sums[1], clip = sums[2], kl = sums[3], kept = sums[4], sx = sums[5], sr = sums[6],
               nh = sums[7];
  const double loss = gmpo ? sums[0] / Bg : sums[0];
  float* m = out_metrics;
  if (gmpo) {
    m[0] = n_act > 0 ? float(clip / n_act) : 0.f;
    m[2] = (cfg->beta != 0.f && n_act > 0) ? float(kl / n_act) : 0.f;
  } else {
    m[0] = float(clip / Bg);
    m[2] = 0.f;
  }
  m[1] = float(clip);
  m[3] = float(n_act);
  m[4] = float(threshold);
  m[5] = float(kept);
  m[6] = nh > 0 ? float(sx / nh) : 0.f;
  m[7] = nh > 0 ? float(sr / nh) : 0.f;
  *out_loss = float(loss);
  return RLLOSS_OK;
}

int rlloss_fwd_bwd(const rlloss_cfg* cfg, const void* X, const void* W, const void* b, const int64_t* targets,
                   const float* old_logp, const float* ref_logp, const float* adv, const uint8_t* mask,
                   float* out_loss, float* out_metrics, float* dX, float* dW, float* db, float* out_logp,
                   float* out_entropy, uint8_t* out_entropy_mask, void* workspace, size_t workspace_bytes,
                   void* stream) {
  int e = validate_full(cfg);
  if (e) return e;
  if (!X || !W || !targets || !old_logp || !adv || !mask || !out_loss || !out_metrics || !dX || !dW || !workspace)
    return RLLOSS_EINVAL;
  if (cfg->has_bias && (!b || !db)) return RLLOSS_EINVAL;
  if (cfg->beta != 0.f && !ref_logp) return RLLOSS_EINVAL;
  if (!aligned(X, 16) || !aligned(W, 16) || !aligned(dX, 16) || !aligned(dW, 16)) return RLLOSS_EINVAL;
  const Plan p = make_plan(cfg, kFull);
  if (!aligned(workspace, 256) || workspace_bytes < p.total) return RLLOSS_EWORKSPACE;
  if (!encode_fn()) return RLLOSS_ECUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  RL_TRY(cudaMemsetAsync(ws + p.o_status, 0, p.o_tickets + size_t(p.B) * 4 - p.o_status, st));

  Head hd;
  // Row tiles whose rows are all masked enter neither the loss nor the
  // gradients; their forward is skipped unless per-token outputs are wanted
  // or advantages are per token (tokens outside the mask then count).
  const bool skip_tiles = !(cfg->flags & (RLLOSS_FLAG_ALL_ROWS | RLLOSS_FLAG_ADV_PER_TOKEN)) && !out_logp &&
                          !out_entropy;
  if (p.seq_group) {
    // ---- groups of whole sequences that each fit the stored-probability buffer
    // (no entropy mask: sequences are coupled only by B and by sums): per group
    // the forward with stores, the loss stage's additive batch sums with the
    // whole batch's B, and the stored backward (dW, db added after the first
    // group); then loss and metrics from the groups' sums.
    double* sums = reinterpret_cast<double*>(ws + p.o_sums);
    int* counters = reinterpret_cast<int*>(ws + p.o_sums + size_t(p.ngroups) * 64);
    int* ctr_dev[4] = {reinterpret_cast<int*>(ws + p.o_status + kFwdTilesOffset),
                       reinterpret_cast<int*>(ws + p.o_status + kStoredRowsOffset),
                       reinterpret_cast<int*>(ws + p.o_status + kBackwardRowsOffset),
                       reinterpret_cast<int*>(ws + p.o_status + kStoredPositionsOffset)};
    RL_TRY(cudaMemsetAsync(counters, 0, 16, st));
    const size_t xrow = size_t(cfg->H) * 2;   // bf16 row bytes
    for (int g = 0; g < p.ngroups; ++g) {
      const int i0 = g * p.seq_group, i1 = std::min(cfg->B, i0 + p.seq_group);
      const long long r0 = (long long)i0 * cfg->T;
      rlloss_cfg cg = *cfg;
      cg.B = i1 - i0;
      Plan pg = p;   // the whole batch's regions, used from their start
      pg.B = cg.B;
      pg.N = cg.B * cg.T;
      pg.R = int(cdiv(pg.N, pg.rows_tile));
      pg.P = choose_segments(pg.R, pg.Vt, pg.fwd_clusters, pg.pcap);
      pg.nchunks = int(cdiv(pg.N, pg.Nc));
      pg.Ncap = int(rup(pg.N, 256));
      // tickets and per-group counters (the status word keeps its bits)
      RL_TRY(cudaMemsetAsync(ws + p.o_status + 4, 0, p.o_tickets + size_t(pg.B) * 4 - p.o_status - 4, st));
      Head hg;
      RL_TRY_RC(run_head(&cg, pg, static_cast<const char*>(X) + size_t(r0) * xrow, W, b, targets + r0,
                         out_logp ? out_logp + r0 : nullptr, out_entropy ? out_entropy + r0 : nullptr, nullptr, ws,
                         st, hg, false, skip_tiles ? mask + r0 : nullptr));
      LossParams lg = loss_params(&cg, pg, ws);
      lg.Bg = double(cfg->B);
      lg.logp = hg.mp.logp64;
      lg.logp_is_f64 = 1;
      lg.old_logp = old_logp + r0;
      lg.ref_logp = ref_logp ? ref_logp + r0 : nullptr;
      lg.adv = adv + i0;
      lg.mask = mask + r0;
      lg.coef = reinterpret_cast<float*>(ws + p.o_coef);
      lg.out_sums = sums + size_t(g) * 8;
      {
        Phase ph(st, 1);
        RL_TRY(launch_merge_loss(hg.mp, lg, st));
        ph.launched(2);
      }
      RL_TRY_RC(run_backward(&cg, pg, hg, targets + r0, 0, hg.mp.lse2, lg.coef, dX + size_t(r0) * cfg->H, dW, db,
                             ws, st, g > 0));
      RL_TRY(launch_counters(ctr_dev, counters, false, st));
      g_launches += 1;
    }
    LossParams lf = loss_params(cfg, p, ws);
    lf.out_loss = out_loss;
    lf.out_metrics = out_metrics;
    {
      Phase ph(st, 1);
      RL_TRY(launch_fold_sums(sums, p.ngroups, lf, st));
      RL_TRY(launch_counters(ctr_dev, counters, true, st));
      ph.launched(2);
    }
    if (out_entropy_mask) RL_TRY(cudaMemcpyAsync(out_entropy_mask, mask, size_t(p.N), cudaMemcpyDeviceToDevice, st));
    return RLLOSS_OK;
  }
  RL_TRY_RC(run_head(cfg, p, X, W, b, targets, out_logp, out_entropy, nullptr, ws, st, hd, !p.fused_loss,
                     skip_tiles ? mask : nullptr));
  const MergeParams& mp = hd.mp;
  LossParams lp{};
  {
  Phase ph_loss(st, 1);
  // ---- entropy mask and loss
  uint8_t* emask = reinterpret_cast<uint8_t*>(ws + p.o_emask);
  if (p.ent) {
    RL_TRY(launch_entropy_mask(mp.ent32, mask, p.N, double(cfg->top_entropy_quantile), ws + p.o_k3, emask, st));
    ph_loss.launched(9);
  }
  lp = loss_params(cfg, p, ws);
  lp.logp = mp.logp64;
  lp.logp_is_f64 = 1;
  lp.old_logp = old_logp;
  lp.ref_logp = ref_logp;
  lp.adv = adv;
  lp.mask = mask;
  lp.emask = p.ent ? emask : nullptr;
  lp.coef = reinterpret_cast<float*>(ws + p.o_coef);
  lp.out_loss = out_loss;
  lp.out_metrics = out_metrics;
  if (p.fused_loss) {
    RL_TRY(launch_merge_loss(mp, lp, st));
    ph_loss.launched(2);
  } else {
    RL_TRY(launch_loss(lp, st));
    ph_loss.launched(2);
  }
  if (out_entropy_mask)
    RL_TRY(cudaMemcpyAsync(out_entropy_mask, p.ent ? emask : mask, size_t(p.N), cudaMemcpyDeviceToDevice, st));
  }

  return run_backward(cfg, p, hd, targets, 0, mp.lse2, lp.coef, dX, dW, db, ws, st);
}

// ---------------------------------------------------------------- vocabulary shards
// The vocabulary-parallel form of the path: each shard of W (a contiguous
// range of vocabulary rows) yields a mergeable per-row softmax state; the
// states of all shards give lse, logp, entropy, loss and dL/dlogp; each shard
// then computes its own dW and db rows and its part of dX (the parts sum to
// dX).  The streamed accumulators are mergeable ("support
// top_entropy_quantile in fused linear GRPO loss", Details: the entropy from
// a second online accumulator beside the log-sum-exp one).

int rlloss_forward_shard(const rlloss_cfg* cfg, const void* X, const void* W, const void* b, const int64_t* targets,
                         int64_t v_begin, float* out_state, void* workspace, size_t workspace_bytes, void* stream) {
  int e = validate_head(cfg);
  if (e) return e;
  if (cfg->dtype == RLLOSS_FP8_E4M3) return RLLOSS_EUNSUPPORTED;
  if (!X || !W || !targets || !out_state || !workspace || v_begin < 0) return RLLOSS_EINVAL;
  if (cfg->has_bias && !b) return RLLOSS_EINVAL;
  if (!aligned(X, 16) || !aligned(W, 16) || !aligned(out_state, 16)) return RLLOSS_EINVAL;
  const Plan p = make_plan(cfg, kForwardOnly);
  if (!aligned(workspace, 256) || workspace_bytes < p.total) return RLLOSS_EWORKSPACE;
  if (!encode_fn()) return RLLOSS_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  RL_TRY(cudaMemsetAsync(ws + p.o_status, 0, 256, st));
  Head hd;
  RL_TRY_RC(run_head(cfg, p, X, W, b, targets, nullptr, nullptr, nullptr, ws, st, hd, false, nullptr, v_begin));
  Phase ph(st, 1);
  RL_TRY(launch_shard_state(hd.mp, reinterpret_cast<float4*>(out_state), st));
  ph.launched();
  return RLLOSS_OK;
}

size_t rlloss_shard_loss_workspace_bytes(const rlloss_cfg* cfg) {
  if (validate_common(cfg) != RLLOSS_OK || cfg->V < 1) return 0;
  return make_plan(cfg, kShardLoss).total;
}

int rlloss_loss_from_shards(const rlloss_cfg* cfg, int32_t nshards, const float* states, const int64_t* targets,
                            const float* old_logp, const float* ref_logp, const float* adv, const uint8_t* mask,
                            float* out_loss, float* out_metrics, float* out_lse, float* out_dlogp, float* out_logp,
                            float* out_entropy, uint8_t* out_entropy_mask, void* workspace, size_t workspace_bytes,
                            void* stream) {
  int e = validate_common(cfg);
  if (e) return e;
  if (cfg->V < 1 || nshards < 1 || nshards > RLLOSS_MAX_SHARDS) return RLLOSS_EINVAL;
  if (!states || !targets || !old_logp || !adv || !mask || !out_loss || !out_metrics || !workspace)
    return RLLOSS_EINVAL;
  if (cfg->beta != 0.f && !ref_logp) return RLLOSS_EINVAL;
  if (!aligned(states, 16)) return RLLOSS_EINVAL;
  const Plan p = make_plan(cfg, kShardLoss);
  if (!aligned(workspace, 256) || workspace_bytes < p.total) return RLLOSS_EWORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws + p.o_status);
  RL_TRY(cudaMemsetAsync(ws + p.o_status, 0, p.o_tickets + size_t(p.B) * 4 - p.o_status, st));
  MergeParams mp{};
  mp.partial = reinterpret_cast<const float4*>(states);
  mp.N = p.N;
  mp.V = cfg->V;
  mp.slots = nshards;
  mp.slot_stride = p.N;
  mp.targets = targets;
  mp.lse2 = reinterpret_cast<float*>(ws + p.o_lse2);
  mp.logp64 = reinterpret_cast<double*>(ws + p.o_logp64);
  mp.ent32 = reinterpret_cast<float*>(ws + p.o_ent);
  mp.out_logp = out_logp;
  mp.out_ent = out_entropy;
  mp.out_lse = out_lse;
  mp.status = status;
  Phase ph(st, 1);
  RL_TRY(launch_merge(mp, st));
  ph.launched();
  uint8_t* emask = reinterpret_cast<uint8_t*>(ws + p.o_emask);
  if (p.ent) {
    RL_TRY(launch_entropy_mask(mp.ent32, mask, p.N, double(cfg->top_entropy_quantile), ws + p.o_k3, emask, st));
    ph.launched(9);
  }
  LossParams lp = loss_params(cfg, p, ws);
  lp.logp = mp.logp64;
  lp.logp_is_f64 = 1;
  lp.old_logp = old_logp;
  lp.ref_logp = ref_logp;
  lp.adv = adv;
  lp.mask = mask;
  lp.emask = p.ent ? emask : nullptr;
  lp.dlogp = out_dlogp;
  lp.out_loss = out_loss;
  lp.out_metrics = out_metrics;
  RL_TRY(launch_loss(lp, st));
  ph.launched(out_dlogp ? 2 : 1);
  if (out_entropy_mask)
    RL_TRY(cudaMemcpyAsync(out_entropy_mask, p.ent ? emask : mask, size_t(p.N), cudaMemcpyDeviceToDevice, st));
  return RLLOSS_OK;
}

size_t rlloss_backward_shard_workspace_bytes(const rlloss_cfg* cfg) {
  if (validate_full(cfg) != RLLOSS_OK) return 0;
  return make_plan(cfg, kBackwardOnly).total;
}

int rlloss_backward_shard(const rlloss_cfg* cfg, const void* X, const void* W, const void* b, const int64_t* targets,
                          int64_t v_begin, const float* lse, const float* dlogp, float* dX, float* dW, float* db,
                          void* workspace, size_t workspace_bytes, void* stream) {
  int e = validate_full(cfg);
  if (e) return e;
  if (!X || !W || !targets || !lse || !dlogp || !dX || !dW || !workspace || v_begin < 0) return RLLOSS_EINVAL;
  if (cfg->has_bias && (!b || !db)) return RLLOSS_EINVAL;
  if (!aligned(X, 16) || !aligned(W, 16) || !aligned(dX, 16) || !aligned(dW, 16)) return RLLOSS_EINVAL;
  const Plan p = make_plan(cfg, kBackwardOnly);
  if (!aligned(workspace, 256) || workspace_bytes < p.total) return RLLOSS_EWORKSPACE;
  if (!encode_fn()) return RLLOSS_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  RL_TRY(cudaMemsetAsync(ws + p.o_status, 0, 256, st));
  Head hd;
  RL_TRY_RC(prepare_head(cfg, p, X, W, b, ws, st, hd));
  float* lse2 = reinterpret_cast<float*>(ws + p.o_lse2);
  float* coef = reinterpret_cast<float*>(ws + p.o_coef);
  {
    Phase ph(st, 5);
    RL_TRY(launch_backward_rows_in(lse, dlogp, p.N, 1.0 / double(cfg->temperature), lse2, coef, st));
    ph.launched();
  }
  return run_backward(cfg, p, hd, targets, v_begin, lse2, coef, dX, dW, db, ws, st);
}

}  // extern "C"
