// Loss-stage kernels.
//
//  K3 entropy quantile: exact order statistics of the active tokens'
//     entropies by a 4-pass, 8-bit radix select on order-preserving uint32
//     keys, then linear interpolation at position (1-q)(n_act-1) and the mask
//     H >= threshold — "support top_entropy_quantile in fused linear GRPO
//     loss", Details (batch-global quantile of active entropies at 1 - q).
//     The passes are also exported one by one (histogram, then select from
//     counts summed over ranks) for batches split over ranks.
//  K2 per-sequence reduction: blocks over slices of each sequence form fp64
//     partial sums; the last slice of a sequence folds them into its record,
//     the last sequence folds the records into the loss and metrics (or into
//     eight batch sums that add over ranks), both in a fixed order; then the
//     per-token gradient coefficient c_n = dL/dlogp_n.  GMPO: "Add GMPO to
//     fused linear GRPO loss", Summary and Details.  GSPO-token: Tinker
//     "GSPO", ratio and objective formulas.
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"
#include "merge_row.cuh"
#include "status.h"

namespace rl {

struct K3State {
  double thr;
  double frac;
  unsigned long long n_act;
  unsigned long long k[2];
  unsigned int prefix[2];
};
constexpr int kK3HistOff = 256;   // 4 passes x 2 x 256 uint32 follow the state

__device__ __forceinline__ uint32_t f2key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

__global__ void k3_hist_kernel(const float* __restrict__ H, const uint8_t* __restrict__ m, long long N, int pass,
                               const K3State* st, uint32_t* hist) {
  __shared__ uint32_t sh[512];
  for (int i = threadIdx.x; i < 512; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  const int shift = 24 - 8 * pass;
  uint32_t p0 = 0, p1 = 0;
  if (pass > 0) {
    if (st->n_act == 0) return;
    p0 = st->prefix[0];
    p1 = st->prefix[1];
  }
  // The two order statistics usually share their prefix (adjacent ranks):
  // then one count serves both halves of the histogram.
  const bool two = pass > 0 && p0 != p1;
  // Passes 0 and 1 (sign, exponent, top mantissa bits) put most tokens of a
  // narrow distribution in a few bins: the lanes of a warp that share a bin
  // add once.  The low key bytes of passes 2 and 3 are spread over the bins,
  // where plain shared-memory atomics are cheaper than the grouping.
  const bool group = pass < 2;
  const int lane = threadIdx.x & 31;
  auto add = [&](int b) {
    if (group) {
      const unsigned g = __match_any_sync(0xffffffffu, b);
      if (b >= 0 && lane == __ffs(g) - 1) atomicAdd(&sh[b], unsigned(__popc(g)));
    } else if (b >= 0) {
      atomicAdd(&sh[b], 1u);
    }
  };
  auto count = [&](bool act, float h) {
    int b0 = -1, b1 = -1;
    if (act) {
      const uint32_t key = f2key(h);
      const int d = int((key >> shift) & 255u);
      if (pass == 0) {
        b0 = d;
      } else {
        const uint32_t hp = key >> (shift + 8);
        if (hp == p0) b0 = d;
        if (two && hp == p1) b1 = 256 + d;
      }
    }
    add(b0);
    if (two) add(b1);
  };
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (((reinterpret_cast<uintptr_t>(H) & 15u) | (reinterpret_cast<uintptr_t>(m) & 3u)) == 0) {
    // four tokens a thread: one 4-byte mask word and, when any is active, one
    // 16-byte entropy load (the last, partial group element by element)
    const long long NG = (N + 3) / 4;
    for (long long g = tid; g - lane < NG; g += stride) {
      uint32_t mw = 0;
      float hv[4] = {0.f, 0.f, 0.f, 0.f};
      if (g < NG) {
        if (4 * g + 3 < N) {
          mw = __ldg(reinterpret_cast<const uint32_t*>(m) + g);
          if (mw) {
            const float4 h4 = __ldg(reinterpret_cast<const float4*>(H) + g);
            hv[0] = h4.x; hv[1] = h4.y; hv[2] = h4.z; hv[3] = h4.w;
          }
        } else {
          for (int k = 0; k < 4; ++k)
            if (4 * g + k < N && m[4 * g + k]) {
              mw |= 1u << (8 * k);
              hv[k] = H[4 * g + k];
            }
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) count(((mw >> (8 * k)) & 255u) != 0u, hv[k]);
    }
  } else {
    for (long long n = tid; n - lane < N; n += stride) {
      const bool act = n < N && m[n];
      count(act, act ? H[n] : 0.f);
    }
  }
  __syncthreads();
  if (pass > 0 && !two) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x)
      if (sh[i]) {
        atomicAdd(&hist[i], sh[i]);
        atomicAdd(&hist[256 + i], sh[i]);
      }
  } else {
    for (int i = threadIdx.x; i < 512; i += blockDim.x)
      if (sh[i]) atomicAdd(&hist[i], sh[i]);
  }
}

__global__ void k3_select_kernel(int pass, K3State* st, const uint32_t* hist, double q) {
  if (threadIdx.x != 0) return;
  if (pass == 0) {
    unsigned long long n = 0;
    for (int b = 0; b < 256; ++b) n += hist[b];
    st->n_act = n;
    st->prefix[0] = st->prefix[1] = 0;
    if (n == 0) {
      st->thr = __longlong_as_double(0x7ff8000000000000ll);
      st->frac = 0.0;
      return;
    }
    const double pos = (1.0 - q) * double(n - 1);
    unsigned long long lo = (unsigned long long)floor(pos);
    if (lo > n - 1) lo = n - 1;
    const unsigned long long hi = lo + 1 < n ? lo + 1 : n - 1;
    st->frac = pos - double(lo);
    st->k[0] = lo;
    st->k[1] = hi;
  }
  if (st->n_act == 0) return;
  for (int j = 0; j < 2; ++j) {
    const uint32_t* h = hist + (pass == 0 ? 0 : 256 * j);
    const unsigned long long k = st->k[j];
    unsigned long long cum = 0;
    int b = 0;
    for (; b < 255; ++b) {
      if (cum + h[b] > k) break;
      cum += h[b];
    }
    st->k[j] = k - cum;
    st->prefix[j] = (st->prefix[j] << 8) | uint32_t(b);
  }
  if (pass == 3) {
    const double vlo = double(key2f(st->prefix[0]));
    const double vhi = double(key2f(st->prefix[1]));
    st->thr = vlo + st->frac * (vhi - vlo);
  }
}

__global__ void k3_mask_kernel(const float* __restrict__ H, const uint8_t* __restrict__ m, long long N,
                               const K3State* st, uint8_t* e) {
  // For a float h, h >= thr exactly when h >= the smallest float >= thr (a
  // NaN threshold keeps nothing either way), so the test runs in fp32.
  const float thr = __double2float_ru(st->thr);
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (((reinterpret_cast<uintptr_t>(H) & 15u) | (reinterpret_cast<uintptr_t>(m) & 3u) |
       (reinterpret_cast<uintptr_t>(e) & 3u)) == 0) {
    const long long NG = N / 4;   // whole groups of four tokens; the rest below
    for (long long g = tid; g < NG; g += stride) {
      const uint32_t mw = __ldg(reinterpret_cast<const uint32_t*>(m) + g);
      uint32_t ew = 0;
      if (mw) {
        const float4 h4 = __ldg(reinterpret_cast<const float4*>(H) + g);
        ew = ((mw & 0xffu) && h4.x >= thr ? 1u : 0u) | ((mw & 0xff00u) && h4.y >= thr ? 1u << 8 : 0u) |
             ((mw & 0xff0000u) && h4.z >= thr ? 1u << 16 : 0u) | ((mw & 0xff000000u) && h4.w >= thr ? 1u << 24 : 0u);
      }
      reinterpret_cast<uint32_t*>(e)[g] = ew;
    }
    for (long long n = 4 * NG + tid; n < N; n += stride) e[n] = (m[n] && H[n] >= thr) ? 1 : 0;
  } else {
    for (long long n = tid; n < N; n += stride) e[n] = (m[n] && H[n] >= thr) ? 1 : 0;
  }
}

cudaError_t launch_entropy_mask(const float* ent, const uint8_t* mask, long long N, double q, void* k3_ws,
                                uint8_t* emask, cudaStream_t st) {
  cudaError_t err = cudaMemsetAsync(k3_ws, 0, kK3Bytes, st);
  if (err != cudaSuccess) return err;
  K3State* s = static_cast<K3State*>(k3_ws);
  uint32_t* hist = reinterpret_cast<uint32_t*>(static_cast<char*>(k3_ws) + kK3HistOff);
  const int threads = 256;
  long long blocks = (N + threads * 8 - 1) / (threads * 8);
  if (blocks < 1) blocks = 1;
  if (blocks > 2048) blocks = 2048;
  for (int pass = 0; pass < 4; ++pass) {
    k3_hist_kernel<<<int(blocks), threads, 0, st>>>(ent, mask, N, pass, s, hist + 512 * pass);
    k3_select_kernel<<<1, 32, 0, st>>>(pass, s, hist + 512 * pass, q);
  }
  k3_mask_kernel<<<int(blocks), threads, 0, st>>>(ent, mask, N, s, emask);
  return cudaGetLastError();
}

static_assert(sizeof(K3State) <= kSelectStateBytes, "select state");
static_assert(kK3HistOff == kSelectStateBytes, "state then histograms");

static int k3_blocks(long long N) {
  long long blocks = (N + 256 * 8 - 1) / (256 * 8);
  if (blocks < 1) blocks = 1;
  if (blocks > 2048) blocks = 2048;
  return int(blocks);
}

cudaError_t launch_entropy_hist(const float* ent, const uint8_t* mask, long long N, int pass, const void* state,
                                uint32_t* counts, cudaStream_t st) {
  cudaError_t err = cudaMemsetAsync(counts, 0, kSelectCounts * sizeof(uint32_t), st);
  if (err != cudaSuccess) return err;
  if (N > 0)
    k3_hist_kernel<<<k3_blocks(N), 256, 0, st>>>(ent, mask, N, pass, static_cast<const K3State*>(state), counts);
  return cudaGetLastError();
}

cudaError_t launch_entropy_select(int pass, const uint32_t* counts, double q, void* state, cudaStream_t st) {
  k3_select_kernel<<<1, 32, 0, st>>>(pass, static_cast<K3State*>(state), counts, q);
  return cudaGetLastError();
}

cudaError_t launch_entropy_apply(const float* ent, const uint8_t* mask, long long N, const void* state,
                                 uint8_t* emask, cudaStream_t st) {
  if (N > 0)
    k3_mask_kernel<<<k3_blocks(N), 256, 0, st>>>(ent, mask, N, static_cast<const K3State*>(state), emask);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------- K2
constexpr int kLossThreads = 256;
constexpr int kFusedRows = 256 / kMergeLanes;   // rows per block of the fused merge + loss kernel
constexpr int kRec = 10;           // doubles per sequence record

template <int K>
__device__ __forceinline__ void warp_sum_k(double (&v)[K]) {
#pragma unroll
  for (int k = 0; k < K; ++k)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_down_sync(0xffffffffu, v[k], o);
}

// K sums over the block, in a fixed order; the result is valid in thread 0.
template <int K>
__device__ __forceinline__ void block_sum_k(double (&v)[K], double (*sh)[32]) {
  warp_sum_k(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0)
#pragma unroll
    for (int k = 0; k < K; ++k) sh[k][w] = v[k];
  __syncthreads();
  if (w == 0) {
    const int nw = int(blockDim.x >> 5);
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] = l < nw ? sh[k][l] : 0.0;
    warp_sum_k(v);
  }
}

// lr = lp - old of two floats, held exactly as hi + lo (two-sum), and the
// clip test of GMPO decided on it exactly: lr > e holds iff hi > e, or
// hi == e and lo > 0 (|lo| is at most half an ulp of hi), for a float bound e.
struct ExactDiff {
  float hi, lo;
};
__device__ __forceinline__ ExactDiff exact_diff(float lp, float old) {
  const float hi = lp - old;
  const float bb = hi - lp;
  return {hi, (lp - (hi - bb)) + (-old - bb)};
}
__device__ __forceinline__ bool gmpo_clipped(const ExactDiff& d, double A, float eh, float el) {
  if (A > 0.0) return d.hi > eh || (d.hi == eh && d.lo > 0.f);
  if (A < 0.0) return d.hi < el || (d.hi == el && d.lo < 0.f);
  return false;
}

__device__ __forceinline__ double logp_at(const LossParams& p, long long n) {
  return p.logp_is_f64 ? __ldcg(static_cast<const double*>(p.logp) + n)
                       : double(static_cast<const float*>(p.logp)[n]);
}
__device__ __forceinline__ double seq_adv(const LossParams& p, int i) {
  return p.adv_per_token ? 0.0 : double(p.adv[i]);
}

// Token n's share of its sequence's sums (lp = its logp):
//   [0] active tokens, [1] sum of (clipped) log ratios, [4] clip count;
//   GMPO: [2] tokens kept by the entropy mask, [3] sum of K3 KL;
//   GSPO: [2] / [3] sums of the positive / negative token advantages.
__device__ __forceinline__ void token_terms(const LossParams& p, long long n, double lp, double A, bool gmpo,
                                            double (&a)[5]) {
  const bool m = p.mask[n] != 0;
  if (gmpo) {
    if (!m) return;
    const double lr = lp - double(p.old_logp[n]);
    a[0] += 1.0;
    const bool clip = (A > 0.0 && lr > p.eps_high) || (A < 0.0 && lr < -p.eps_low);
    a[1] += clip ? (A > 0.0 ? p.eps_high : -p.eps_low) : lr;
    a[4] += clip ? 1.0 : 0.0;
    a[2] += p.emask ? (p.emask[n] ? 1.0 : 0.0) : 1.0;
    if (p.beta != 0.0) {
      const double d = double(p.ref_logp[n]) - lp;
      a[3] += exp(d) - d - 1.0;
    }
  } else {
    if (m) {
      a[0] += 1.0;
      a[1] += lp - double(p.old_logp[n]);
    }
    const double An = p.adv_per_token ? double(p.adv[n]) : (m ? A : 0.0);
    if (An > 0.0) a[2] += An; else a[3] += An;
  }
}

// Sequence record from the sequence's sums: [0] term of the loss, [1] n_i,
// [2] clip count, [3] sum of KL, [4] tokens kept by the entropy mask, [5]
// sequence log ratio, [6] sequence ratio, [7] GMPO: kept fraction ebar_i;
// GMPO coefficient factors [8] 1/(B n_i) and [9] -A_i r_i ebar_i/(B n_i).
__device__ __forceinline__ void seq_record(const LossParams& p, const double (&s5)[5], double A, bool gmpo,
                                           double (&r8)[kRec]) {
  const double ni = s5[0];
  for (int k = 0; k < kRec; ++k) r8[k] = 0.0;
  r8[1] = ni;
  if (gmpo) {
    const double mean_x = ni > 0 ? s5[1] / ni : 0.0;
    const double r = ni > 0 ? exp(mean_x) : 0.0;
    const double ebar = ni > 0 ? s5[2] / ni : 0.0;
    const double klt = ni > 0 ? s5[3] / ni : 0.0;
    r8[0] = ni > 0 ? -A * r * ebar + p.beta * klt : 0.0;
    r8[2] = s5[4]; r8[3] = s5[3]; r8[4] = s5[2]; r8[5] = mean_x; r8[6] = r; r8[7] = ebar;
    if (ni > 0) {
      r8[8] = 1.0 / (p.Bg * ni);
      r8[9] = -A * r * ebar * r8[8];
    }
  } else if (ni == 0) {
    if (p.status) atomicOr(p.status, RLLOSS_DEV_EEMPTYSEQ);
  } else {
    // min(s A, clip(s) A) = A min(s, clip(s)) for A > 0 and A max(s, clip(s)) for A < 0
    const double slr = s5[1] / ni;
    const double sv = exp(slr);
    const double sc = fmin(fmax(sv, p.clip_lo), p.clip_hi);
    r8[0] = -(fmin(sv, sc) * s5[2] + fmax(sv, sc) * s5[3]);
    r8[2] = (sv < p.clip_lo || sv > p.clip_hi) ? 1.0 : 0.0;
    r8[4] = ni; r8[5] = slr; r8[6] = sv;
  }
}

// Token n's gradient coefficient c_n = dL/dlogp_n (r = its sequence record).
__device__ __forceinline__ double token_coef(const LossParams& p, long long n, int i, const double* r, bool gmpo) {
  const double ni = r[1];
  double c = 0.0;
  if (!gmpo && ni > 0) {
    const double An = p.adv_per_token ? double(p.adv[n]) : (p.mask[n] ? double(p.adv[i]) : 0.0);
    const double sv = r[6];
    const bool flat = (An > 0.0 && sv > p.clip_hi) || (An < 0.0 && sv < p.clip_lo);
    c = flat ? 0.0 : -An * sv;
  } else if (gmpo && p.mask[n] && ni > 0) {
    const double A = double(p.adv[i]);
    const double lp = logp_at(p, n);
    const double lr = lp - double(p.old_logp[n]);
    const bool clip = (A > 0.0 && lr > p.eps_high) || (A < 0.0 && lr < -p.eps_low);
    c = clip ? 0.0 : r[9];
    if (p.beta != 0.0) c += p.beta * (1.0 - exp(double(p.ref_logp[n]) - lp)) * r[8];
  }
  return c;
}
__device__ __forceinline__ void store_coef(const LossParams& p, long long n, double c) {
  if (p.coef) p.coef[n] = float(c * p.inv_tau);
  if (p.dlogp) p.dlogp[n] = float(c);
}

// The slices of sequence i folded by warp 0 of the block that finished last
// (lane k takes slices k, k+32, ...; then a fixed shuffle tree).  Writes the
// sequence record; returns it on lane 0.
__device__ __forceinline__ void fold_sequence(const LossParams& p, int i, int lane, bool gmpo, double (&r8)[kRec]) {
  double s5[5] = {0, 0, 0, 0, 0};
  for (int k = lane; k < p.slices; k += 32) {
    const double* pr = p.part + (size_t(i) * p.slices + k) * 5;
#pragma unroll
    for (int j = 0; j < 5; ++j) s5[j] += __ldcg(pr + j);
  }
  warp_sum_k(s5);
  if (lane == 0) {
    seq_record(p, s5, seq_adv(p, i), gmpo, r8);
    for (int k = 0; k < kRec; ++k) p.seqres[size_t(i) * kRec + k] = r8[k];
  }
}

// Loss and metrics from all sequence records, by one warp, in a fixed order.
// The eight batch sums (written to out_sums when set; each adds over ranks
// that hold different sequences of one batch): [0] sum of the sequence terms
// (GMPO: before the 1/B of the mean), [1] active tokens, [2] clipped tokens
// (GSPO: clipped sequences), [3] sum of K3 KL, [4] tokens kept by the entropy
// mask (GSPO: active tokens), [5] sum of sequence log ratios, [6] sum of
// sequence ratios (both over sequences with tokens), [7] sequences with tokens.
__device__ __forceinline__ void finish_batch(const LossParams& p, const double (&f)[8], bool gmpo);
__device__ __forceinline__ void fold_batch(const LossParams& p, int lane, bool gmpo) {
  double f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int j = lane; j < p.B; j += 32) {
    const double* r = p.seqres + size_t(j) * kRec;
    const double nj = __ldcg(r + 1);
    f[0] += __ldcg(r + 0);
    f[1] += nj;
    f[2] += __ldcg(r + 2);
    f[3] += __ldcg(r + 3);
    f[4] += __ldcg(r + 4);
    if (nj > 0) {
      f[5] += __ldcg(r + 5);
      f[6] += __ldcg(r + 6);
      f[7] += 1.0;
    }
  }
  warp_sum_k(f);
  if (lane != 0) return;
  if (p.out_sums) {
#pragma unroll
    for (int k = 0; k < 8; ++k) p.out_sums[k] = f[k];
  }
  if (!p.out_loss) {
    if (!isfinite(f[0]) && p.status) atomicOr(p.status, RLLOSS_DEV_ENONFINITE);
    return;
  }
  finish_batch(p, f, gmpo);
}

// Loss and metrics from the eight batch sums (the layout of fold_batch).
__device__ __forceinline__ void finish_batch(const LossParams& p, const double (&f)[8], bool gmpo) {
  double loss = f[0];
  const double n_act = f[1], clip = f[2], kl = f[3], kept = f[4], sx = f[5], sr = f[6], nh = f[7];
  float* m = p.out_metrics;
  if (gmpo) {
    loss /= p.Bg;
    m[0] = n_act > 0 ? float(clip / n_act) : 0.f;
    m[2] = (p.beta != 0.0 && n_act > 0) ? float(kl / n_act) : 0.f;
  } else {
    m[0] = float(clip / p.Bg);
    m[2] = 0.f;
  }
  m[1] = float(clip);
  m[3] = float(n_act);
  m[4] = p.k3 ? float(p.k3[0]) : __int_as_float(0x7fc00000);
  m[5] = float(kept);
  m[6] = nh > 0 ? float(sx / nh) : 0.f;
  m[7] = nh > 0 ? float(sr / nh) : 0.f;
  *p.out_loss = float(loss);
  if (!isfinite(loss) && p.status) atomicOr(p.status, RLLOSS_DEV_ENONFINITE);
}

// Thread 0: publish this block's slice sums and take a ticket; true (for the
// whole block) if this was the sequence's last slice.
__device__ __forceinline__ bool publish_slice(const LossParams& p, int i, int sl, const double (&a)[5], int* flag) {
  if (threadIdx.x == 0) {
    double* pr = p.part + (size_t(i) * p.slices + sl) * 5;
#pragma unroll
    for (int j = 0; j < 5; ++j) pr[j] = a[j];
    __threadfence();
    const bool last = atomicAdd(p.seq_ticket + i, 1u) == unsigned(p.slices) - 1u;
    if (last) __threadfence();
    *flag = last ? 1 : 0;
  }
  __syncthreads();
  return *flag != 0;
}

// Lane 0: take the batch ticket after writing a sequence record; true (for
// the whole warp) if this was the last sequence.
__device__ __forceinline__ bool take_batch_ticket(const LossParams& p, int lane) {
  unsigned last = 0;
  if (lane == 0) {
    __threadfence();
    last = atomicAdd(p.ticket, 1u) == unsigned(p.B) - 1u;
    if (last) __threadfence();
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  __syncwarp();
  return last != 0;
}

// Partial sums of one slice of one sequence; the last slice block of a
// sequence folds the slices in order into the sequence record, and the last
// sequence folds the records into the loss and metrics (fixed order, so the
// result does not depend on block timing).
__global__ void __launch_bounds__(kLossThreads) loss_partial_kernel(LossParams p) {
  __shared__ double sh[5][32];
  __shared__ int is_last;
  const int i = blockIdx.y;
  const int sl = blockIdx.x;
  const long long base = (long long)i * p.T;
  const int t0 = int((long long)sl * p.T / p.slices);
  const int t1 = int((long long)(sl + 1) * p.T / p.slices);
  const double A = seq_adv(p, i);
  const bool gmpo = p.loss_type == RLLOSS_GMPO;
  double a[5] = {0, 0, 0, 0, 0};
  if (gmpo && !p.logp_is_f64) {
    // fp32 log-probs: the same terms with the clip test exact in fp32 (two-sum),
    // integer counts, and the clipped log ratios summed in compensated fp32
    // (one thread's few hundred tokens) before the fp64 block sums
    const float* lpf = static_cast<const float*>(p.logp);
    const float eh = float(p.eps_high), el = float(-p.eps_low);   // the fp32 bounds, exactly
    int cnt = 0, clips = 0, kept = 0;
    float sum = 0.f, comp = 0.f, slo = 0.f, nonfin = 0.f;   // nonfin: infinite or NaN terms, as fp64 adds them
    double kl = 0.0;
    auto term = [&](long long n, float lp, float old, bool kept_bit) {
      const ExactDiff d = exact_diff(lp, old);
      const bool clip = gmpo_clipped(d, A, eh, el);
      const float x = clip ? (A > 0.0 ? eh : el) : d.hi;
      if (!isfinite(x)) {
        nonfin += x;
      } else {
        if (!clip) slo += d.lo;
        const float y = x - comp;   // Kahan
        const float tt = sum + y;
        comp = (tt - sum) - y;
        sum = tt;
      }
      ++cnt;
      clips += clip ? 1 : 0;
      kept += kept_bit ? 1 : 0;
      if (p.beta != 0.0) {
        const double dk = double(p.ref_logp[n]) - double(lp);
        kl += exp(dk) - dk - 1.0;
      }
    };
    auto scalar = [&](long long n) {
      if (p.mask[n]) term(n, lpf[n], p.old_logp[n], p.emask ? p.emask[n] != 0 : true);
    };
    const long long n0 = base + t0, n1 = base + t1;
    const bool vec = ((reinterpret_cast<uintptr_t>(lpf) | reinterpret_cast<uintptr_t>(p.old_logp)) & 15u) == 0 &&
                     ((reinterpret_cast<uintptr_t>(p.mask) | reinterpret_cast<uintptr_t>(p.emask)) & 3u) == 0;
    if (vec) {
      // four tokens a thread over the slice's aligned groups; the ends one by one
      const long long g0 = (n0 + 3) / 4, g1 = n1 / 4;
      if (g0 < g1) {
        for (long long n = n0 + threadIdx.x; n < 4 * g0; n += blockDim.x) scalar(n);
        for (long long n = 4 * g1 + threadIdx.x; n < n1; n += blockDim.x) scalar(n);
#pragma unroll 2
        for (long long g = g0 + threadIdx.x; g < g1; g += blockDim.x) {
          const uint32_t mw = __ldg(reinterpret_cast<const uint32_t*>(p.mask) + g);
          if (!mw) continue;
          const uint32_t ew = p.emask ? __ldg(reinterpret_cast<const uint32_t*>(p.emask) + g) : 0x01010101u;
          const float4 l4 = __ldg(reinterpret_cast<const float4*>(lpf) + g);
          const float4 o4 = __ldg(reinterpret_cast<const float4*>(p.old_logp) + g);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, ov[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if ((mw >> (8 * k)) & 255u) term(4 * g + k, lv[k], ov[k], ((ew >> (8 * k)) & 255u) != 0u);
        }
      } else {
        for (long long n = n0 + threadIdx.x; n < n1; n += blockDim.x) scalar(n);
      }
    } else {
#pragma unroll 4
      for (long long n = n0 + threadIdx.x; n < n1; n += blockDim.x) scalar(n);
    }
    a[0] = double(cnt);
    a[1] = ((double(sum) - double(comp)) + double(slo)) + double(nonfin);
    a[2] = double(kept);
    a[3] = kl;
    a[4] = double(clips);
  } else {
#pragma unroll 4
    for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
      const long long n = base + t;
      token_terms(p, n, logp_at(p, n), A, gmpo, a);
    }
  }
  block_sum_k(a, sh);
  if (!publish_slice(p, i, sl, a, &is_last) || threadIdx.x >= 32) return;
  double r8[kRec];
  fold_sequence(p, i, threadIdx.x, gmpo, r8);
  if (take_batch_ticket(p, threadIdx.x)) fold_batch(p, threadIdx.x, gmpo);
}

// Per-token gradient coefficient c_n = dL/dlogp_n from the sequence records:
// block (sl, i) takes slice sl of sequence i, with the sequence's record in
// shared memory.
__global__ void loss_coef_kernel(LossParams p) {
  __shared__ double rec[kRec];
  const int i = blockIdx.y;
  if (threadIdx.x < kRec) rec[threadIdx.x] = __ldcg(p.seqres + size_t(i) * kRec + threadIdx.x);
  __syncthreads();
  const bool gmpo = p.loss_type == RLLOSS_GMPO;
  const long long base = (long long)i * p.T;
  const int t0 = int((long long)blockIdx.x * p.T / gridDim.x);
  const int t1 = int((long long)(blockIdx.x + 1) * p.T / gridDim.x);
  if (gmpo && !p.logp_is_f64 && p.beta == 0.0) {
    // fp32 log-probs without KL: c_n is the sequence's factor for unclipped
    // active tokens and 0 otherwise, the clip test exact in fp32 (two-sum)
    const float* lpf = static_cast<const float*>(p.logp);
    const float eh = float(p.eps_high), el = float(-p.eps_low);
    const double A = double(p.adv[i]);
    const bool live = rec[1] > 0;
    const float cf = float(rec[9] * p.inv_tau), cd = float(rec[9]);
    auto one = [&](long long n, bool m, float lp, float old) {
      return live && m && !gmpo_clipped(exact_diff(lp, old), A, eh, el);
    };
    auto scalar = [&](long long n) {
      const bool on = one(n, p.mask[n] != 0, lpf[n], p.old_logp[n]);
      if (p.coef) p.coef[n] = on ? cf : 0.f;
      if (p.dlogp) p.dlogp[n] = on ? cd : 0.f;
    };
    const long long n0 = base + t0, n1 = base + t1;
    const bool vec = ((reinterpret_cast<uintptr_t>(lpf) | reinterpret_cast<uintptr_t>(p.old_logp) |
                       reinterpret_cast<uintptr_t>(p.coef) | reinterpret_cast<uintptr_t>(p.dlogp)) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(p.mask) & 3u) == 0;
    const long long g0 = (n0 + 3) / 4, g1 = n1 / 4;
    if (vec && g0 < g1) {
      // four tokens a thread over the slice's aligned groups; the ends one by one
      for (long long n = n0 + threadIdx.x; n < 4 * g0; n += blockDim.x) scalar(n);
      for (long long n = 4 * g1 + threadIdx.x; n < n1; n += blockDim.x) scalar(n);
#pragma unroll 2
      for (long long g = g0 + threadIdx.x; g < g1; g += blockDim.x) {
        const uint32_t mw = __ldg(reinterpret_cast<const uint32_t*>(p.mask) + g);
        float4 c4 = make_float4(0.f, 0.f, 0.f, 0.f), d4 = c4;
        if (mw && live) {
          const float4 l4 = __ldg(reinterpret_cast<const float4*>(lpf) + g);
          const float4 o4 = __ldg(reinterpret_cast<const float4*>(p.old_logp) + g);
          const bool b0 = one(4 * g, mw & 0xffu, l4.x, o4.x), b1 = one(4 * g + 1, mw & 0xff00u, l4.y, o4.y),
                     b2 = one(4 * g + 2, mw & 0xff0000u, l4.z, o4.z), b3 = one(4 * g + 3, mw & 0xff000000u, l4.w, o4.w);
          c4 = make_float4(b0 ? cf : 0.f, b1 ? cf : 0.f, b2 ? cf : 0.f, b3 ? cf : 0.f);
          d4 = make_float4(b0 ? cd : 0.f, b1 ? cd : 0.f, b2 ? cd : 0.f, b3 ? cd : 0.f);
        }
        if (p.coef) reinterpret_cast<float4*>(p.coef)[g] = c4;
        if (p.dlogp) reinterpret_cast<float4*>(p.dlogp)[g] = d4;
      }
    } else {
      for (long long n = n0 + threadIdx.x; n < n1; n += blockDim.x) scalar(n);
    }
    return;
  }
#pragma unroll 4
  for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
    const long long n = base + t;
    store_coef(p, n, token_coef(p, n, i, rec, gmpo));
  }
}

// Row merge and loss sums in one launch, for batches without the entropy
// mask (no batch-global threshold sits between the two): block (sl, i)
// merges rows [16 sl, 16 sl + 16) of sequence i (a warp per row) and sums
// their loss terms; the sequence's last block folds the slices into the
// sequence record and the last sequence folds the batch.  The coefficients
// follow in loss_coef_kernel (one sequence's tokens are too many for the
// one block that holds its record).
__global__ void __launch_bounds__(kLossThreads) merge_loss_kernel(MergeParams mp, LossParams p) {
  __shared__ double sh[5][32];
  __shared__ int is_last;
  const int i = blockIdx.y;
  const int sl = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long base = (long long)i * p.T;
  const int t0 = sl * kFusedRows;
  const int t1 = min(p.T, t0 + kFusedRows);
  const double A = seq_adv(p, i);
  const bool gmpo = p.loss_type == RLLOSS_GMPO;
  double a[5] = {0, 0, 0, 0, 0};
  {
    const int t = t0 + warp * kMergeRowsPerWarp + (lane / kMergeLanes);   // this lane group's row
    const long long n = base + t;
    const bool live = t < t1 && row_has_forward(mp, int(n));   // skipped tiles: every row masked, no terms
    const double lp = merge_row(mp, live ? int(n) : -1, lane % kMergeLanes);
    if (live && lane % kMergeLanes == 0) token_terms(p, n, lp, A, gmpo, a);
    if (lane % kMergeLanes == 0) __threadfence();   // this row's outputs before the slice ticket
  }
  block_sum_k(a, sh);
  if (!publish_slice(p, i, sl, a, &is_last) || warp != 0) return;
  double r8[kRec];
  fold_sequence(p, i, lane, gmpo, r8);
  if (take_batch_ticket(p, lane)) fold_batch(p, lane, gmpo);
}

int loss_slices(int B, int T, int sms) {
  long long s = (16ll * sms + B - 1) / B;
  const long long smax = (T + 255) / 256;
  if (s > smax) s = smax;
  if (s < 1) s = 1;
  return int(s);
}

int fused_loss_slices(int T) { return (T + kFusedRows - 1) / kFusedRows; }

// Slices of >= 256 tokens per sequence for the coefficient kernel, about 16
// blocks per SM over the batch.
int coef_slices(int B, int T, int sms) {
  long long s = (16ll * sms + B - 1) / B;
  const long long smax = (T + 255) / 256;
  if (s > smax) s = smax;
  if (s < 1) s = 1;
  return int(s);
}

static cudaError_t launch_coef(const LossParams& p, cudaStream_t st) {
  long long s = p.coef_slices > 0 ? p.coef_slices : (p.T + 255) / 256;
  if (s < 1) s = 1;
  loss_coef_kernel<<<dim3(unsigned(s), unsigned(p.B)), 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_merge_loss(const MergeParams& mp, const LossParams& p, cudaStream_t st) {
  merge_loss_kernel<<<dim3(p.slices, p.B), kLossThreads, 0, st>>>(mp, p);
  if (p.coef || p.dlogp) return launch_coef(p, st);
  return cudaGetLastError();
}

// Loss and metrics from the batch sums of several groups of sequences
// ([ngroups][8], each written as LossParams::out_sums), added in group order.
__global__ void fold_sums_kernel(const double* sums, int ngroups, LossParams p) {
  if (threadIdx.x != 0) return;
  double f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int g = 0; g < ngroups; ++g)
#pragma unroll
    for (int k = 0; k < 8; ++k) f[k] += __ldcg(sums + size_t(g) * 8 + k);
  finish_batch(p, f, p.loss_type == RLLOSS_GMPO);
}

cudaError_t launch_fold_sums(const double* sums, int ngroups, const LossParams& p, cudaStream_t st) {
  fold_sums_kernel<<<1, 32, 0, st>>>(sums, ngroups, p);
  return cudaGetLastError();
}

cudaError_t launch_loss(const LossParams& p, cudaStream_t st) {
  loss_partial_kernel<<<dim3(p.slices, p.B), kLossThreads, 0, st>>>(p);
  if (p.coef || p.dlogp) return launch_coef(p, st);
  return cudaGetLastError();
}

}  // namespace rl
