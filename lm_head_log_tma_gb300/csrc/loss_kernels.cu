// Loss-stage kernels.
//
//  K3 entropy quantile: exact order statistics of the active tokens'
//     entropies by a 4-pass, 8-bit radix select on order-preserving uint32
//     keys, then linear interpolation at position (1-q)(n_act-1) and the mask
//     H >= threshold — "support top_entropy_quantile in fused linear GRPO
//     loss", Details (batch-global quantile of active entropies at 1 - q).
//  K2 per-sequence reduction: one block per sequence, fp64 sums, then the
//     per-token gradient coefficient c_n = dL/dlogp_n; the last block to
//     finish folds the per-sequence terms into the loss and metrics in a
//     fixed order.  GMPO: "Add GMPO to fused linear GRPO loss", Summary and
//     Details.  GSPO-token: Tinker "GSPO", ratio and objective formulas.
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"
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
  for (long long n = blockIdx.x * (long long)blockDim.x + threadIdx.x; n < N; n += (long long)gridDim.x * blockDim.x) {
    if (!m[n]) continue;
    const uint32_t key = f2key(H[n]);
    const uint32_t d = (key >> shift) & 255u;
    if (pass == 0) {
      atomicAdd(&sh[d], 1u);
    } else {
      const uint32_t hp = key >> (shift + 8);
      if (hp == p0) atomicAdd(&sh[d], 1u);
      if (hp == p1) atomicAdd(&sh[256 + d], 1u);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 512; i += blockDim.x)
    if (sh[i]) atomicAdd(&hist[i], sh[i]);
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
  const double thr = st->thr;
  for (long long n = blockIdx.x * (long long)blockDim.x + threadIdx.x; n < N; n += (long long)gridDim.x * blockDim.x)
    e[n] = (m[n] && double(H[n]) >= thr) ? 1 : 0;
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

// ----------------------------------------------------------------------- K2
constexpr int kLossThreads = 256;

__device__ __forceinline__ double block_sum(double v, double* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  double r = 0.0;
  if (threadIdx.x == 0)
    for (int i = 0; i < int(blockDim.x >> 5); ++i) r += sh[i];
  return r;   // valid in thread 0
}

__device__ __forceinline__ double logp_at(const LossParams& p, long long n) {
  return p.logp_is_f64 ? static_cast<const double*>(p.logp)[n] : double(static_cast<const float*>(p.logp)[n]);
}

// Partial sums of one slice of one sequence; the last slice block of a
// sequence folds the slices in order into the sequence record, and the last
// sequence folds the records into the loss and metrics (fixed order, so the
// result does not depend on block timing).
//
// Sequence record: [0] term of the loss, [1] n_i, [2] clip count, [3] sum of
// KL, [4] tokens kept by the entropy mask, [5] sequence log ratio, [6]
// sequence ratio, [7] GMPO: kept fraction ebar_i; GSPO: gradient gate.
__global__ void __launch_bounds__(kLossThreads) loss_partial_kernel(LossParams p) {
  __shared__ double sh[32];
  __shared__ int is_last;
  const int i = blockIdx.y;
  const int sl = blockIdx.x;
  const long long base = (long long)i * p.T;
  const int t0 = int((long long)sl * p.T / p.slices);
  const int t1 = int((long long)(sl + 1) * p.T / p.slices);
  const double A = p.adv_per_token ? 0.0 : double(p.adv[i]);
  const bool gmpo = p.loss_type == RLLOSS_GMPO;
  // GMPO: a_e = tokens kept by the entropy mask, a_kl = sum of K3 KL.
  // GSPO: a_e / a_kl = sums of the positive / negative token advantages.
  double a_m = 0, a_x = 0, a_e = 0, a_kl = 0, a_clip = 0;
  for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
    const long long n = base + t;
    const bool m = p.mask[n] != 0;
    if (gmpo) {
      if (!m) continue;
      const double lp = logp_at(p, n);
      const double lr = lp - double(p.old_logp[n]);
      a_m += 1.0;
      const bool clip = (A > 0.0 && lr > p.eps_high) || (A < 0.0 && lr < -p.eps_low);
      a_x += clip ? (A > 0.0 ? p.eps_high : -p.eps_low) : lr;
      a_clip += clip ? 1.0 : 0.0;
      a_e += p.emask ? (p.emask[n] ? 1.0 : 0.0) : 1.0;
      if (p.beta != 0.0) {
        const double d = double(p.ref_logp[n]) - lp;
        a_kl += exp(d) - d - 1.0;
      }
    } else {
      if (m) {
        a_m += 1.0;
        a_x += logp_at(p, n) - double(p.old_logp[n]);
      }
      const double An = p.adv_per_token ? double(p.adv[n]) : (m ? A : 0.0);
      if (An > 0.0) a_e += An; else a_kl += An;
    }
  }
  a_m = block_sum(a_m, sh);
  a_x = block_sum(a_x, sh);
  a_e = block_sum(a_e, sh);
  a_kl = block_sum(a_kl, sh);
  a_clip = block_sum(a_clip, sh);
  if (threadIdx.x == 0) {
    double* pr = p.part + (size_t(i) * p.slices + sl) * 5;
    pr[0] = a_m; pr[1] = a_x; pr[2] = a_e; pr[3] = a_kl; pr[4] = a_clip;
    __threadfence();
    is_last = atomicAdd(p.seq_ticket + i, 1u) == unsigned(p.slices) - 1u;
  }
  __syncthreads();
  if (!is_last || threadIdx.x != 0) return;
  __threadfence();
  double s5[5] = {0, 0, 0, 0, 0};
  for (int k = 0; k < p.slices; ++k) {
    const double* pr = p.part + (size_t(i) * p.slices + k) * 5;
    for (int j = 0; j < 5; ++j) s5[j] += __ldcg(pr + j);
  }
  const double ni = s5[0];
  double r8[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  r8[1] = ni;
  if (gmpo) {
    const double mean_x = ni > 0 ? s5[1] / ni : 0.0;
    const double r = ni > 0 ? exp(mean_x) : 0.0;
    const double ebar = ni > 0 ? s5[2] / ni : 0.0;
    const double klt = ni > 0 ? s5[3] / ni : 0.0;
    r8[0] = ni > 0 ? -A * r * ebar + p.beta * klt : 0.0;
    r8[2] = s5[4]; r8[3] = s5[3]; r8[4] = s5[2]; r8[5] = mean_x; r8[6] = r; r8[7] = ebar;
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
  for (int k = 0; k < 8; ++k) p.seqres[size_t(i) * 8 + k] = r8[k];
  __threadfence();
  if (atomicAdd(p.ticket, 1u) != unsigned(p.B) - 1u) return;
  __threadfence();
  double loss = 0, n_act = 0, clip = 0, kl = 0, kept = 0, sx = 0, sr = 0, nh = 0;
  for (int j = 0; j < p.B; ++j) {
    const double* r = p.seqres + size_t(j) * 8;
    const double nj = __ldcg(r + 1);
    loss += __ldcg(r + 0);
    n_act += nj;
    clip += __ldcg(r + 2);
    kl += __ldcg(r + 3);
    kept += __ldcg(r + 4);
    if (nj > 0) {
      sx += __ldcg(r + 5);
      sr += __ldcg(r + 6);
      nh += 1.0;
    }
  }
  float* m = p.out_metrics;
  if (gmpo) {
    loss /= double(p.B);
    m[0] = n_act > 0 ? float(clip / n_act) : 0.f;
    m[2] = (p.beta != 0.0 && n_act > 0) ? float(kl / n_act) : 0.f;
  } else {
    m[0] = float(clip / double(p.B));
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

// Per-token gradient coefficient c_n = dL/dlogp_n from the sequence records.
__global__ void loss_coef_kernel(LossParams p) {
  const long long N = (long long)p.B * p.T;
  const bool gmpo = p.loss_type == RLLOSS_GMPO;
  for (long long n = blockIdx.x * (long long)blockDim.x + threadIdx.x; n < N; n += (long long)gridDim.x * blockDim.x) {
    const int i = int(n / p.T);
    const double* r = p.seqres + size_t(i) * 8;
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
      c = clip ? 0.0 : -A * r[6] * r[7];
      if (p.beta != 0.0) c += p.beta * (1.0 - exp(double(p.ref_logp[n]) - lp));
      c /= double(p.B) * ni;
    }
    if (p.coef) p.coef[n] = float(c * p.inv_tau);
    if (p.dlogp) p.dlogp[n] = float(c);
  }
}

int loss_slices(int B, int T, int sms) {
  long long s = (4ll * sms + B - 1) / B;
  const long long smax = (T + 255) / 256;
  if (s > smax) s = smax;
  if (s < 1) s = 1;
  return int(s);
}

cudaError_t launch_loss(const LossParams& p, cudaStream_t st) {
  loss_partial_kernel<<<dim3(p.slices, p.B), kLossThreads, 0, st>>>(p);
  if (p.coef || p.dlogp) {
    const long long N = (long long)p.B * p.T;
    long long nb = (N + 255) / 256;
    if (nb > 4096) nb = 4096;
    loss_coef_kernel<<<int(nb), 256, 0, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace rl
