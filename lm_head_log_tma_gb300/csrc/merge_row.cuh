// Row merge of the forward's partial softmax states, shared by the merge
// kernel and the fused merge + loss kernel.
#pragma once
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"
#include "status.h"

namespace rl {

// Merge the 2P partial states of each row.  Each partial holds, for one
// vocabulary segment and column half: reference m (log2 units, integer),
// s = sum 2^(t-m) and w = sum 2^(t-m) (t-m) as hi + lo pairs, and the
// target's t if it fell there.  With M the largest m,
//   S = sum_k 2^(m_k-M) s_k,   W = sum_k 2^(m_k-M) (w_k + (m_k-M) s_k).
// Scaling by 2^(m_k-M) is exact in fp32, the sums are carried as
// double-float (hi + lo) pairs, and only the final row values use fp64.
//
// Eight lanes merge one row (a warp holds 4 rows): each lane takes every
// eighth slot, with the slot loops unrolled so a lane's loads are in flight
// together (the merge is bound by load latency), the group combines with
// three shuffle steps, and the group's first lane finishes the row, so the
// per-row fp64 work runs for 4 rows at once (fp64 is a narrow unit on this
// GPU; a warp instruction costs the same with one active lane as with four).
constexpr int kMergeLanes = 8;
constexpr int kMergeRowsPerWarp = 32 / kMergeLanes;

__device__ __forceinline__ float pow2_int(int d) {
  // 2^d for an integer d <= 0; 0 below 2^-126 (such a slot weighs less than
  // 2^-90 of the row sum: the forward keeps every s of the maximal slot >= 1/2)
  return d < -126 ? 0.f : __int_as_float((127 + d) << 23);
}
// Sum of a double-float pair over the lanes of a group (every lane of the
// group gets a sum; the group's first lane's is the one used).
__device__ __forceinline__ void df_group_sum(float& hi, float& lo) {
#pragma unroll
  for (int o = 1; o < kMergeLanes; o <<= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, hi, o);
    const float ol = __shfl_xor_sync(0xffffffffu, lo, o);
    two_sum_acc(hi, lo, oh);
    lo += ol;
  }
}

// False for rows of row tiles the forward skipped (every row there is masked).
__device__ __forceinline__ bool row_has_forward(const MergeParams& p, int row) {
  return !p.tile_active || p.tile_active[row >> p.tile_shift];
}

// A row's merged softmax state, valid on the first lane of its group: the
// reference M, S and W as hi + lo pairs against M, the target's t and the
// group lanes whose slot held it (who), and the row's target id (y).
struct RowSums {
  float M, shi, slo, whi, wlo, zy;
  unsigned who;
  long long y;
};

// Slot k of `row`: layout [N][slots][2] float4 (slot_stride == 0), or
// [slots][slot_stride][2] float4 (states gathered from vocabulary shards).
__device__ __forceinline__ const float4* slot_ptr(const MergeParams& p, int row, int slots, int k) {
  return p.slot_stride ? p.partial + (size_t(k) * p.slot_stride + row) * 2
                       : p.partial + (size_t(row) * slots + k) * 2;
}

// Merges the slots of `row` over the lanes of this lane's group (sub = lane %
// kMergeLanes; all 32 lanes of the warp must call it, with `row` < 0 for
// groups without a row).
__device__ __forceinline__ RowSums merge_slots(const MergeParams& p, int row, int sub) {
  const bool live = row >= 0;
  RowSums r;
  r.y = (live && sub == 0) ? p.targets[row] : 0;   // issued early, used at the end
  const int slots = p.P_dev ? 2 * *p.P_dev : p.slots;
  const int nk = live ? slots : 0;
  const int rr = live ? row : 0;
  float M = -INFINITY;
#pragma unroll 4
  for (int k = sub; k < nk; k += kMergeLanes) {
    const float4 a = slot_ptr(p, rr, slots, k)[0];
    if (a.y + a.z > 0.f) M = fmaxf(M, a.x);
  }
#pragma unroll
  for (int o = 1; o < kMergeLanes; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float shi = 0.f, slo = 0.f, whi = 0.f, wlo = 0.f, zy = 0.f;
  int found = 0;
#pragma unroll 4
  for (int k = sub; k < nk; k += kMergeLanes) {
    const float4* sp = slot_ptr(p, rr, slots, k);
    const float4 a = sp[0];
    const float4 b = sp[1];
    if (a.y + a.z > 0.f) {
      const float d = a.x - M;                   // integer, <= 0, exact
      const float f = pow2_int(int(d));
      two_sum_acc(shi, slo, a.y * f);
      slo += a.z * f;
      const float ds = d * a.y;                  // d * s_hi = ds + dse exactly
      const float dse = fmaf(d, a.y, -ds);
      two_sum_acc(whi, wlo, a.w * f);
      two_sum_acc(whi, wlo, ds * f);
      wlo += ((b.x + dse) + d * a.z) * f;
    }
    if (b.z != 0.f) {
      zy = b.y;
      found = 1;
    }
  }
  df_group_sum(shi, slo);
  df_group_sum(whi, wlo);
  const int lane = threadIdx.x & 31;
  const int g0 = lane & ~(kMergeLanes - 1);   // first lane of this group
  const unsigned gmask = ((1u << kMergeLanes) - 1u) << g0;
  r.who = __ballot_sync(0xffffffffu, found) & gmask;
  r.zy = __shfl_sync(0xffffffffu, zy, r.who ? __ffs(r.who) - 1 : g0);
  r.M = M;
  r.shi = shi;
  r.slo = slo;
  r.whi = whi;
  r.wlo = wlo;
  return r;
}

// Writes the row's lse, logp and entropy from its merged state (first lane
// of the group only) and returns the logp (NaN for a bad target).
__device__ __forceinline__ double finish_row(const MergeParams& p, int row, const RowSums& r) {
  const float M = r.M, shi = r.shi, slo = r.slo, whi = r.whi, wlo = r.wlo;
  // log2 S = e + log2(mh) + log2(1 + slo/shi), with shi = 2^e mh, mh in
  // [1, 2) (S >= 1/2, so shi is a normal number): log2f on [1, 2) is within
  // an ulp of [0, 1); the last term is slo/shi/ln2 to first order
  // (|slo/shi| < 2^-23).  W/S = q + q_lo with q = whi/shi and the exact
  // division residual.  Both log2 S and log2 S - W/S are formed as fp32
  // hi + lo pairs; fp64 only joins and scales them.
  const uint32_t sb = __float_as_uint(shi);
  const float e = float(int(sb >> 23) - 127);
  const float l2m = log2f(__uint_as_float((sb & 0x7fffffu) | 0x3f800000u));
  const float corr = (slo / shi) * 1.44269504f;
  const float q = whi / shi;
  const float q_lo = (fmaf(-q, shi, whi) + fmaf(-q, slo, wlo)) / shi;
  float yh = e, yl = 0.f;                  // log2 S
  two_sum_acc(yh, yl, l2m);
  yl += corr;
  float xh = yh, xl = yl;                  // log2 S - W/S
  two_sum_acc(xh, xl, -q);
  xl -= q_lo;
  const double ln2 = 0.6931471805599453;
  const double l2s = double(yh) + double(yl);
  const double lse2 = double(M) + l2s;
  const double ent = ln2 * (double(xh) + double(xl));
  double logp = ln2 * (double(r.zy) - lse2);
  if (r.y < 0 || r.y >= p.V || !r.who) {
    logp = __longlong_as_double(0x7ff8000000000000ll);
    if (p.status) atomicOr(p.status, RLLOSS_DEV_EBADTARGET);
  }
  p.lse2[row] = float(lse2);
  p.logp64[row] = logp;
  p.ent32[row] = float(ent);
  if (p.out_logp) p.out_logp[row] = float(logp);
  if (p.out_ent) p.out_ent[row] = float(ent);
  if (p.out_lse) p.out_lse[row] = float(ln2 * lse2);
  return logp;
}

// Merges `row` (see merge_slots) and writes its lse, logp and entropy.
// Returns the row's logp on the group's first lane (NaN for a bad target),
// 0 elsewhere.
__device__ __forceinline__ double merge_row(const MergeParams& p, int row, int sub) {
  const RowSums r = merge_slots(p, row, sub);
  if (row < 0 || sub != 0) return 0.0;
  return finish_row(p, row, r);
}

}  // namespace rl
