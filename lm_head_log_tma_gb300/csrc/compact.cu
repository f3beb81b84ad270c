// Backward row compaction.
//
// The backward's per-row factor is the gradient coefficient c_n (GMPO page,
// Details: the input/weight/bias gradients are sums over tokens of
// c_n (onehot - p_n) against W or X).  A row with c_n = 0 -- a prompt or
// padding token, a token whose log ratio is clipped (no KL term), every token
// of a clipped GSPO sequence -- adds exactly nothing to dX, dW or db, so the
// recompute and both GEMMs run over the other rows only.  The compaction is
// ordered (a prefix sum over 32-row groups, ranks within a group by a warp
// ballot), so repeated calls see the same row order and give the same bits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace rl {

constexpr int kCompactBlock = 256;
constexpr int kGroup = 32;        // rows per compaction group (one warp's ballot)

// Per 32-row group: rows with c != 0.  The block that finishes last turns
// the counts into exclusive offsets (fixed order), writes the total and
// zero-fills the compacted arrays from the total up to the next multiple of
// 256 rows (the backward reads whole 256-row tiles).
__global__ void __launch_bounds__(kCompactBlock) compact_count_kernel(CompactParams p) {
  __shared__ int is_last;
  __shared__ int part[kCompactBlock];
  const int n = blockIdx.x * kCompactBlock + threadIdx.x;
  const unsigned bal = __ballot_sync(0xffffffffu, n < p.N && p.coef[n] != 0.f && !(p.done && p.done[n]));
  const int ngroups = (p.N + kGroup - 1) / kGroup;
  const int grp = n / kGroup;
  if ((threadIdx.x & 31) == 0 && grp < ngroups) p.blk_cnt[grp] = __popc(bal);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    is_last = atomicAdd(p.ticket, 1u) == gridDim.x - 1;
    if (is_last) __threadfence();
  }
  __syncthreads();
  if (!is_last) return;
  const int per = (ngroups + kCompactBlock - 1) / kCompactBlock;   // consecutive groups per thread
  int s = 0;
  for (int k = 0; k < per; ++k) {
    const int i = threadIdx.x * per + k;
    if (i < ngroups) s += __ldcg(p.blk_cnt + i);
  }
  part[threadIdx.x] = s;
  __syncthreads();
  for (int o = 1; o < kCompactBlock; o <<= 1) {   // inclusive scan of part[]
    const int v = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int base = threadIdx.x ? part[threadIdx.x - 1] : 0;
  for (int k = 0; k < per; ++k) {
    const int i = threadIdx.x * per + k;
    if (i < ngroups) {
      p.blk_off[i] = base;
      base += __ldcg(p.blk_cnt + i);
    }
  }
  const int total = part[kCompactBlock - 1];
  if (threadIdx.x == 0) *p.total = total;
  const int tail_end = min((total + 255) / 256 * 256, p.Ncap);
  for (int r = total + threadIdx.x; r < tail_end; r += kCompactBlock) {
    p.idx[r] = 0;
    p.coefc[r] = 0.f;
    p.lse2c[r] = 0.f;
    p.tgtc[r] = -1;
    if (p.errc) p.errc[r] = 0.f;
  }
  if (p.xc) {
    const int words = p.Kx / 8;   // 16-byte words per row
    const long long tail_words = (long long)(tail_end - total) * words;
    for (long long w = threadIdx.x; w < tail_words; w += kCompactBlock) {
      const long long r = total + w / words;
      reinterpret_cast<uint4*>(p.xc + r * p.Kx)[w % words] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// Block b handles the 32 rows of group b: each kept row goes to its group's
// offset plus its rank in the group, with its index, coefficient, lse and
// target; then the block copies the kept X rows (16-byte words spread over
// all threads) and, with dx_zero set, zeroes the group's gradient rows.
__global__ void __launch_bounds__(kCompactBlock) compact_gather_kernel(CompactParams p) {
  __shared__ int rows[kGroup];
  __shared__ int cnt;
  const int g = blockIdx.x;
  if (threadIdx.x < 32) {
    const int n = g * kGroup + threadIdx.x;
    const bool keep = n < p.N && p.coef[n] != 0.f && !(p.done && p.done[n]);
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    const int rank = __popc(bal & ((1u << threadIdx.x) - 1u));
    if (keep && RL_DCHECK(p.blk_off[g] + rank < p.Ncap, p.status)) {
      const int pos = p.blk_off[g] + rank;
      p.idx[pos] = n;
      p.coefc[pos] = p.coef[n];
      p.lse2c[pos] = p.lse2[n];
      p.tgtc[pos] = p.targets[n];
      if (p.errc) p.errc[pos] = 0.f;
      rows[rank] = n;
    }
    if (threadIdx.x == 0) cnt = __popc(bal);
  }
  __syncthreads();
  if (p.xc) {
    const int base = p.blk_off[g];
    const int words = p.Kx / 8;
    const int total_words = cnt * words;
    for (int w = threadIdx.x; w < total_words; w += kCompactBlock) {
      const int r = w / words, c = w - r * words;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.x + size_t(rows[r]) * p.Kx) + c);
      reinterpret_cast<uint4*>(p.xc + size_t(base + r) * p.Kx)[c] = v;
    }
  }
  if (p.dx_zero) {
    const int r0 = g * kGroup;
    const int nr = min(kGroup, p.N - r0);
    float* d = p.dx_zero + size_t(r0) * p.H;
    if (p.dx_vec) {
      const int n4 = nr * (p.H / 4);
      for (int i = threadIdx.x; i < n4; i += kCompactBlock)
        reinterpret_cast<float4*>(d)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      const int n1 = nr * p.H;
      for (int i = threadIdx.x; i < n1; i += kCompactBlock) d[i] = 0.f;
    }
  }
}

// Block b: does row tile b hold a row with mask != 0?  The last block to
// finish lists the flagged tiles in ascending order.
__global__ void __launch_bounds__(kCompactBlock) tile_scan_kernel(const uint8_t* mask, int N, int tile_rows,
                                                                   uint8_t* flags, int* list, int* count,
                                                                   unsigned int* ticket) {
  __shared__ int is_last;
  __shared__ int part[kCompactBlock];
  const int r = blockIdx.x * tile_rows + threadIdx.x;
  const int any = __syncthreads_or(threadIdx.x < tile_rows && r < N && mask[r] != 0);
  if (threadIdx.x == 0) {
    flags[blockIdx.x] = any ? 1 : 0;
    __threadfence();
    is_last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    if (is_last) __threadfence();
  }
  __syncthreads();
  if (!is_last) return;
  const int nt = int(gridDim.x);
  const int per = (nt + kCompactBlock - 1) / kCompactBlock;   // consecutive tiles per thread
  int s = 0;
  for (int k = 0; k < per; ++k) {
    const int i = threadIdx.x * per + k;
    if (i < nt) s += __ldcg(flags + i);
  }
  part[threadIdx.x] = s;
  __syncthreads();
  for (int o = 1; o < kCompactBlock; o <<= 1) {   // inclusive scan of part[]
    const int v = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int pos = threadIdx.x ? part[threadIdx.x - 1] : 0;
  for (int k = 0; k < per; ++k) {
    const int i = threadIdx.x * per + k;
    if (i < nt && __ldcg(flags + i)) list[pos++] = i;
  }
  if (threadIdx.x == 0) *count = part[kCompactBlock - 1];
}

cudaError_t launch_tile_scan(const uint8_t* mask, int N, int tile_rows, uint8_t* flags, int* list, int* count,
                             unsigned int* ticket, cudaStream_t st) {
  tile_scan_kernel<<<(N + tile_rows - 1) / tile_rows, kCompactBlock, 0, st>>>(mask, N, tile_rows, flags, list, count,
                                                                             ticket);
  return cudaGetLastError();
}

__global__ void set_total_kernel(int* total, int N) { *total = N; }

__global__ void scatter_rows_kernel(const float4* src, const int* idx, const int* total, int n0, int nc_max, int H4,
                                    float4* dst, int accumulate) {
  const int nc = min(max(*total - n0, 0), nc_max);
  const long long n = (long long)nc * H4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long j = i / H4;
    const int c = int(i - j * H4);
    float4* d = dst + (long long)idx[n0 + j] * H4 + c;
    float4 v = src[i];
    if (accumulate) {   // each kept row appears once: a plain read-modify-write
      const float4 o = *d;
      v = make_float4(o.x + v.x, o.y + v.y, o.z + v.z, o.w + v.w);
    }
    *d = v;
  }
}

// Stored-probability rows (see StoredParams) in blocks of kStoredBlock buffer
// rows: a block that holds a kept row is taken whole, in buffer order, its
// other rows with zero factors; a block without one is left out.  The count
// kernel marks every 32-row group with its block's decision and its kept rows
// (packed: marked << 16 | kept); the block that finishes last turns the marks
// into positions and fills the tail up to a whole 256-row tile; then every
// marked group writes its rows at their positions.
constexpr int kStoredBlock = 128;
static_assert(kCompactBlock % kStoredBlock == 0 && kStoredBlock % kGroup == 0, "block split");
__device__ __forceinline__ int stored_source(const StoredParams& p, int j) {
  const int slot = j >> 8;
  return (p.tiles ? p.tiles[slot] : slot) * 256 + (j & 255);
}
__device__ __forceinline__ bool stored_keep(const StoredParams& p, int n) {
  if (n >= p.N) return false;
  const float l2 = p.lse2[n];
  const long long y = p.targets[n];
  return p.coef[n] != 0.f && l2 >= kStoredLse2Min && l2 <= kStoredLse2Max && y >= 0 && y < p.V;
}
__device__ __forceinline__ int stored_rows_of(const StoredParams& p) {
  const int nt = p.tiles ? *p.ntiles : p.R;
  return min(nt, p.pu_tiles) * 256;
}

__global__ void __launch_bounds__(kCompactBlock) stored_count_kernel(StoredParams p) {
  constexpr int kWarps = kCompactBlock / 32, kWarpsPerBlock = kStoredBlock / 32;
  __shared__ int is_last, kept_sum, first_mark;
  __shared__ unsigned any[kWarps];
  __shared__ int part[kCompactBlock];
  const int rows = stored_rows_of(p);
  const int j = blockIdx.x * kCompactBlock + threadIdx.x;   // every block of the launch takes part
  const bool keep = j < rows && stored_keep(p, stored_source(p, j));
  const unsigned bal = __ballot_sync(0xffffffffu, keep);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) any[w] = bal;
  __syncthreads();
  const int ngroups = rows / kGroup;
  const int grp = j / kGroup;
  if ((threadIdx.x & 31) == 0 && grp < ngroups) {
    unsigned a = 0;
    for (int k = 0; k < kWarpsPerBlock; ++k) a |= any[(w & ~(kWarpsPerBlock - 1)) + k];
    p.blk_cnt[grp] = (a ? 1 << 16 : 0) | __popc(bal);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    is_last = atomicAdd(p.ticket, 1u) == gridDim.x - 1;
    if (is_last) __threadfence();
    kept_sum = 0;
    first_mark = ngroups;
  }
  __syncthreads();
  if (!is_last) return;
  const int per = (ngroups + kCompactBlock - 1) / kCompactBlock;
  int s = 0, kc = 0;
  for (int k = 0; k < per; ++k) {
    const int i = threadIdx.x * per + k;
    if (i < ngroups) {
      const int v = __ldcg(p.blk_cnt + i);
      s += v >> 16;
      kc += v & 0xffff;
      if ((v >> 16) && i < first_mark) atomicMin(&first_mark, i);
    }
  }
  part[threadIdx.x] = s;
  if (kc) atomicAdd(&kept_sum, kc);
  __syncthreads();
  for (int o = 1; o < kCompactBlock; o <<= 1) {
    const int v = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int base = threadIdx.x ? part[threadIdx.x - 1] : 0;   // marked groups before
  for (int k = 0; k < per; ++k) {
    const int i = threadIdx.x * per + k;
    if (i < ngroups) {
      p.blk_off[i] = base * kGroup;
      base += __ldcg(p.blk_cnt + i) >> 16;
    }
  }
  const int total = part[kCompactBlock - 1] * kGroup;   // positions: a multiple of kStoredBlock
  if (threadIdx.x == 0) {
    *p.kept = kept_sum;
    *p.positions = total;
  }
  // positions past the taken blocks read the first taken block (finite
  // probabilities) against zero X rows and drop their dX rows
  const int fill = first_mark < ngroups ? first_mark * kGroup : 0;
  const int tail_end = min((total + 255) / 256 * 256, p.rows_cap);
  if (threadIdx.x == 0 && tail_end > total) p.rows[total / kStoredBlock] = fill;
  for (int r = total + threadIdx.x; r < tail_end; r += kCompactBlock) {
    p.idx[r] = -1;
    p.k2[r] = 0.f;
    p.err[r] = 0.f;
    p.tgt[r] = -1;
  }
  const int words = p.xs_ld / 8;
  const long long tail_words = (long long)(tail_end - total) * words;
  for (long long w2 = threadIdx.x; w2 < tail_words; w2 += kCompactBlock) {
    const long long r = total + w2 / words;
    reinterpret_cast<uint4*>(p.xs + r * p.xs_ld)[w2 % words] = make_uint4(0u, 0u, 0u, 0u);
  }
}

__global__ void __launch_bounds__(kCompactBlock) stored_gather_kernel(StoredParams p) {
  __shared__ int src_row[kGroup];
  __shared__ float scale[kGroup];
  const int g = blockIdx.x;
  const int rows = stored_rows_of(p);
  if (g * kGroup >= rows || !(p.blk_cnt[g] >> 16)) return;   // uniform over the block
  const int base = p.blk_off[g];
  if (threadIdx.x < kGroup) {
    const int j = g * kGroup + int(threadIdx.x);
    const int n = stored_source(p, j);
    const bool keep = stored_keep(p, n);
    const int pos = base + int(threadIdx.x);   // < positions <= stored rows <= rows_cap
    float k2 = 0.f, er = 0.f;
    long long y = -1;
    if (keep) {
      // G = (c/tau)(onehot - p) with p = pu 2^-lse2: off the target G = k2 pu,
      // at the target k1 = (c/tau)(1 - p_y), 1 - p_y = -expm1(logp).  fp32 (the
      // values feed bf16 entries and fp32 scales); err = k1 - k2 tv from one
      // fused multiply-add, exact but for its final rounding
      const float cf = p.coef[n];
      y = p.targets[n];
      k2 = -cf * exp2f(-p.lse2[n]);
      const float k1 = cf * -expm1f(float(p.logp64[n]));
      const __nv_bfloat16 tv = __float2bfloat16_rn(k1 / k2);
      er = fmaf(-k2, __bfloat162float(tv), k1);
      p.pu[size_t(j) * p.pu_ld + size_t(y)] = tv;
      p.done[n] = 1;
    }
    if (threadIdx.x == 0 && pos % kStoredBlock == 0) p.rows[pos / kStoredBlock] = j;
    p.idx[pos] = keep ? n : -1;
    p.k2[pos] = k2;
    p.err[pos] = er;
    p.tgt[pos] = y;
    src_row[threadIdx.x] = keep ? n : -1;
    scale[threadIdx.x] = k2;
  }
  __syncthreads();
  const int words = p.H / 8;          // 16-byte words of an X row
  const int owords = p.xs_ld / 8;     // of an xs row (one more with the db column)
  for (int w = int(threadIdx.x); w < kGroup * owords; w += kCompactBlock) {
    const int r = w / owords, c = w - r * owords;
    const int n = src_row[r];
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (n < 0) {
      // a row left out inside a taken block: zero X~ row (and db column)
    } else if (c < words) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(p.x + size_t(n) * p.H) + c);
      const float k2 = scale[r];
      const uint32_t in[4] = {u.x, u.y, u.z, u.w};
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&in[k]);
        const __nv_bfloat162 r2 = __floats2bfloat162_rn(k2 * __low2float(b2), k2 * __high2float(b2));
        o[k] = *reinterpret_cast<const uint32_t*>(&r2);
      }
      out = make_uint4(o[0], o[1], o[2], o[3]);
    } else if (c == words && p.xcol >= 0) {   // the db column: k2, zeros after it
      const __nv_bfloat162 k2p = __floats2bfloat162_rn(scale[r], 0.f);
      out.x = *reinterpret_cast<const uint32_t*>(&k2p);
    }
    reinterpret_cast<uint4*>(p.xs + size_t(base + r) * p.xs_ld)[c] = out;
  }
}

cudaError_t launch_stored_rows(const StoredParams& p, cudaStream_t st) {
  const int blocks = (p.rows_cap + kCompactBlock - 1) / kCompactBlock;
  stored_count_kernel<<<blocks > 0 ? blocks : 1, kCompactBlock, 0, st>>>(p);
  stored_gather_kernel<<<(p.rows_cap + kGroup - 1) / kGroup, kCompactBlock, 0, st>>>(p);
  return cudaGetLastError();
}

// Row counters of a call run in groups: acc[k] += *c[k] after each group, and
// *c[k] = acc[k] after the last (what the counter queries then report).
__global__ void counters_kernel(int* c0, int* c1, int* c2, int* c3, int* acc, int write_back) {
  if (threadIdx.x != 0) return;
  int* c[4] = {c0, c1, c2, c3};
  for (int k = 0; k < 4; ++k) {
    if (write_back)
      *c[k] = acc[k];
    else
      acc[k] += *c[k];
  }
}

cudaError_t launch_counters(int* const (&c)[4], int* acc, bool write_back, cudaStream_t st) {
  counters_kernel<<<1, 32, 0, st>>>(c[0], c[1], c[2], c[3], acc, write_back ? 1 : 0);
  return cudaGetLastError();
}

int compact_groups(int N) { return (N + kGroup - 1) / kGroup; }

cudaError_t launch_compact(const CompactParams& p, cudaStream_t st) {
  compact_count_kernel<<<(p.N + kCompactBlock - 1) / kCompactBlock, kCompactBlock, 0, st>>>(p);
  compact_gather_kernel<<<compact_groups(p.N), kCompactBlock, 0, st>>>(p);
  return cudaGetLastError();
}

// A chunk's X buffer: row j = X row idx[n0 + j] for the chunk's compacted rows
// (j < kept = clamp(*total - n0, 0, nc)), zero rows after them up to a whole
// 256-row tile (at most `rows`); nothing when the chunk keeps no row.
__global__ void __launch_bounds__(kCompactBlock) gather_chunk_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                                                         int Kx, const int* __restrict__ idx,
                                                                         const int* total, int n0, int nc, int rows,
                                                                         __nv_bfloat16* out) {
  const int kept = min(max(*total - n0, 0), nc);
  const int lim = min(rows, (kept + 255) / 256 * 256);   // the recompute reads whole 256-row tiles
  const int words = Kx / 8;   // 16-byte words per row
  const long long n = (long long)lim * words;
  for (long long w = blockIdx.x * (long long)blockDim.x + threadIdx.x; w < n; w += (long long)gridDim.x * blockDim.x) {
    const int j = int(w / words), c = int(w - (long long)j * words);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (j < kept) v = __ldg(reinterpret_cast<const uint4*>(x + size_t(idx[n0 + j]) * Kx) + c);
    reinterpret_cast<uint4*>(out + size_t(j) * Kx)[c] = v;
  }
}

cudaError_t launch_gather_chunk_rows(const __nv_bfloat16* x, int Kx, const int* idx, const int* total, int n0, int nc,
                                     int rows, __nv_bfloat16* out, cudaStream_t st) {
  // grid-stride over at most 512 blocks: the kept count is known only on the
  // device, and a chunk without kept rows then costs one short wave
  long long blocks = ((long long)rows * (Kx / 8) + kCompactBlock - 1) / kCompactBlock;
  if (blocks > 512) blocks = 512;
  if (blocks < 1) blocks = 1;
  gather_chunk_rows_kernel<<<int(blocks), kCompactBlock, 0, st>>>(x, Kx, idx, total, n0, nc, rows, out);
  return cudaGetLastError();
}

cudaError_t launch_set_total(int* total, int N, cudaStream_t st) {
  set_total_kernel<<<1, 1, 0, st>>>(total, N);
  return cudaGetLastError();
}

cudaError_t launch_scatter_rows(const float* src, const int* idx, const int* total, int n0, int nc_max, int H,
                                float* dst, bool accumulate, cudaStream_t st) {
  const long long n = (long long)nc_max * (H / 4);
  long long blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  scatter_rows_kernel<<<int(blocks), 256, 0, st>>>(reinterpret_cast<const float4*>(src), idx, total, n0, nc_max,
                                                   H / 4, reinterpret_cast<float4*>(dst), accumulate ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace rl
