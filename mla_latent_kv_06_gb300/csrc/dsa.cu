// dsa.cu -- DSA lightning-indexer scores and causal top-k key selection.
//
// The page "MLA 注意力与 KV 缓存", §2.2 "DSA lightning indexer": a light
// indexer scores every past key with a ReLU-gated, head-weighted sum, and the
// top-2048 causal keys are kept in dsa_sel for the attention (and reused by
// the shared layers).  The indexer keys Ic hold index_hd fp32 values per token
// (page "第 7 章 · 03 token 精确前向验证与 faithful DSA", §二).
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

// ---------------------------------------------------------------------------
// Index scores.  CTA = (token tile of kTile keys, s, b).  The key tile is
// staged in shared memory with coalesced loads; each thread then owns one key
// and half of the index heads.
// ---------------------------------------------------------------------------
constexpr int kIdxThreads = 256;
constexpr int kTile = 128;

__global__ void __launch_bounds__(kIdxThreads) index_scores_kernel(IndexArgs a) {
  const int tile = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int hd = a.hd, nh = a.n_ih;
  const int ld = hd + 1;  // padded row: thread i reads bank (i + d) % 32
  extern __shared__ float sm[];
  float* qs = sm;                     // [nh][hd]
  float* ws = qs + nh * hd;           // [nh]
  float* ks = ws + nh;                // [kTile][hd + 1]
  float* part = ks + kTile * ld;      // [2][kTile]

  const int Tb = a.T[b];
  const int t0 = tile * kTile;
  float* srow = a.scores + ((size_t)b * a.S + s) * a.T_cap;
  if (Tb < a.S || Tb > a.T_cap) {
    if (tid == 0 && tile == 0 && s == 0) raise_flag(a.flags, MLA_DEV_BAD_LENGTH);
    for (int i = tid; i < kTile; i += kIdxThreads)
      if (t0 + i < a.T_cap) srow[t0 + i] = qnan();
    return;
  }
  const int pos = Tb - a.S + s;
  if (t0 > pos) {  // whole tile is in the future of this query
    for (int i = tid; i < kTile; i += kIdxThreads)
      if (t0 + i < a.T_cap) srow[t0 + i] = -INFINITY;
    return;
  }
  const float* qsrc = a.q_idx + ((size_t)b * a.S + s) * nh * hd;
  for (int i = tid; i < nh * hd; i += kIdxThreads) qs[i] = qsrc[i];
  for (int i = tid; i < nh; i += kIdxThreads) ws[i] = a.w[((size_t)b * a.S + s) * nh + i];
  const float* Ic = a.Ic + (size_t)b * a.T_cap * hd;
  // Stage keys t0 .. t0+kTile-1 that are <= pos (others are zero; never read past pos).
  for (int e = tid; e < kTile * hd; e += kIdxThreads) {
    int i = e / hd, d = e - i * hd;
    int t = t0 + i;
    ks[i * ld + d] = (t <= pos) ? Ic[(size_t)t * hd + d] : 0.f;
  }
  __syncthreads();
  const int i = tid % kTile, grp = tid / kTile;  // two head groups
  float acc = 0.f;
  for (int h = grp; h < nh; h += 2) {
    const float* qh = qs + h * hd;
    const float* kr = ks + i * ld;
    float dot = 0.f;
    for (int d = 0; d < hd; ++d) dot = fmaf(qh[d], kr[d], dot);
    acc = fmaf(ws[h], fmaxf(dot, 0.f), acc);
  }
  part[grp * kTile + i] = acc;
  __syncthreads();
  if (tid < kTile) {
    int t = t0 + tid;
    if (t < a.T_cap) srow[t] = (t <= pos) ? part[tid] + part[kTile + tid] : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// Top-k.  One CTA per (b, s).  Radix select on 8-bit digits of the ordered
// key (most significant first) finds the k-th largest key K and how many keys
// equal to K must be kept; an index-ordered compaction then writes the kept
// keys in ascending order, taking equal keys from the lowest index up.
// ---------------------------------------------------------------------------
constexpr int kTopkThreads = 1024;

__device__ __forceinline__ int block_exclusive_scan(int v, int* red, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int nw = blockDim.x >> 5;
    int w = (lane < nw) ? red[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    red[lane] = w;  // inclusive prefix over warps
  }
  __syncthreads();
  int before = (warp > 0 ? red[warp - 1] : 0) + x - v;
  *total = red[(blockDim.x >> 5) - 1];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kTopkThreads) topk_select_kernel(TopkArgs a) {
  const int row = blockIdx.x;
  const int b = row / a.S, s = row - b * a.S;
  const int tid = threadIdx.x;
  const int k = a.topk;
  int32_t* sel = a.sel + (size_t)row * k;
  __shared__ int hist[256];
  __shared__ int red[32];
  __shared__ uint32_t sh_prefix;
  __shared__ int sh_remaining;

  const int Tb = a.T[b];
  if (Tb < a.S || Tb > a.T_cap) {
    if (tid == 0) {
      raise_flag(a.flags, MLA_DEV_BAD_LENGTH);
      a.nsel[row] = 0;
    }
    for (int j = tid; j < k; j += kTopkThreads) sel[j] = -1;
    return;
  }
  const int n = Tb - a.S + s + 1;
  if (n <= k) {  // keep all keys 0..pos
    for (int j = tid; j < k; j += kTopkThreads) sel[j] = (j < n) ? j : -1;
    if (tid == 0) a.nsel[row] = n;
    return;
  }
  const float* sc = a.scores + (size_t)row * a.T_cap;
  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int t = tid; t < n; t += kTopkThreads) {
      uint32_t key = ordered_key(sc[t]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int cum = 0, d = 255;
      for (; d > 0; --d) {
        if (cum + hist[d] >= remaining) break;
        cum += hist[d];
      }
      sh_prefix = prefix | ((uint32_t)d << shift);
      sh_remaining = remaining - cum;
    }
    __syncthreads();
    prefix = sh_prefix;
    remaining = sh_remaining;
    mask |= 255u << shift;
    __syncthreads();
  }
  // prefix = key of the k-th largest score; `remaining` keys equal to it are kept.
  const int seg = (n + kTopkThreads - 1) / kTopkThreads;
  const int ta = min(n, tid * seg), tb = min(n, ta + seg);
  int n_eq = 0;
  for (int t = ta; t < tb; ++t) n_eq += (ordered_key(sc[t]) == prefix);
  int tot;
  const int eq_before = block_exclusive_scan(n_eq, red, &tot);
  int n_sel = 0;
  {
    int eq_rank = eq_before;
    for (int t = ta; t < tb; ++t) {
      uint32_t key = ordered_key(sc[t]);
      if (key > prefix) ++n_sel;
      else if (key == prefix) n_sel += (eq_rank++ < remaining);
    }
  }
  const int out_before = block_exclusive_scan(n_sel, red, &tot);
  {
    int eq_rank = eq_before, o = out_before;
    for (int t = ta; t < tb; ++t) {
      uint32_t key = ordered_key(sc[t]);
      bool take = (key > prefix) || (key == prefix && eq_rank++ < remaining);
      if (take) sel[o++] = t;
    }
  }
  for (int j = tot + tid; j < k; j += kTopkThreads) sel[j] = -1;
  if (tid == 0) a.nsel[row] = tot;
}

}  // namespace

cudaError_t launch_index_scores(const IndexArgs& a, cudaStream_t st) {
  size_t smem = sizeof(float) * ((size_t)a.n_ih * a.hd + a.n_ih + (size_t)kTile * (a.hd + 1) + 2 * kTile);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(index_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((a.T_cap + kTile - 1) / kTile, a.S, a.B);
  index_scores_kernel<<<grid, kIdxThreads, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_topk_select(const TopkArgs& a, cudaStream_t st) {
  topk_select_kernel<<<a.B * a.S, kTopkThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
