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
// Index scores.  CTA = (128 keys, s, b), 256 threads.  The key tile (fp32,
// rows padded to 132 floats) and the query block sit in shared memory.  Warp
// w owns index heads 4w..4w+3 (broadcast reads); lane l owns keys l, l+32,
// l+64, l+96 (consecutive lanes hit consecutive rows: no bank conflicts), so
// every float4 of keys and of queries feeds 64 FMAs.  The eight head groups
// meet in shared memory and are summed in a fixed order.
// General head counts / widths fall back to a plain one-key-per-thread loop.
// ---------------------------------------------------------------------------
constexpr int kIdxThreads = 256;
constexpr int kTile = 128;
constexpr int kKPitch = 132;  // floats per staged key row

template <bool kFast>
__global__ void __launch_bounds__(kIdxThreads) index_scores_kernel(IndexArgs a) {
  const int tile = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hd = a.hd, nh = a.n_ih;
  extern __shared__ __align__(16) float sm[];
  float* qs = sm;                       // [nh][hd]
  float* ws = qs + nh * hd;             // [nh] (padded to 4)
  float* ks = ws + ((nh + 3) & ~3);     // [kTile][kKPitch]  (fast path) or [kTile][hd + 1]
  const int ld = kFast ? kKPitch : hd + 1;
  float* part = ks + kTile * ld;        // [8][kTile]

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
  const int nvalid = min(kTile, pos + 1 - t0);  // keys t0 .. t0+nvalid-1 are <= pos
  if (kFast) {
    // 128 rows x 32 float4; every load is issued before the first store
    float4 v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int e = tid + u * kIdxThreads, i = e >> 5, c4 = e & 31;
      v[u] = i < nvalid ? __ldg(reinterpret_cast<const float4*>(Ic + (size_t)(t0 + i) * 128) + c4)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int e = tid + u * kIdxThreads, i = e >> 5, c4 = e & 31;
      *reinterpret_cast<float4*>(ks + i * kKPitch + 4 * c4) = v[u];
    }
  } else {
    for (int e = tid; e < kTile * hd; e += kIdxThreads) {
      const int i = e / hd, d = e - i * hd;
      ks[i * ld + d] = i < nvalid ? Ic[(size_t)(t0 + i) * hd + d] : 0.f;
    }
  }
  __syncthreads();
  if (kFast) {
    // 32 index heads x 128 dims: warp w -> heads 4w..4w+3, lane -> keys lane + 32i
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    const float* q0 = qs + (4 * warp) * 128;
    const float* k0 = ks + lane * kKPitch;
#pragma unroll 4
    for (int d = 0; d < 128; d += 4) {
      float4 kv[4], qv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) kv[i] = *reinterpret_cast<const float4*>(k0 + 32 * i * kKPitch + d);
#pragma unroll
      for (int j = 0; j < 4; ++j) qv[j] = *reinterpret_cast<const float4*>(q0 + j * 128 + d);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float x = acc[i][j];
          x = fmaf(qv[j].x, kv[i].x, x);
          x = fmaf(qv[j].y, kv[i].y, x);
          x = fmaf(qv[j].z, kv[i].z, x);
          x = fmaf(qv[j].w, kv[i].w, x);
          acc[i][j] = x;
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float sc = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) sc = fmaf(ws[4 * warp + j], fmaxf(acc[i][j], 0.f), sc);
      part[warp * kTile + lane + 32 * i] = sc;
    }
    __syncthreads();
    if (tid < kTile) {
      float sc = 0.f;
#pragma unroll
      for (int w8 = 0; w8 < 8; ++w8) sc += part[w8 * kTile + tid];
      const int t = t0 + tid;
      if (t < a.T_cap) srow[t] = (t <= pos) ? sc : -INFINITY;
    }
  } else {
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
      const int t = t0 + tid;
      if (t < a.T_cap) srow[t] = (t <= pos) ? part[tid] + part[kTile + tid] : -INFINITY;
    }
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

constexpr int kCand = 16384;  // candidate keys of the threshold bin kept in shared memory

// Finds, among the keys k with (k & mask) == prefix, the digit d (of the
// `nbins` digits at `shift`) holding the remaining-th largest key.  hist[]
// holds the digit histogram.  Returns the new prefix; *remaining becomes the
// rank inside that digit.  Called by all threads; uses red[] for the scan.
__device__ __forceinline__ uint32_t pick_digit(const int* hist, int nbins, int shift, uint32_t prefix,
                                               int* remaining, int* red, uint32_t* sh_prefix, int* sh_rem) {
  // suffix counts from the top bin down: thread i owns bins nbins-1-2i and nbins-2-2i
  const int tid = threadIdx.x;
  const int per = nbins / kTopkThreads;  // 1 or 2
  int c = 0;
  for (int u = 0; u < per; ++u) c += hist[nbins - 1 - (tid * per + u)];
  int tot;
  const int before = block_exclusive_scan(c, red, &tot);  // keys in higher bins than my group
  const int need = *remaining;
  if (before < need && before + c >= need) {
    int cum = before;
    for (int u = 0; u < per; ++u) {
      const int bin = nbins - 1 - (tid * per + u);
      if (cum + hist[bin] >= need) {
        *sh_prefix = prefix | ((uint32_t)bin << shift);
        *sh_rem = need - cum;
        break;
      }
      cum += hist[bin];
    }
  }
  __syncthreads();
  *remaining = *sh_rem;
  const uint32_t np = *sh_prefix;
  __syncthreads();
  return np;
}

// Top-k.  One CTA per (b, s).  (1) histogram of the top 11 bits of the
// ordered keys (one pass over the scores); (2) the keys of the bin holding
// the k-th largest go to shared memory; (3) radix select of their low 21 bits
// there (11 + 10 bits) gives the exact k-th largest key K and how many keys
// equal to K are kept; (4) an index-ordered compaction writes the kept keys in
// ascending order, equal keys from the lowest index up.  A threshold bin with
// more than kCand keys falls back to 8-bit radix passes over global memory.
__global__ void __launch_bounds__(kTopkThreads) topk_select_kernel(TopkArgs a) {
  const int row = blockIdx.x;
  const int b = row / a.S, s = row - b * a.S;
  const int tid = threadIdx.x;
  const int k = a.topk;
  int32_t* sel = a.sel + (size_t)row * k;
  __shared__ int hist[2048];
  __shared__ int red[32];
  __shared__ uint32_t sh_prefix;
  __shared__ int sh_rem, sh_cnt;
  extern __shared__ uint32_t cand[];  // [kCand]

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
  int remaining = k;
  uint32_t prefix;
  // (1) top 11 bits
  for (int i = tid; i < 2048; i += kTopkThreads) hist[i] = 0;
  if (tid == 0) sh_cnt = 0;
  __syncthreads();
  for (int t = tid; t < n; t += kTopkThreads) atomicAdd(&hist[ordered_key(sc[t]) >> 21], 1);
  __syncthreads();
  prefix = pick_digit(hist, 2048, 21, 0u, &remaining, red, &sh_prefix, &sh_rem);
  // (2) candidates of that bin
  for (int t = tid; t < n; t += kTopkThreads) {
    const uint32_t key = ordered_key(sc[t]);
    if ((key >> 21) == (prefix >> 21)) {
      const int at = atomicAdd(&sh_cnt, 1);
      if (at < kCand) cand[at] = key;
    }
  }
  __syncthreads();
  const int ncand = sh_cnt;
  if (ncand <= kCand) {
    // (3) bits 20..10, then 9..0, on the candidates
    for (int i = tid; i < 2048; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < ncand; i += kTopkThreads) atomicAdd(&hist[(cand[i] >> 10) & 2047u], 1);
    __syncthreads();
    prefix = pick_digit(hist, 2048, 10, prefix, &remaining, red, &sh_prefix, &sh_rem);
    for (int i = tid; i < 1024; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < ncand; i += kTopkThreads)
      if ((cand[i] >> 10) == (prefix >> 10)) atomicAdd(&hist[cand[i] & 1023u], 1);
    __syncthreads();
    prefix = pick_digit(hist, 1024, 0, prefix, &remaining, red, &sh_prefix, &sh_rem);
  } else {
    // fallback: 8-bit digits 20..13, 12..5, 4..0 over global memory
    uint32_t mask = 0xFFE00000u;
    const int shifts[3] = {13, 5, 0}, widths[3] = {8, 8, 5};
    for (int pass = 0; pass < 3; ++pass) {
      const int sh = shifts[pass], nb = 1 << widths[pass];
      for (int i = tid; i < 2048; i += kTopkThreads) hist[i] = 0;
      __syncthreads();
      for (int t = tid; t < n; t += kTopkThreads) {
        const uint32_t key = ordered_key(sc[t]);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & (uint32_t)(nb - 1)], 1);
      }
      __syncthreads();
      if (tid == 0) {  // small histograms: serial scan from the top
        int cum = 0, d = nb - 1;
        for (; d > 0; --d) {
          if (cum + hist[d] >= remaining) break;
          cum += hist[d];
        }
        sh_prefix = prefix | ((uint32_t)d << sh);
        sh_rem = remaining - cum;
      }
      __syncthreads();
      prefix = sh_prefix;
      remaining = sh_rem;
      mask |= (uint32_t)(nb - 1) << sh;
      __syncthreads();
    }
  }
  // prefix = key of the k-th largest score; `remaining` keys equal to it are kept.
  // (4) ordered compaction over contiguous segments
  const int seg = (n + kTopkThreads - 1) / kTopkThreads;
  const int ta = min(n, tid * seg), tb = min(n, ta + seg);
  int n_eq = 0, n_gt = 0;
  for (int t = ta; t < tb; ++t) {
    const uint32_t key = ordered_key(sc[t]);
    n_eq += key == prefix;
    n_gt += key > prefix;
  }
  int tot;
  const int eq_before = block_exclusive_scan(n_eq, red, &tot);
  const int n_take_eq = max(0, min(n_eq, remaining - eq_before));
  const int out_before = block_exclusive_scan(n_gt + n_take_eq, red, &tot);
  {
    int eq_rank = eq_before, o = out_before;
    for (int t = ta; t < tb; ++t) {
      const uint32_t key = ordered_key(sc[t]);
      const bool take = (key > prefix) || (key == prefix && eq_rank++ < remaining);
      if (take) sel[o++] = t;
    }
  }
  for (int j = tot + tid; j < k; j += kTopkThreads) sel[j] = -1;
  if (tid == 0) a.nsel[row] = tot;
}


// ---------------------------------------------------------------------------
// Cluster top-k.  A cluster of kTkC CTAs (1024 threads each) handles one
// (b, s) row: thread t of cluster rank r holds the ordered keys of scores
// [(r*1024 + t)*per, +per) in registers, so the scores are read once.  Three
// radix passes (digits 31..21, 20..10, 9..0) each build a shared-memory
// histogram per CTA; every CTA then sums the kTkC histograms through
// distributed shared memory and picks the same digit.  The result is the key
// K of the k-th largest score and the number of keys equal to K to keep; an
// index-ordered compaction (CTA totals exchanged the same way) writes the
// kept indices in ascending order, equal keys from the lowest index up.
// ---------------------------------------------------------------------------
constexpr int kTkC = 8;          // CTAs per row (portable cluster size)
constexpr int kTkMaxPer = 16;    // keys per thread held in registers

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Read an int from the shared memory of CTA `rank` of this cluster, at the
// address that `p` has in this CTA.
__device__ __forceinline__ int ld_cluster_int(const int* p, uint32_t rank) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  int v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
  return v;
}

// Adds 1 to hist[bin] for every lane with active != 0, one atomic per
// distinct bin in the warp (the integer-valued scores crowd a few bins).
__device__ __forceinline__ void warp_hist_add(int* hist, uint32_t bin, bool active) {
  const unsigned am = __ballot_sync(0xffffffffu, active);
  if (!active) return;
  const unsigned peers = __match_any_sync(am, bin);
  const int leader = __ffs(peers) - 1;
  if ((int)(threadIdx.x & 31) == leader) atomicAdd(&hist[bin], __popc(peers));
}

// Global histogram of one pass: the kTkC per-CTA histograms summed into
// tot[] (bins split over the threads).  Bracketed by cluster barriers: local
// histograms complete before, tot[] ready after.
__device__ __forceinline__ void cluster_hist_sum(const int* local, int* tot, int nbins) {
  cluster_sync_all();
  for (int i = threadIdx.x; i < nbins; i += kTopkThreads) {
    int v = 0;
#pragma unroll
    for (int c = 0; c < kTkC; ++c) v += ld_cluster_int(local + i, (uint32_t)c);
    tot[i] = v;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kTopkThreads) topk_cluster_kernel(TopkArgs a, int per) {
  const uint32_t rank = cluster_rank();
  const int row = blockIdx.x / kTkC;
  const int b = row / a.S, s = row - b * a.S;
  const int tid = threadIdx.x;
  const int k = a.topk;
  int32_t* sel = a.sel + (size_t)row * k;
  __shared__ int hist[3][2048];  // this CTA's histogram of each pass (read by the cluster)
  __shared__ int tot[2048];      // the pass's cluster-wide histogram
  __shared__ int red[32];
  __shared__ uint32_t sh_prefix;
  __shared__ int sh_rem;
  __shared__ int cta_cnt[2];     // this CTA's keys > K and keys == K (read by the cluster)

  grid_dep_wait();  // scores (and histograms) come from the indexer
  const int Tb = a.T[b];
  // Rows that need no selection: every CTA of the cluster takes the same branch.
  if (Tb < a.S || Tb > a.T_cap) {
    if (rank == 0) {
      if (tid == 0) {
        raise_flag(a.flags, MLA_DEV_BAD_LENGTH);
        a.nsel[row] = 0;
      }
      for (int j = tid; j < k; j += kTopkThreads) sel[j] = -1;
    }
    return;
  }
  const int n = Tb - a.S + s + 1;
  if (n <= k) {  // keep all keys 0..pos
    if (rank == 0) {
      for (int j = tid; j < k; j += kTopkThreads) sel[j] = (j < n) ? j : -1;
      if (tid == 0) a.nsel[row] = n;
    }
    return;
  }
  const float* sc = a.scores + (size_t)row * a.T_cap;
  const int base = ((int)rank * kTopkThreads + tid) * per;
  uint32_t key[kTkMaxPer];
#pragma unroll
  for (int i = 0; i < kTkMaxPer; ++i) key[i] = (i < per && base + i < n) ? ordered_key(sc[base + i]) : 0u;
  for (int i = tid; i < 3 * 2048; i += kTopkThreads) (&hist[0][0])[i] = 0;
  __syncthreads();

  // pass 1: bits 31..21
  if (a.hpart) {
    // The indexer's per-CTA histograms of this row: CTA `rank` sums bins
    // 256*rank .. 256*rank+255 over them, the cluster gathers the slices.
    const uint32_t* hp = a.hpart + (size_t)row * a.hparts * 2048 + 256 * rank;
    // kTopkThreads / 256 threads per bin, each summing every such part with
    // its loads in flight together; the sums meet in shared memory.
    constexpr int kPerBin = kTopkThreads / 256;
    static_assert(kTopkThreads % 256 == 0, "whole bins per thread group");
    const int bin = tid & 255, grp = tid >> 8;
    int v = 0;
#pragma unroll 8
    for (int c = grp; c < a.hparts; c += kPerBin) v += (int)__ldg(hp + (size_t)c * 2048 + bin);
    atomicAdd(&hist[0][256 * rank + bin], v);
    cluster_sync_all();
    for (int i = tid; i < 2048; i += kTopkThreads) tot[i] = ld_cluster_int(&hist[0][i], (uint32_t)(i >> 8));
    __syncthreads();
  } else {
#pragma unroll
    for (int i = 0; i < kTkMaxPer; ++i)
      if (i < per) warp_hist_add(hist[0], key[i] >> 21, base + i < n);
    cluster_hist_sum(hist[0], tot, 2048);
  }
  int remaining = k;
  uint32_t prefix = pick_digit(tot, 2048, 21, 0u, &remaining, red, &sh_prefix, &sh_rem);
  // pass 2: bits 20..10 of the keys in the chosen bin
#pragma unroll
  for (int i = 0; i < kTkMaxPer; ++i)
    if (i < per) warp_hist_add(hist[1], (key[i] >> 10) & 2047u, base + i < n && (key[i] >> 21) == (prefix >> 21));
  cluster_hist_sum(hist[1], tot, 2048);
  prefix = pick_digit(tot, 2048, 10, prefix, &remaining, red, &sh_prefix, &sh_rem);
  // pass 3: bits 9..0
#pragma unroll
  for (int i = 0; i < kTkMaxPer; ++i)
    if (i < per) warp_hist_add(hist[2], key[i] & 1023u, base + i < n && (key[i] >> 10) == (prefix >> 10));
  cluster_hist_sum(hist[2], tot, 1024);
  prefix = pick_digit(tot, 1024, 0, prefix, &remaining, red, &sh_prefix, &sh_rem);
  // prefix = key K of the k-th largest score; `remaining` keys equal to K are kept.

  int n_gt = 0, n_eq = 0;
#pragma unroll
  for (int i = 0; i < kTkMaxPer; ++i)
    if (i < per && base + i < n) {
      n_gt += key[i] > prefix;
      n_eq += key[i] == prefix;
    }
  int cta_eq, cta_gt;
  const int eq_before_cta = block_exclusive_scan(n_eq, red, &cta_eq);
  const int gt_before_cta = block_exclusive_scan(n_gt, red, &cta_gt);
  if (tid == 0) {
    cta_cnt[0] = cta_gt;
    cta_cnt[1] = cta_eq;
  }
  cluster_sync_all();
  // keys kept by the lower-ranked CTAs
  int eq_lower = 0, out_lower = 0;
  for (uint32_t c = 0; c < rank; ++c) {
    const int g_c = ld_cluster_int(&cta_cnt[0], c), e_c = ld_cluster_int(&cta_cnt[1], c);
    out_lower += g_c + max(0, min(e_c, remaining - eq_lower));
    eq_lower += e_c;
  }
  const int eq_before = eq_lower + eq_before_cta;
  // equal keys kept before this thread's segment, inside this CTA
  const int take_before_cta = max(0, min(eq_before_cta, remaining - eq_lower));
  int o = out_lower + gt_before_cta + take_before_cta;
  int eq_rank = eq_before;
#pragma unroll
  for (int i = 0; i < kTkMaxPer; ++i)
    if (i < per && base + i < n) {
      const bool take = (key[i] > prefix) || (key[i] == prefix && eq_rank++ < remaining);
      if (take) sel[o++] = base + i;
    }
  if (rank == 0 && tid == 0) a.nsel[row] = k;
  cluster_sync_all();  // no CTA leaves while another may still read its shared memory
}

}  // namespace

cudaError_t launch_index_scores(const IndexArgs& a, cudaStream_t st) {
  // 32 heads x 128: the tensor-core kernel (index_tc.cu); other shapes stay on the CUDA cores
  const cudaError_t tc = launch_index_scores_tc(a, st);
  if (tc != cudaErrorNotSupported) return tc;
  const bool fast = a.n_ih == 32 && a.hd == 128;
  const int ld = fast ? kKPitch : a.hd + 1;
  size_t smem = sizeof(float) * ((size_t)a.n_ih * a.hd + ((a.n_ih + 3) & ~3) + (size_t)kTile * ld + 8 * kTile);
  auto kern = fast ? index_scores_kernel<true> : index_scores_kernel<false>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((a.T_cap + kTile - 1) / kTile, a.S, a.B);
  kern<<<grid, kIdxThreads, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_topk_select(const TopkArgs& a, cudaStream_t st) {
  // Rows up to kTkC * 1024 * kTkMaxPer keys: one cluster per row, keys in registers.
  const long long per = ((long long)a.T_cap + kTkC * kTopkThreads - 1) / (kTkC * kTopkThreads);
  if (per <= kTkMaxPer) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.B * a.S * kTkC);
    cfg.blockDim = dim3(kTopkThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kTkC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, topk_cluster_kernel, a, (int)(per < 1 ? 1 : per));
    if (e == cudaSuccess) return cudaSuccess;
    (void)cudaGetLastError();  // clusters unavailable: single-CTA kernel below
  }
  const int smem = kCand * 4;
  cudaError_t e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  topk_select_kernel<<<a.B * a.S, kTopkThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
