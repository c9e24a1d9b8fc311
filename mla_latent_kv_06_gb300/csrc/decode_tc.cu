// decode_tc.cu -- tensor-core weight-absorbed decode (dense and DSA-sparse)
// for the GLM-5.2 head geometry (64 heads, 512-wide latent, 64-wide rope key).
//
// The method is the absorbed path of the page "MLA 注意力与 KV 缓存", §2.3:
// fold W_UK into the query (qabs), score straight on the latent cache Lc plus
// the shared rotated key Rc, softmax, form the latent context clat, lift it
// with W_UV; and §2.2 for the sparse variant, where each query attends only to
// the keys its DSA selection kept.
//
// Three kernels, chained with programmatic dependent launch:
//  1. absorb   : qcat[r,h,:] = [qabs (512) | RoPE(q_rope) (64)] in bf16, one
//                read of W_UK; block (0,0) also lays out the tile plan.
//  2. attention: persistent, one CTA per SM, split-K over 128-key tiles.
//                Transposed products so that the 128 keys fill the M=128
//                tcgen05 rows and the 64 heads are N:
//                  S^T[128 keys x 64 heads]  = [Lc|Rc] tile (smem, K-major) x qcat^T
//                  O^T[512 latent x 64 heads] += Lc^T (smem, MN-major) x P^T (smem, MN-major)
//                Warp 0 streams the tile's nine 64-column atoms with TMA,
//                warp 1 issues the MMAs,
//                warps 2-5 run the online softmax (one key per thread) and
//                write the per-split (m, l, O) partials.
//  3. combine  : log-sum-exp merge of the splits, then out = W_UV clat / l.
// The sparse variant first gathers each query's selected [Lc | Rc] rows into
// a contiguous staging buffer (row-major, 576 values per key, zero past nsel),
// so that its attention pass uses the same 1024-byte-aligned tile loads.
#include <atomic>
#include <cmath>

#include "decode_tc.h"
#include "gemm_tc.h"
#include "sm100.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace sm100;

constexpr int kH = 64, kDl = 512, kDr = 64, kDc = 576;  // kDc = kv_lora + qk_rope
constexpr int kTile = 128;
constexpr int kSlots = 9;                      // 8 latent atoms + 1 rope atom per key tile
constexpr uint32_t kSlotBytes = 16384;         // 128 keys x 64 bf16
constexpr uint32_t kQAtomBytes = 8192;         // 64 heads x 64 bf16
constexpr uint32_t kQBytes = 9 * kQAtomBytes;  // 73728
constexpr uint32_t kKVBytes = 9 * kSlotBytes;  // 147456
constexpr uint32_t kAttnDynSmem = kQBytes + kKVBytes + 1024;
constexpr int kAttnThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;    // S^T: 64 columns
constexpr uint32_t kTmemO = 128;  // O^T: 4 M-tiles x 64 columns
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTau = 8.f;  // lazy rescale threshold (log2 units)
constexpr int kPlanMax = 1024;
constexpr int kPrefetchTiles = 2;  // key tiles pulled into L2 ahead of the tile loads  // tile-list rows whose plan the attention CTA builds itself
// Waits that drain in-flight copies / MMAs before a CTA exits use at least
// this limit, whatever the caller's wait limit.
constexpr long long kDrainNs = 1000000000LL;

struct AttnParams {
  CUtensorMap mQ;  // qcat [R*64, 576]
  CUtensorMap mL;  // latent rows: Lc [B*T_cap, 512] (dense) or staging [R*Kpad, 576] cols 0..511
  CUtensorMap mR;  // rope rows:   Rc [B*T_cap, 64]  (dense) or staging cols 512..575
  const int32_t* T;
  const int32_t* sel;
  const int32_t* nsel;
  const int32_t* tile_start;  // [NR + 1]
  int B, S, T_cap, G, topk;
  int kv_rows;  // rows of the key source per tile-list row: T_cap (dense) or Kpad (sparse)
  float c;  // softmax scale * log2(e)
  float* o_part;
  float* ml_part;
  unsigned int* flags;
  long long wait_ns;
};

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ bool bar_red_or(int id, int n, bool x) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)x), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Reduce 64 per-lane values over the 32 lanes of a warp; afterwards lane L
// holds the results for entries 2L and 2L+1 in v[0], v[1].
template <bool kMax>
__device__ __forceinline__ void transpose_reduce64(float (&v)[64], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int o = 16 >> step;
    const int half = 32 >> step;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&t);
}

// Chunk g of the flattened tile list covers tiles [N*g/G, N*(g+1)/G).
__device__ __forceinline__ long long chunk_begin(long long N, int g, int G) { return (N * g) / G; }

__device__ __forceinline__ int chunk_of(long long x, long long N, int G) {
  int g = (int)((x * G) / N);
  if (g > G - 1) g = G - 1;
  while (g + 1 < G && chunk_begin(N, g + 1, G) <= x) ++g;
  while (g > 0 && chunk_begin(N, g, G) > x) --g;
  return g;
}

// Tiles of row `row` that chunk g processes for query position s: [lo, hi).
template <bool kSparse>
__device__ __forceinline__ void piece_range(const int32_t* ts, const int32_t* T, int S, int s, int row, int g,
                                            int G, long long N, int* lo, int* hi) {
  const long long a = ts[row], e = ts[row + 1];
  const long long c0 = chunk_begin(N, g, G), c1 = chunk_begin(N, g + 1, G);
  long long l = (a > c0 ? a : c0) - a, h = (e < c1 ? e : c1) - a;
  if (!kSparse && h > l) {
    const int pos = T[row] - S + s;
    const long long vt = (pos + kTile) / kTile;  // tiles holding keys 0..pos
    if (h > vt) h = vt;
  }
  *lo = (int)l;
  *hi = (int)(h > l ? h : l);
}

// Next row >= *row holding a non-empty piece for chunk g; false when none.
template <bool kSparse>
__device__ __forceinline__ bool next_piece(const AttnParams& p, const int32_t* ts, int NR, long long N, int g,
                                           int s, int* row, int* lo, int* hi) {
  const long long c1 = chunk_begin(N, g + 1, p.G);
  for (; *row < NR; ++*row) {
    if (ts[*row] >= c1) return false;
    piece_range<kSparse>(ts, p.T, p.S, s, *row, g, p.G, N, lo, hi);
    if (*lo < *hi) return true;
  }
  return false;
}

// Tiles of a tile-list row (0 for a row the absorb kernel flags as bad).
template <bool kSparse>
__device__ __forceinline__ int row_tiles(const AttnParams& p, int row) {
  const int b = kSparse ? row / p.S : row;
  const int Tb = p.T[b];
  if (Tb < p.S || Tb > p.T_cap) return 0;
  int nk = Tb;
  if (kSparse) {
    nk = p.nsel[row];
    if (nk < 1 || nk > p.topk) return 0;
  }
  return (nk + kTile - 1) / kTile;
}

// First row whose tiles reach past the chunk start.
__device__ __forceinline__ int first_row(const int32_t* ts, int NR, long long c0) {
  int lo = 0, hi = NR;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (ts[mid + 1] > c0) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}

// ===========================================================================
// Attention kernel
// ===========================================================================
template <bool kSparse>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  unsigned char* sQ = smem;
  unsigned char* sKV = smem + kQBytes;

  __shared__ uint64_t full_bar[kSlots], empty_bar[kSlots];
  __shared__ uint64_t q_full, q_empty, s_full, s_free, p_full, o_done, o_free, mma_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ __align__(16) float red_max[4][kH];
  __shared__ __align__(16) float red_sum[4][kH];
  __shared__ __align__(16) float m_sh[kH];
  __shared__ __align__(16) float alpha_sh[kH];
  __shared__ int plan_ts[kPlanMax + 1];
  __shared__ int plan_wsum[kAttnThreads / 32];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.S;
  const int g = kSparse ? (int)blockIdx.x : (int)blockIdx.x / S;
  const int s = kSparse ? 0 : (int)blockIdx.x % S;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    mbar_init(&q_full, 1);
    mbar_init(&q_empty, 1);
    mbar_init(&s_full, 1);
    mbar_init(&s_free, 128);
    mbar_init(&p_full, 128);
    mbar_init(&o_done, 1);
    mbar_init(&o_free, 128);
    mbar_init(&mma_done, 1);
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&p.mQ);
    prefetch_tensormap(&p.mL);
    prefetch_tensormap(&p.mR);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  volatile int* abort = &abort_flag;

  // The combine kernel may start now: it only prefetches W_UV before waiting
  // for this grid to finish.
  grid_dep_launch();

  // Tile plan.  Built here from T / nsel (kernel inputs, ready at launch)
  // so that the key tiles can stream in while the absorb kernel still runs;
  // only the qcat loads wait for it.  Very long batches use the absorb
  // kernel's copy of the same plan.
  const int NR = kSparse ? p.B * S : p.B;
  const bool local_plan = NR <= kPlanMax;
  const int32_t* ts = p.tile_start;
  if (local_plan) {
    int carry = 0;
    for (int base = 0; base < NR; base += kAttnThreads) {
      const int r = base + threadIdx.x;
      int x = r < NR ? row_tiles<kSparse>(p, r) : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) plan_wsum[warp] = x;
      __syncthreads();
      int off = carry;
      for (int i = 0; i < warp; ++i) off += plan_wsum[i];
      if (r < NR) plan_ts[r + 1] = off + x;
      int tot = 0;
      for (int i = 0; i < kAttnThreads / 32; ++i) tot += plan_wsum[i];
      carry += tot;
      __syncthreads();
    }
    if (threadIdx.x == 0) plan_ts[0] = 0;
    __syncthreads();
    ts = plan_ts;
  } else {
    grid_dep_wait();
  }
  const long long N = ts[NR];
  const long long c0 = chunk_begin(N, g, p.G);
  const int row0 = first_row(ts, NR, c0);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int it = 0, pc = 0, row = row0, lo, hi;
    bool ok = true;
    int last_it[kSlots];
    for (int a = 0; a < kSlots; ++a) last_it[a] = -1;
    int last_q = -1;
    bool waited = !local_plan;
    // L2 prefetch cursor, kPrefetchTiles key tiles ahead of the tile loads:
    // HBM keeps streaming while a tile's score product, softmax and value
    // product run, and the tile loads then hit L2.
    int pf_row = row0, pf_lo = 0, pf_hi = 0, pf_k = 0;
    bool pf_live = true;
    auto prefetch_next = [&]() {
      if (!pf_live) return;
      if (pf_k >= pf_hi) {
        if (pf_hi > 0) ++pf_row;
        if (!next_piece<kSparse>(p, ts, NR, N, g, s, &pf_row, &pf_lo, &pf_hi)) {
          pf_live = false;
          return;
        }
        pf_k = pf_lo;
      }
      const int y = (kSparse ? pf_row : pf_row) * p.kv_rows + pf_k * kTile;
      for (int a = 0; a < 8; ++a) tma_prefetch_l2_2d(&p.mL, 64 * a, y);
      tma_prefetch_l2_2d(&p.mR, 0, y);
      ++pf_k;
    };
    if (lane == 0)
      for (int i = 0; i <= kPrefetchTiles; ++i) prefetch_next();
    while (ok && next_piece<kSparse>(p, ts, NR, N, g, s, &row, &lo, &hi)) {
      const int qrow = kSparse ? row : row * S + s;
      const int b = kSparse ? row / S : row;
      const int kvrow = kSparse ? row : b;
      for (int k = lo; ok && k < hi; ++k, ++it) {
        const uint32_t par = (it & 1) ^ 1;
        if (lane == 0 && it > 0) prefetch_next();
        if (lane == 0) {
          const int y = kvrow * p.kv_rows + k * kTile;
          for (int a = 0; a < kSlots && ok; ++a) {
            ok = mbar_wait(&empty_bar[a], par, abort, p.flags, p.wait_ns);
            if (!ok) break;
            mbar_arrive_expect_tx(&full_bar[a], kSlotBytes);
            if (a < 8) tma_load_2d(sKV + a * kSlotBytes, &p.mL, 64 * a, y, &full_bar[a]);
            else tma_load_2d(sKV + a * kSlotBytes, &p.mR, 0, y, &full_bar[a]);
            last_it[a] = it;
          }
          if (ok && k == lo) {  // the piece's query block, once its first key tile is on its way
            if (!waited) {
              grid_dep_wait();  // qcat comes from the absorb kernel
              waited = true;
            }
            ok = mbar_wait(&q_empty, (pc & 1) ^ 1, abort, p.flags, p.wait_ns);
            if (ok) {
              mbar_arrive_expect_tx(&q_full, kQBytes);
              for (int a = 0; a < kSlots; ++a) tma_load_2d(sQ + a * kQAtomBytes, &p.mQ, 64 * a, qrow * kH, &q_full);
              last_q = pc;
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      ++pc;
      ++row;
    }
    // Never leave with copies in flight: wait for the last load of each slot.
    if (lane == 0) {
      volatile int no_abort = 0;
      const long long drain_ns = p.wait_ns > kDrainNs ? p.wait_ns : kDrainNs;
      for (int a = 0; a < kSlots; ++a)
        if (last_it[a] >= 0) mbar_wait(&full_bar[a], last_it[a] & 1, &no_abort, p.flags, drain_ns);
      if (last_q >= 0) mbar_wait(&q_full, last_q & 1, &no_abort, p.flags, drain_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc1 = idesc_bf16_f32(128, 64, 0, 0);
      const uint32_t idesc2 = idesc_bf16_f32(128, 64, 1, 1);
      const uint32_t kv0 = smem_u32(sKV), q0 = smem_u32(sQ);
      int it = 0, pc = 0, row = row0, lo, hi;
      bool ok = true, issued = false;
      while (ok && next_piece<kSparse>(p, ts, NR, N, g, s, &row, &lo, &hi)) {
        ok = mbar_wait(&q_full, pc & 1, abort, p.flags, p.wait_ns);
        if (ok && pc > 0) ok = mbar_wait(&o_free, (pc - 1) & 1, abort, p.flags, p.wait_ns);
        for (int k = lo; ok && k < hi; ++k, ++it) {
          ok = mbar_wait(&s_free, (it & 1) ^ 1, abort, p.flags, p.wait_ns);
          if (!ok) break;
          tc_fence_after();
          for (int a = 0; a < kSlots && ok; ++a) {
            ok = mbar_wait(&full_bar[a], it & 1, abort, p.flags, p.wait_ns);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t da = smem_desc_sw128(kv0 + a * kSlotBytes + kk * 32, 16, 1024);
              const uint64_t db = smem_desc_sw128(q0 + a * kQAtomBytes + kk * 32, 16, 1024);
              mma_bf16(tmem + kTmemS, da, db, idesc1, (a | kk) != 0);
            }
            issued = true;
          }
          if (!ok) break;
          mma_commit(&s_full);
          if (k == hi - 1) mma_commit(&q_empty);
          ok = mbar_wait(&p_full, it & 1, abort, p.flags, p.wait_ns);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int m = 0; m < 4; ++m) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t da = smem_desc_sw128(kv0 + (2 * m) * kSlotBytes + kk * 2048, kSlotBytes, 1024);
              const uint64_t db = smem_desc_sw128(kv0 + 8 * kSlotBytes + kk * 2048, kSlotBytes, 1024);
              mma_bf16(tmem + kTmemO + 64 * m, da, db, idesc2, (kk > 0 || k > lo) ? 1u : 0u);
            }
            mma_commit(&empty_bar[2 * m]);
            mma_commit(&empty_bar[2 * m + 1]);
          }
          mma_commit(&empty_bar[8]);
          mma_commit(&o_done);
        }
        ++pc;
        ++row;
      }
      if (issued) {  // all MMAs retired before TMEM is released
        mma_commit(&mma_done);
        volatile int no_abort = 0;
        mbar_wait(&mma_done, 0, &no_abort, p.flags, p.wait_ns > kDrainNs ? p.wait_ns : kDrainNs);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps 2..5
    const int tr = threadIdx.x - 64;                 // 0..127
    const int wq = warp & 3;                         // TMEM lane quadrant of this warp
    const int trow = 32 * wq + lane;                 // key row of the tile / latent row of O^T
    const int widx = warp - 2;
    const uint32_t t_lane = (uint32_t)(32 * wq) << 16;
    const float c = p.c;
    int it = 0, pc = 0, row = row0, lo, hi;
    bool ok = true;
    while (ok && next_piece<kSparse>(p, ts, NR, N, g, s, &row, &lo, &hi)) {
      const int b = kSparse ? row / S : row;
      const int qs = kSparse ? row % S : s;
      const int pos = p.T[b] - S + qs;
      const int nkeys = kSparse ? p.nsel[row] : pos + 1;
      const int32_t* srow = kSparse ? p.sel + (size_t)row * p.topk : nullptr;
      float lp[kH];
#pragma unroll
      for (int h = 0; h < kH; ++h) lp[h] = 0.f;
      bool bad_idx = false;
      for (int k = lo; ok && k < hi; ++k, ++it) {
        const bool first = (k == lo);
        // A failed wait is decided jointly by the 128 softmax threads (bar.red
        // below), so that no thread is left waiting at a barrier the others quit.
        bool fail = !mbar_wait(&s_full, it & 1, abort, p.flags, p.wait_ns);
        if (bar_red_or(1, 128, fail)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float v[kH];
        tmem_ld64(tmem + t_lane + kTmemS, v);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&s_free);
        const int j = k * kTile + trow;
        bool valid = j < nkeys;
        if (kSparse && valid) {
          const int idx = srow[j];
          if (idx < 0 || idx > pos) {
            valid = false;
            bad_idx = true;
          }
        }
        if (!valid) {
#pragma unroll
          for (int h = 0; h < kH; ++h) v[h] = -INFINITY;
        }
        float mx[kH];
#pragma unroll
        for (int h = 0; h < kH; ++h) mx[h] = v[h];
        transpose_reduce64<true>(mx, lane);
        *reinterpret_cast<float2*>(&red_max[widx][2 * lane]) = make_float2(mx[0], mx[1]);
        named_barrier(1, 128);
        bool need = false;
        if (tr < kH) {
          const float tmax = fmaxf(fmaxf(red_max[0][tr], red_max[1][tr]), fmaxf(red_max[2][tr], red_max[3][tr]));
          const float cand = tmax * c;
          const float mo = first ? -INFINITY : m_sh[tr];
          float mn = mo, al = 1.f;
          if (cand > mo + kTau) {
            mn = cand;
            al = exp2f(mo - mn);
          }
          m_sh[tr] = mn;
          alpha_sh[tr] = al;
          need = !first && al != 1.f;
        }
        const bool rescale = bar_red_or(2, 128, need);
        // probabilities, row sums, P^T row into the rope slot (free after the score MMAs)
        uint32_t pk[kH / 2];
#pragma unroll
        for (int h2 = 0; h2 < kH; h2 += 4) {
          const float4 mu = *reinterpret_cast<const float4*>(&m_sh[h2]);
          const float e0 = exp2f(fmaf(v[h2 + 0], c, -mu.x));
          const float e1 = exp2f(fmaf(v[h2 + 1], c, -mu.y));
          const float e2 = exp2f(fmaf(v[h2 + 2], c, -mu.z));
          const float e3 = exp2f(fmaf(v[h2 + 3], c, -mu.w));
          pk[h2 / 2] = pack_bf16(e0, e1);
          pk[h2 / 2 + 1] = pack_bf16(e2, e3);
        }
        if (rescale || first) {
#pragma unroll
          for (int h2 = 0; h2 < kH; h2 += 4) {
            const float4 al = *reinterpret_cast<const float4*>(&alpha_sh[h2]);
            lp[h2 + 0] *= al.x;
            lp[h2 + 1] *= al.y;
            lp[h2 + 2] *= al.z;
            lp[h2 + 3] *= al.w;
          }
        }
#pragma unroll
        for (int i = 0; i < kH / 2; ++i) {
          __nv_bfloat162 t = *reinterpret_cast<__nv_bfloat162*>(&pk[i]);
          const float2 f = __bfloat1622float2(t);
          lp[2 * i] += f.x;
          lp[2 * i + 1] += f.y;
        }
        unsigned char* prow = sKV + 8 * kSlotBytes + trow * 128;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint4 val = make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
          *reinterpret_cast<uint4*>(prow + ((cc ^ (trow & 7)) << 4)) = val;
        }
        if (!valid) {  // masked key: its latent row must be finite for the value product
#pragma unroll
          for (int a = 0; a < 8; ++a) {
            unsigned char* lr = sKV + a * kSlotBytes + trow * 128;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) *reinterpret_cast<uint4*>(lr + 16 * cc) = make_uint4(0, 0, 0, 0);
          }
        }
        if (rescale) {  // O^T columns scaled by alpha once the previous value product retired
          fail = !mbar_wait(&o_done, (it - 1) & 1, abort, p.flags, p.wait_ns);
          if (bar_red_or(2, 128, fail)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int m = 0; m < 4; ++m) {
            float w[kH];
            tmem_ld64(tmem + t_lane + kTmemO + 64 * m, w);
            tmem_wait_ld();
#pragma unroll
            for (int h2 = 0; h2 < kH; h2 += 4) {
              const float4 al = *reinterpret_cast<const float4*>(&alpha_sh[h2]);
              w[h2] *= al.x;
              w[h2 + 1] *= al.y;
              w[h2 + 2] *= al.z;
              w[h2 + 3] *= al.w;
            }
            tmem_st64(tmem + t_lane + kTmemO + 64 * m, w);
          }
          tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full);
      }
      if (!ok) break;
      // ---- end of piece: write the split's partials
      const int slot = kSparse ? g + row : (g + row) * S + s;
      const bool fail_end = !mbar_wait(&o_done, (it - 1) & 1, abort, p.flags, p.wait_ns);
      if (bar_red_or(1, 128, fail_end)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float* op = p.o_part + (size_t)slot * kH * kDl;
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
        float w[kH];
        tmem_ld64(tmem + t_lane + kTmemO + 64 * m, w);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < kH; ++h) op[(size_t)h * kDl + 128 * m + trow] = w[h];
      }
      tc_fence_before();
      mbar_arrive(&o_free);
      transpose_reduce64<false>(lp, lane);
      *reinterpret_cast<float2*>(&red_sum[widx][2 * lane]) = make_float2(lp[0], lp[1]);
      const bool bad = bar_red_or(1, 128, bad_idx);
      if (tr < kH) {
        const float l = red_sum[0][tr] + red_sum[1][tr] + red_sum[2][tr] + red_sum[3][tr];
        float* ml = p.ml_part + ((size_t)slot * kH + tr) * 2;
        ml[0] = m_sh[tr];
        ml[1] = bad ? __int_as_float(0x7fc00000) : l;
      }
      if (bad && tr == 0) raise_flag(p.flags, MLA_DEV_BAD_INDEX);
      ++pc;
      ++row;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ===========================================================================
// Absorb kernel: qcat[r,h,0:512] = sum_i q_nope[r,h,i] W_UK[h,i,:] (bf16),
// qcat[r,h,512:576] = RoPE(q_rope[r,h], pos_r) (bf16).  Block (0,0) first
// validates the lengths / selections and writes the tile plan.
// ===========================================================================
constexpr int kAbsThreads = 256;
constexpr int kAbsCols = 128;
constexpr int kAbsRows = 16;

struct AbsorbParams {
  const __nv_bfloat16* q;     // [R, 64, Dn+64]
  const __nv_bfloat16* kv_b;  // [64, Dn+Dv, 512]
  const int32_t* T;
  const int32_t* nsel;
  __nv_bfloat16* qcat;  // [R, 64, 576]
  int32_t* tile_start;  // [NR + 1]
  int32_t* bad;         // [NR]
  int B, S, T_cap, Dn, Dv, topk, sparse;
  int do_qabs;            // 0: plan and rotary part only (qabs comes from the GEMM kernel)
  // L2 prefetch (small batches): the latent cache rows [0, T[b]) of every
  // sequence and the W_UV rows this CTA's combine counterpart will read
  const __nv_bfloat16* Lc;
  const __nv_bfloat16* Rc;
  int prefetch;
  double theta[kDr / 2];  // RoPE frequencies rope_base^(-2j/qk_rope), from the host
  unsigned int* flags;
};

// Partial dot products of NR query rows with one W_UK column over i in [i0, i1).
template <int NR>
__device__ __forceinline__ void absorb_rows(const __nv_bfloat16* Ws, const float* qn, int Dn, int col, int i0,
                                            int i1, float* part, int half) {
  float acc[NR];
#pragma unroll
  for (int u = 0; u < NR; ++u) acc[u] = 0.f;
  for (int i = i0; i < i1; ++i) {
    const float wv = __bfloat162float(Ws[i * kAbsCols + col]);
#pragma unroll
    for (int u = 0; u < NR; ++u) acc[u] = fmaf(qn[u * Dn + i], wv, acc[u]);
  }
#pragma unroll
  for (int u = 0; u < NR; ++u) part[(half * kAbsRows + u) * kAbsCols + col] = acc[u];
}

__global__ void __launch_bounds__(kAbsThreads) absorb_kernel(const AbsorbParams p) {
  // Under programmatic serialization this kernel may start before the
  // previous kernel of the stream retires (for example the combine of an
  // earlier call that still reads the workspace): wait before touching memory.
  grid_dep_wait();
  grid_dep_launch();
  extern __shared__ __align__(16) unsigned char sm[];
  const int cb = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  if (p.prefetch && tid == 0) {
    // Everything the later kernels of this call read streams from HBM now,
    // while this kernel works on W_UK: W_UV rows (64 per CTA) and 1/nblk of
    // every sequence's cache rows.
    const int nblk = gridDim.x * gridDim.y, me = h * gridDim.x + cb;
    const __nv_bfloat16* wuv = p.kv_b + ((size_t)h * (p.Dn + p.Dv) + p.Dn + (size_t)cb * (p.Dv / gridDim.x)) * kDl;
    l2_prefetch(wuv, (uint32_t)(p.Dv / gridDim.x) * kDl * 2);
    for (int b = 0; b < p.B; ++b) {
      const int Tb = min(max(p.T[b], 0), p.T_cap);
      const size_t lb = (size_t)Tb * kDl * 2, rb = (size_t)Tb * kDr * 2;
      const size_t l0 = (lb * me / nblk) & ~(size_t)15, l1 = (lb * (me + 1) / nblk) & ~(size_t)15;
      const size_t r0 = (rb * me / nblk) & ~(size_t)15, r1 = (rb * (me + 1) / nblk) & ~(size_t)15;
      const unsigned char* lbase = reinterpret_cast<const unsigned char*>(p.Lc + (size_t)b * p.T_cap * kDl);
      const unsigned char* rbase = reinterpret_cast<const unsigned char*>(p.Rc + (size_t)b * p.T_cap * kDr);
      if (l1 > l0) l2_prefetch(lbase + l0, (uint32_t)(l1 - l0));
      if (r1 > r0) l2_prefetch(rbase + r0, (uint32_t)(r1 - r0));
    }
  }
  const int Dn = p.Dn, Dq = Dn + kDr;
  const int R = p.B * p.S;
  __nv_bfloat16* Ws = reinterpret_cast<__nv_bfloat16*>(sm);                      // [Dn][128]
  float* qn = reinterpret_cast<float*>(sm + (size_t)Dn * kAbsCols * 2);           // [kAbsRows][Dn]

  // W_UK[h][:, cb*128 : cb*128+128] -> smem: every 16-byte load is issued
  // before the first store so that the whole tile is in flight at once.
  const __nv_bfloat16* W = p.kv_b + (size_t)h * (Dn + p.Dv) * kDl + cb * kAbsCols;
  const int nvec = p.do_qabs ? Dn * kAbsCols / 8 : 0;
  constexpr int kMaxVec = 256 * kAbsCols / 8 / kAbsThreads;  // qk_nope <= 256
  uint4 wv[kMaxVec];
#pragma unroll
  for (int u = 0; u < kMaxVec; ++u) {
    const int e = tid + u * kAbsThreads;
    if (e < nvec) {
      const int i = e / (kAbsCols / 8), c8 = e % (kAbsCols / 8);
      wv[u] = __ldg(reinterpret_cast<const uint4*>(W + (size_t)i * kDl + c8 * 8));
    }
  }
#pragma unroll
  for (int u = 0; u < kMaxVec; ++u) {
    const int e = tid + u * kAbsThreads;
    if (e < nvec) {
      const int i = e / (kAbsCols / 8), c8 = e % (kAbsCols / 8);
      *reinterpret_cast<uint4*>(Ws + i * kAbsCols + c8 * 8) = wv[u];
    }
  }

  if (cb == 0 && h == 0) {  // tile plan: tile_start[row] (exclusive prefix), bad[row]
    const int NR = p.sparse ? R : p.B;
    __shared__ int carry;
    __shared__ int wsum[kAbsThreads / 32];
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < NR; base += kAbsThreads) {
      const int r = base + tid;
      int tiles = 0;
      if (r < NR) {
        const int b = p.sparse ? r / p.S : r;
        const int Tb = p.T[b];
        int bad = (Tb < p.S || Tb > p.T_cap) ? MLA_DEV_BAD_LENGTH : 0;
        int nk = Tb;
        if (!bad && p.sparse) {
          nk = p.nsel[r];
          if (nk < 1 || nk > p.topk) bad = MLA_DEV_BAD_INDEX;
        }
        if (bad) raise_flag(p.flags, bad);
        p.bad[r] = bad;
        tiles = bad ? 0 : (nk + kTile - 1) / kTile;
      }
      // block inclusive scan of `tiles`
      int x = tiles;
      const int lane = tid & 31, w = tid >> 5;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) wsum[w] = x;
      __syncthreads();
      int off = 0;
      for (int i = 0; i < w; ++i) off += wsum[i];
      const int incl = carry + off + x;
      if (r < NR) p.tile_start[r + 1] = incl;
      __syncthreads();
      if (tid == kAbsThreads - 1) carry = incl;
      __syncthreads();
    }
    if (tid == 0) p.tile_start[0] = 0;
  }
  __syncthreads();

  if (!p.do_qabs) {  // rotary part only, every (row, pair) in parallel
    for (int e = tid; e < R * (kDr / 2); e += kAbsThreads) {
      const int r = e / (kDr / 2), j = e % (kDr / 2), b = r / p.S, s = r % p.S;
      const int Tb = p.T[b];
      const int pos = (Tb < p.S || Tb > p.T_cap) ? 0 : Tb - p.S + s;
      const double ang = (double)pos * p.theta[j];
      const double k = rint(ang * 0.15915494309189535);
      const float red = (float)fma(-k, 6.283185307179586, ang);
      float sn, cs;
      sincosf(red, &sn, &cs);
      const __nv_bfloat16* qr = p.q + ((size_t)r * kH + h) * Dq + Dn;
      const float x0 = __bfloat162float(qr[2 * j]), x1 = __bfloat162float(qr[2 * j + 1]);
      __nv_bfloat16* dst = p.qcat + ((size_t)r * kH + h) * kDc + kDl;
      dst[j] = __float2bfloat16_rn(x0 * cs - x1 * sn);
      dst[kDr / 2 + j] = __float2bfloat16_rn(x1 * cs + x0 * sn);
    }
    return;
  }
  // Thread (col, half) sums i over one half of qk_nope; the halves meet in smem.
  const int col = tid % kAbsCols, half = tid / kAbsCols;
  const int i0 = half * (Dn / 2), i1 = i0 + Dn / 2;
  float* part = qn + kAbsRows * Dn;  // [2][kAbsRows][kAbsCols]
  for (int r0 = 0; r0 < R; r0 += kAbsRows) {
    const int nr = min(kAbsRows, R - r0);
    for (int e = tid; e < nr * Dn; e += kAbsThreads) {
      const int rr = e / Dn, i = e % Dn;
      qn[rr * Dn + i] = __bfloat162float(p.q[((size_t)(r0 + rr) * kH + h) * Dq + i]);
    }
    __syncthreads();
    if (!p.do_qabs) {
    } else if (nr == 1) absorb_rows<1>(Ws, qn, Dn, col, i0, i1, part, half);
    else if (nr <= 4) absorb_rows<4>(Ws, qn, Dn, col, i0, i1, part, half);
    else if (nr <= 8) absorb_rows<8>(Ws, qn, Dn, col, i0, i1, part, half);
    else absorb_rows<kAbsRows>(Ws, qn, Dn, col, i0, i1, part, half);
    __syncthreads();
    for (int e = tid; e < (p.do_qabs ? nr * kAbsCols : 0); e += kAbsThreads) {
      const int u = e / kAbsCols, c = e % kAbsCols;
      const float v = part[u * kAbsCols + c] + part[(kAbsRows + u) * kAbsCols + c];
      p.qcat[((size_t)(r0 + u) * kH + h) * kDc + cb * kAbsCols + c] = __float2bfloat16_rn(v);
    }
    if (cb == 0) {  // rotary part of the query, rotated to the row's own position
      for (int e = tid; e < nr * (kDr / 2); e += kAbsThreads) {
        const int rr = e / (kDr / 2), j = e % (kDr / 2);
        const int r = r0 + rr, b = r / p.S, s = r % p.S;
        const int Tb = p.T[b];
        const int pos = (Tb < p.S || Tb > p.T_cap) ? 0 : Tb - p.S + s;
        // angle in double, reduced to [-pi, pi] before the float sincos
        const double ang = (double)pos * p.theta[j];
        const double k = rint(ang * 0.15915494309189535);
        const float red = (float)fma(-k, 6.283185307179586, ang);
        float sn, cs;
        sincosf(red, &sn, &cs);
        const __nv_bfloat16* qr = p.q + ((size_t)r * kH + h) * Dq + Dn;
        const float x0 = __bfloat162float(qr[2 * j]), x1 = __bfloat162float(qr[2 * j + 1]);
        __nv_bfloat16* dst = p.qcat + ((size_t)r * kH + h) * kDc + kDl;
        dst[j] = __float2bfloat16_rn(x0 * cs - x1 * sn);
        dst[kDr / 2 + j] = __float2bfloat16_rn(x1 * cs + x0 * sn);
      }
    }
    __syncthreads();
  }
}

// ===========================================================================
// Combine kernel: merge the splits of every (row, head) and lift with W_UV.
// CTA = (64 output columns j, head h).  W_UV[h][j0:j0+64][:] is one
// contiguous 64 KiB block, fetched with a single bulk async copy that runs
// while the kernel waits for the attention grid.
// ===========================================================================
constexpr int kCmbThreads = 256;
constexpr int kCmbJ = 64;
constexpr int kCmbRows = 8;
constexpr int kCPitch = kDl + 4;   // floats per clat row in smem
constexpr int kMaxPieces = 256;    // splits per row (<= CTAs of the attention grid)
constexpr uint32_t kCmbWBytes = kCmbJ * kDl * 2;

struct CombineParams {
  const __nv_bfloat16* kv_b;
  const float* o_part;
  const float* ml_part;
  const int32_t* tile_start;
  const int32_t* T;
  const int32_t* bad;
  float* out;  // [R, 64, Dv]
  int B, S, G, Dn, Dv, sparse;
  unsigned int* flags;
};

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__global__ void __launch_bounds__(kCmbThreads) combine_kernel(const CombineParams p) {
  extern __shared__ __align__(128) unsigned char sm[];
  const __nv_bfloat16* Ws = reinterpret_cast<const __nv_bfloat16*>(sm);   // [64][512]
  float* clat = reinterpret_cast<float*>(sm + kCmbWBytes);                 // [kCmbRows][kCPitch]
  float* inv_l = clat + kCmbRows * kCPitch;                                // [kCmbRows]
  int* pcnt = reinterpret_cast<int*>(inv_l + kCmbRows);                    // [kCmbRows]
  int* pslot = pcnt + kCmbRows;                                            // [kCmbRows][kMaxPieces]
  float* pm = reinterpret_cast<float*>(pslot + kCmbRows * kMaxPieces);     // split weights
  float* pw = pm + kCmbRows * kMaxPieces;                                  // split row sums
  __shared__ uint64_t wbar;
  const int jb = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int j0 = jb * kCmbJ;
  if (tid == 0) {
    mbar_init(&wbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(&wbar, kCmbWBytes);
    bulk_copy_g2s(sm, p.kv_b + ((size_t)h * (p.Dn + p.Dv) + p.Dn + j0) * kDl, kCmbWBytes, &wbar);
  }
  grid_dep_launch();
  grid_dep_wait();  // partials come from the attention kernel
  const int R = p.B * p.S;
  const int NR = p.sparse ? R : p.B;
  const long long N = p.tile_start[NR];
  bool w_ready = false;
  for (int r0 = 0; r0 < R; r0 += kCmbRows) {
    const int nr = min(kCmbRows, R - r0);
    // (a) warp w lists the splits of row r0 + w with their normalised weights
    if (warp < nr) {
      const int r = r0 + warp, b = r / p.S, s = r % p.S;
      const int row = p.sparse ? r : b;
      int cnt = 0;
      if (!p.bad[row] && N > 0) {
        const long long a = p.tile_start[row], e = p.tile_start[row + 1];
        const int glo = chunk_of(a, N, p.G), ghi = chunk_of(e - 1, N, p.G);
        float M = -INFINITY;
        for (int g0 = glo; g0 <= ghi; g0 += 32) {
          const int gg = g0 + lane;
          int lo = 0, hi = 0;
          if (gg <= ghi) {
            if (p.sparse) piece_range<true>(p.tile_start, p.T, p.S, s, row, gg, p.G, N, &lo, &hi);
            else piece_range<false>(p.tile_start, p.T, p.S, s, row, gg, p.G, N, &lo, &hi);
          }
          const bool has = lo < hi;
          const int slot = p.sparse ? gg + row : (gg + row) * p.S + s;
          float2 ml = make_float2(-INFINITY, 0.f);
          if (has) ml = *reinterpret_cast<const float2*>(p.ml_part + ((size_t)slot * kH + h) * 2);
          const unsigned m = __ballot_sync(0xffffffffu, has);
          const int at = cnt + __popc(m & ((1u << lane) - 1));
          if (has) {
            pslot[warp * kMaxPieces + at] = slot;
            pm[warp * kMaxPieces + at] = ml.x;
            pw[warp * kMaxPieces + at] = ml.y;
          }
          cnt += __popc(m);
          M = fmaxf(M, ml.x);
        }
        M = warp_max(M);
        __syncwarp();  // entries were listed by other lanes
        float L = 0.f;
        for (int i = lane; i < cnt; i += 32) {
          const float wg = exp2f(pm[warp * kMaxPieces + i] - M);
          pm[warp * kMaxPieces + i] = wg;
          L = fmaf(wg, pw[warp * kMaxPieces + i], L);
        }
        L = warp_sum(L);
        for (int i = lane; i < cnt; i += 32) pm[warp * kMaxPieces + i] /= L;
        if (lane == 0) inv_l[warp] = 1.f;
      } else if (lane == 0) {
        inv_l[warp] = __int_as_float(0x7fc00000);
      }
      if (lane == 0) pcnt[warp] = cnt;
    }
    __syncthreads();
    // (b) clat[w][l] = sum_i weight_i * O_i[h][l]: all threads, two latents each
    for (int w = 0; w < nr; ++w) {
      const int cnt = pcnt[w];
      float2 acc = make_float2(0.f, 0.f);
      int i = 0;
      for (; i + 4 <= cnt; i += 4) {
        float2 o[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          o[u] = *reinterpret_cast<const float2*>(p.o_part + ((size_t)pslot[w * kMaxPieces + i + u] * kH + h) * kDl +
                                                  2 * tid);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float wg = pm[w * kMaxPieces + i + u];
          acc.x = fmaf(wg, o[u].x, acc.x);
          acc.y = fmaf(wg, o[u].y, acc.y);
        }
      }
      for (; i < cnt; ++i) {
        const float2 o =
            *reinterpret_cast<const float2*>(p.o_part + ((size_t)pslot[w * kMaxPieces + i] * kH + h) * kDl + 2 * tid);
        const float wg = pm[w * kMaxPieces + i];
        acc.x = fmaf(wg, o.x, acc.x);
        acc.y = fmaf(wg, o.y, acc.y);
      }
      *reinterpret_cast<float2*>(clat + w * kCPitch + 2 * tid) = acc;
    }
    if (!w_ready) {
      volatile int no_abort = 0;
      if (!mbar_wait(&wbar, 0, &no_abort, p.flags, kDrainNs)) raise_flag(p.flags, MLA_DEV_TIMEOUT);
      w_ready = true;
    }
    __syncthreads();
    // (c) out[r][h][j0 + j] = W_UV[j] . clat[r] (lanes split the latent axis)
#pragma unroll 1
    for (int jj = 0; jj < kCmbJ / 8; ++jj) {
      const int j = warp * (kCmbJ / 8) + jj;
      const __nv_bfloat16* wr = Ws + (size_t)j * kDl;
      const uint4 wlo = *reinterpret_cast<const uint4*>(wr + 8 * lane);
      const uint4 whi = *reinterpret_cast<const uint4*>(wr + 256 + 8 * lane);
      float wf[16];
      {
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&wlo);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&whi);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 fa = __bfloat1622float2(a2[q]);
          const float2 fb = __bfloat1622float2(b2[q]);
          wf[2 * q] = fa.x;
          wf[2 * q + 1] = fa.y;
          wf[8 + 2 * q] = fb.x;
          wf[8 + 2 * q + 1] = fb.y;
        }
      }
      for (int w = 0; w < nr; ++w) {
        const float* cr = clat + w * kCPitch;
        const float4 c0 = *reinterpret_cast<const float4*>(cr + 8 * lane);
        const float4 c1 = *reinterpret_cast<const float4*>(cr + 8 * lane + 4);
        const float4 c2 = *reinterpret_cast<const float4*>(cr + 256 + 8 * lane);
        const float4 c3 = *reinterpret_cast<const float4*>(cr + 256 + 8 * lane + 4);
        float d = wf[0] * c0.x;
        d = fmaf(wf[1], c0.y, d); d = fmaf(wf[2], c0.z, d); d = fmaf(wf[3], c0.w, d);
        d = fmaf(wf[4], c1.x, d); d = fmaf(wf[5], c1.y, d); d = fmaf(wf[6], c1.z, d); d = fmaf(wf[7], c1.w, d);
        d = fmaf(wf[8], c2.x, d); d = fmaf(wf[9], c2.y, d); d = fmaf(wf[10], c2.z, d); d = fmaf(wf[11], c2.w, d);
        d = fmaf(wf[12], c3.x, d); d = fmaf(wf[13], c3.y, d); d = fmaf(wf[14], c3.z, d); d = fmaf(wf[15], c3.w, d);
        d = warp_sum(d);
        if (lane == 0) p.out[((size_t)(r0 + w) * kH + h) * p.Dv + j0 + j] = d * inv_l[w];
      }
    }
    __syncthreads();
  }
  if (!w_ready) {  // R == 0 cannot happen, but never exit with the copy in flight
    volatile int no_abort = 0;
    mbar_wait(&wbar, 0, &no_abort, p.flags, kDrainNs);
  }
}

// ===========================================================================
// Merge kernel (batches with more than kSmallRows query rows): one warp per
// (row, head) forms the normalised latent context clat = sum_i w_i O_i / L
// (bf16) for the W_UV GEMM; inv_l is 1, or NaN for a flagged row.
// ===========================================================================
struct MergeParams {
  const float* o_part;
  const float* ml_part;
  const int32_t* tile_start;
  const int32_t* T;
  const int32_t* bad;
  __nv_bfloat16* clat;  // [R, 64, 512]
  float* inv_l;         // [R, 64]
  int B, S, G, sparse;
};

__global__ void __launch_bounds__(256) merge_kernel(const MergeParams p) {
  grid_dep_wait();
  grid_dep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = p.B * p.S;
  const int gw = blockIdx.x * 8 + warp;
  if (gw >= R * kH) return;
  const int r = gw / kH, h = gw % kH, b = r / p.S, s = r % p.S;
  const int row = p.sparse ? r : b;
  const int NR = p.sparse ? R : p.B;
  const long long N = p.tile_start[NR];
  __nv_bfloat16* dst = p.clat + ((size_t)r * kH + h) * kDl + 16 * lane;
  if (p.bad[row] || N <= 0) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(dst + 8) = make_uint4(0, 0, 0, 0);
    if (lane == 0) p.inv_l[(size_t)r * kH + h] = qnan();
    return;
  }
  const long long a = p.tile_start[row], e = p.tile_start[row + 1];
  const int glo = chunk_of(a, N, p.G), ghi = chunk_of(e - 1, N, p.G);
  float M = -INFINITY;
  for (int gg = glo + lane; gg <= ghi; gg += 32) {
    int lo, hi;
    if (p.sparse) piece_range<true>(p.tile_start, p.T, p.S, s, row, gg, p.G, N, &lo, &hi);
    else piece_range<false>(p.tile_start, p.T, p.S, s, row, gg, p.G, N, &lo, &hi);
    if (lo < hi) {
      const int slot = p.sparse ? gg + row : (gg + row) * p.S + s;
      M = fmaxf(M, p.ml_part[((size_t)slot * kH + h) * 2]);
    }
  }
  M = warp_max(M);
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  float L = 0.f;
  for (int gg = glo; gg <= ghi; ++gg) {
    int lo, hi;
    if (p.sparse) piece_range<true>(p.tile_start, p.T, p.S, s, row, gg, p.G, N, &lo, &hi);
    else piece_range<false>(p.tile_start, p.T, p.S, s, row, gg, p.G, N, &lo, &hi);
    if (lo >= hi) continue;
    const int slot = p.sparse ? gg + row : (gg + row) * p.S + s;
    const float2 ml = *reinterpret_cast<const float2*>(p.ml_part + ((size_t)slot * kH + h) * 2);
    const float wgt = exp2f(ml.x - M);
    L = fmaf(wgt, ml.y, L);
    const float4* op = reinterpret_cast<const float4*>(p.o_part + ((size_t)slot * kH + h) * kDl + 16 * lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 o = op[i];
      acc[4 * i] = fmaf(wgt, o.x, acc[4 * i]);
      acc[4 * i + 1] = fmaf(wgt, o.y, acc[4 * i + 1]);
      acc[4 * i + 2] = fmaf(wgt, o.z, acc[4 * i + 2]);
      acc[4 * i + 3] = fmaf(wgt, o.w, acc[4 * i + 3]);
    }
  }
  const float il = 1.f / L;
  uint4 w0, w1;
  w0.x = pack2(acc[0] * il, acc[1] * il);
  w0.y = pack2(acc[2] * il, acc[3] * il);
  w0.z = pack2(acc[4] * il, acc[5] * il);
  w0.w = pack2(acc[6] * il, acc[7] * il);
  w1.x = pack2(acc[8] * il, acc[9] * il);
  w1.y = pack2(acc[10] * il, acc[11] * il);
  w1.z = pack2(acc[12] * il, acc[13] * il);
  w1.w = pack2(acc[14] * il, acc[15] * il);
  *reinterpret_cast<uint4*>(dst) = w0;
  *reinterpret_cast<uint4*>(dst + 8) = w1;
  if (lane == 0) p.inv_l[(size_t)r * kH + h] = (L == L) ? 1.f : qnan();
}

// ===========================================================================
// Gather kernel (sparse only): staging[r, j, 0:512 | 512:576] = Lc | Rc of key
// sel[r, j] for j < nsel[r]; zero rows past nsel or for an index outside
// [0, pos] (flagged).  CTA = (32 keys, row r); one warp per key row.
// ===========================================================================
struct GatherParams {
  const __nv_bfloat16* Lc;
  const __nv_bfloat16* Rc;
  const int32_t* T;
  const int32_t* sel;
  const int32_t* nsel;
  __nv_bfloat16* stage;  // [R, Kpad, 576]
  int B, S, T_cap, topk, Kpad;
  unsigned int* flags;
};

__global__ void __launch_bounds__(256) gather_kernel(const GatherParams p) {
  const int r = blockIdx.y, b = r / p.S, s = r % p.S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Tb = p.T[b];
  const int n = p.nsel[r];
  const bool row_ok = Tb >= p.S && Tb <= p.T_cap && n >= 1 && n <= p.topk;
  const int pos = Tb - p.S + s;
  for (int kk = 0; kk < 4; ++kk) {
    const int j = blockIdx.x * 32 + warp * 4 + kk;
    int idx = -1;
    if (row_ok && j < n) {
      idx = p.sel[(size_t)r * p.topk + j];
      if (idx < 0 || idx > pos) {
        if (lane == 0) raise_flag(p.flags, MLA_DEV_BAD_INDEX);
        idx = -1;
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(p.stage + ((size_t)r * p.Kpad + j) * kDc);
    const uint4* lsrc = reinterpret_cast<const uint4*>(p.Lc + ((size_t)b * p.T_cap + (idx < 0 ? 0 : idx)) * kDl);
    const uint4* rsrc = reinterpret_cast<const uint4*>(p.Rc + ((size_t)b * p.T_cap + (idx < 0 ? 0 : idx)) * kDr);
    for (int c = lane; c < kDc / 8; c += 32) {
      uint4 v = make_uint4(0, 0, 0, 0);
      if (idx >= 0) v = c < kDl / 8 ? __ldg(lsrc + c) : __ldg(rsrc + (c - kDl / 8));
      dst[c] = v;
    }
  }
}

// ===========================================================================
// Host side
// ===========================================================================
struct Plan {
  int G, NR, P, R, Kpad;
  size_t off_q, off_ts, off_bad, off_o, off_ml, off_stage, off_clat, off_invl, total;
};

// Query rows above which the weight products run as tcgen05 GEMMs; below it
// they are weight-bandwidth-bound GEMVs on the CUDA cores.
constexpr int kSmallRows = 8;

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Raise a kernel's dynamic shared memory limit once per device.
template <typename Kern>
cudaError_t set_smem_once(Kern kern, int bytes, std::atomic<unsigned long long>* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (done->load() & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done->fetch_or(bit);
  return e;
}

std::atomic<unsigned long long> g_abs_attr{0}, g_attn_attr[2] = {{0}, {0}}, g_cmb_attr{0};

Plan make_plan(int B, int S, int T_cap, int sparse_topk) {
  Plan pl{};
  const int sms = sm_count();
  pl.R = B * S;
  if (!sparse_topk) {
    pl.NR = B;
    const long long tiles = (long long)B * ((T_cap + kTile - 1) / kTile);
    long long G = sms / S;
    if (G < 1) G = 1;
    if (G > tiles) G = tiles;
    if (G > kMaxPieces) G = kMaxPieces;
    pl.G = (int)G;
    pl.P = (pl.G + B - 1) * S;
  } else {
    pl.NR = pl.R;
    const long long tiles = (long long)pl.R * ((sparse_topk + kTile - 1) / kTile);
    long long G = sms;
    if (G > tiles) G = tiles;
    if (G > kMaxPieces) G = kMaxPieces;
    pl.G = (int)G;
    pl.P = pl.G + pl.R - 1;
  }
  size_t off = 0;
  pl.off_q = off;
  off = align256(off + (size_t)pl.R * kH * kDc * 2);
  pl.off_ts = off;
  off = align256(off + (size_t)(pl.NR + 1) * 4);
  pl.off_bad = off;
  off = align256(off + (size_t)pl.NR * 4);
  pl.off_o = off;
  off = align256(off + (size_t)pl.P * kH * kDl * 4);
  pl.off_ml = off;
  off = align256(off + (size_t)pl.P * kH * 2 * 4);
  pl.Kpad = sparse_topk ? (sparse_topk + kTile - 1) / kTile * kTile : 0;
  pl.off_stage = off;
  off = align256(off + (size_t)pl.R * pl.Kpad * kDc * 2);
  pl.off_clat = off;
  off = align256(off + (pl.R > kSmallRows ? (size_t)pl.R * kH * kDl * 2 : 0));
  pl.off_invl = off;
  off = align256(off + (pl.R > kSmallRows ? (size_t)pl.R * kH * 4 : 0));
  pl.total = off;
  return pl;
}

template <typename Kern, typename Arg>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const Arg& arg) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, arg);
}

cudaError_t run(const DecodeArgs& a, void* ws, bool sparse, cudaStream_t st) {
  const Geometry& g = a.g;
  const int B = a.B, S = a.S;
  const Plan pl = make_plan(B, S, a.T_cap, sparse ? a.topk : 0);
  if ((long long)B * a.T_cap >= (1ll << 31)) return cudaErrorInvalidValue;
  unsigned char* w = static_cast<unsigned char*>(ws);
  __nv_bfloat16* qcat = reinterpret_cast<__nv_bfloat16*>(w + pl.off_q);
  int32_t* ts = reinterpret_cast<int32_t*>(w + pl.off_ts);
  int32_t* bad = reinterpret_cast<int32_t*>(w + pl.off_bad);
  float* o_part = reinterpret_cast<float*>(w + pl.off_o);
  float* ml_part = reinterpret_cast<float*>(w + pl.off_ml);
  __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(w + pl.off_stage);
  cudaError_t e;

  // 0. sparse: gather the selected key rows (plain launch: the absorb kernel,
  //    launched next with programmatic serialization, starts once it retires)
  if (sparse) {
    GatherParams gp{};
    gp.Lc = static_cast<const __nv_bfloat16*>(a.Lc);
    gp.Rc = static_cast<const __nv_bfloat16*>(a.Rc);
    gp.T = a.T;
    gp.sel = a.sel;
    gp.nsel = a.nsel;
    gp.stage = stage;
    gp.B = B;
    gp.S = S;
    gp.T_cap = a.T_cap;
    gp.topk = a.topk;
    gp.Kpad = pl.Kpad;
    gp.flags = a.flags;
    kernel_mark(st, "gather");
    gather_kernel<<<dim3(pl.Kpad / 32, pl.R), 256, 0, st>>>(gp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }

  // 1. absorb
  AbsorbParams ap{};
  ap.q = static_cast<const __nv_bfloat16*>(a.q);
  ap.kv_b = static_cast<const __nv_bfloat16*>(a.kv_b);
  ap.T = a.T;
  ap.nsel = a.nsel;
  ap.qcat = qcat;
  ap.tile_start = ts;
  ap.bad = bad;
  ap.B = B;
  ap.S = S;
  ap.T_cap = a.T_cap;
  ap.Dn = g.Dn;
  ap.Dv = g.Dv;
  ap.topk = a.topk;
  ap.sparse = sparse ? 1 : 0;
  const bool big = pl.R > kSmallRows;
  ap.do_qabs = big ? 0 : 1;
  ap.Lc = static_cast<const __nv_bfloat16*>(a.Lc);
  ap.Rc = static_cast<const __nv_bfloat16*>(a.Rc);
  // L2 prefetch on the small-batch path while the cache stays well inside L2
  ap.prefetch = (!big && !sparse && (long long)B * a.T_cap * (kDl + kDr) * 2 <= (48ll << 20)) ? 1 : 0;
  for (int j = 0; j < kDr / 2; ++j) ap.theta[j] = std::pow(g.rope_base, -2.0 * j / kDr);
  ap.flags = a.flags;
  const size_t abs_smem = (size_t)g.Dn * kAbsCols * 2 + (size_t)kAbsRows * g.Dn * 4 +
                          (size_t)2 * kAbsRows * kAbsCols * 4;
  e = set_smem_once(absorb_kernel, 200 * 1024, &g_abs_attr);
  if (e != cudaSuccess) return e;
  kernel_mark(st, big ? "plan_rope" : "absorb");
  e = launch_pdl(absorb_kernel, dim3(big ? 1 : kDl / kAbsCols, kH), dim3(kAbsThreads), abs_smem, st, ap);
  if (e != cudaSuccess) return e;
  if (big) {  // qabs for many rows: per-head GEMM [R x qk_nope] x W_UK[h] on the tensor cores
    GemmArgs ga{};
    ga.a_base = a.q;
    ga.a_ld_z = g.Dn + kDr;
    ga.a_ld_m = (long long)kH * (g.Dn + kDr);
    ga.b_base = a.kv_b;
    ga.b_rows = (long long)kH * (g.Dn + g.Dv);
    ga.b_cols = kDl;
    ga.b_ld = kDl;
    ga.b_mn_major = 1;
    ga.b_row0 = 0;
    ga.b_rows_per_z = g.Dn + g.Dv;
    ga.b_col0 = 0;
    ga.c_base = qcat;
    ga.c_ld_m = (long long)kH * kDc;
    ga.c_ld_z = kDc;
    ga.out_kind = kGemmOutBf16;
    ga.M = pl.R;
    ga.N = kDl;
    ga.K = g.Dn;
    ga.Z = kH;
    ga.flags = a.flags;
    ga.wait_ns = a.wait_limit_ns;
    kernel_mark(st, "absorb_gemm");
    e = launch_gemm_tc(ga, true, st);
    if (e != cudaSuccess) return e;
  }

  // 2. attention
  AttnParams tp{};
  bool maps_ok = make_tmap_2d_bf16(&tp.mQ, qcat, (uint64_t)pl.R * kH, kDc, kDc, kH, 64);
  if (!sparse) {
    const uint64_t rows = (uint64_t)B * a.T_cap;
    maps_ok = maps_ok && make_tmap_2d_bf16(&tp.mL, a.Lc, rows, kDl, kDl, kTile, 64) &&
              make_tmap_2d_bf16(&tp.mR, a.Rc, rows, kDr, kDr, kTile, 64);
    tp.kv_rows = a.T_cap;
  } else {
    const uint64_t rows = (uint64_t)pl.R * pl.Kpad;
    maps_ok = maps_ok && make_tmap_2d_bf16(&tp.mL, stage, rows, kDl, kDc, kTile, 64) &&
              make_tmap_2d_bf16(&tp.mR, stage + kDl, rows, kDr, kDc, kTile, 64);
    tp.kv_rows = pl.Kpad;
  }
  if (!maps_ok) return cudaErrorInvalidValue;
  tp.T = a.T;
  tp.sel = a.sel;
  tp.nsel = a.nsel;
  tp.tile_start = ts;
  tp.B = B;
  tp.S = S;
  tp.T_cap = a.T_cap;
  tp.G = pl.G;
  tp.topk = a.topk;
  tp.c = g.scale * kLog2e;
  tp.o_part = o_part;
  tp.ml_part = ml_part;
  tp.flags = a.flags;
  tp.wait_ns = a.wait_limit_ns;
  auto kern = sparse ? attn_kernel<true> : attn_kernel<false>;
  e = set_smem_once(kern, (int)kAttnDynSmem, &g_attn_attr[sparse ? 1 : 0]);
  if (e != cudaSuccess) return e;
  const int nblk = sparse ? pl.G : pl.G * S;
  kernel_mark(st, "attention");
  e = launch_pdl(kern, dim3(nblk), dim3(kAttnThreads), kAttnDynSmem, st, tp);
  if (e != cudaSuccess) return e;

  // 3. merge of the splits and the W_UV lift
  if (big) {
    MergeParams mp{};
    mp.o_part = o_part;
    mp.ml_part = ml_part;
    mp.tile_start = ts;
    mp.T = a.T;
    mp.bad = bad;
    mp.clat = reinterpret_cast<__nv_bfloat16*>(w + pl.off_clat);
    mp.inv_l = reinterpret_cast<float*>(w + pl.off_invl);
    mp.B = B;
    mp.S = S;
    mp.G = pl.G;
    mp.sparse = sparse ? 1 : 0;
    kernel_mark(st, "merge");
    e = launch_pdl(merge_kernel, dim3((pl.R * kH + 7) / 8), dim3(256), 0, st, mp);
    if (e != cudaSuccess) return e;
    GemmArgs gu{};
    gu.a_base = mp.clat;
    gu.a_ld_z = kDl;
    gu.a_ld_m = (long long)kH * kDl;
    gu.b_base = a.kv_b;
    gu.b_rows = (long long)kH * (g.Dn + g.Dv);
    gu.b_cols = kDl;
    gu.b_ld = kDl;
    gu.b_mn_major = 0;
    gu.b_row0 = g.Dn;
    gu.b_rows_per_z = g.Dn + g.Dv;
    gu.b_col0 = 0;
    gu.c_base = a.out;
    gu.c_ld_m = (long long)kH * g.Dv;
    gu.c_ld_z = g.Dv;
    gu.out_kind = kGemmOutF32Scaled;
    gu.scale = mp.inv_l;
    gu.M = pl.R;
    gu.N = g.Dv;
    gu.K = kDl;
    gu.Z = kH;
    gu.flags = a.flags;
    gu.wait_ns = a.wait_limit_ns;
    kernel_mark(st, "up_gemm");
    return launch_gemm_tc(gu, true, st);
  }
  CombineParams cp{};
  cp.kv_b = static_cast<const __nv_bfloat16*>(a.kv_b);
  cp.o_part = o_part;
  cp.ml_part = ml_part;
  cp.tile_start = ts;
  cp.T = a.T;
  cp.bad = bad;
  cp.out = a.out;
  cp.B = B;
  cp.S = S;
  cp.G = pl.G;
  cp.Dn = g.Dn;
  cp.Dv = g.Dv;
  cp.sparse = sparse ? 1 : 0;
  cp.flags = a.flags;
  const size_t cmb_smem = (size_t)kCmbWBytes + (size_t)kCmbRows * kCPitch * 4 + kCmbRows * 8 +
                          (size_t)kCmbRows * kMaxPieces * 12;
  e = set_smem_once(combine_kernel, (int)cmb_smem, &g_cmb_attr);
  if (e != cudaSuccess) return e;
  kernel_mark(st, "combine");
  return launch_pdl(combine_kernel, dim3(g.Dv / kCmbJ, kH), dim3(kCmbThreads), cmb_smem, st, cp);
}

}  // namespace

bool tc_decode_geometry_ok(const Geometry& g) {
  return g.H == kH && g.Dl == kDl && g.Dr == kDr && g.Dn >= 64 && g.Dn % 64 == 0 && g.Dn <= 256 &&
         g.Dv >= kCmbJ && g.Dv % kCmbJ == 0;
}

int tc_decode_launch_count(bool sparse, int B, int S) {
  return (sparse ? 1 : 0) + ((long long)B * S > kSmallRows ? 5 : 3);
}

size_t tc_decode_workspace_bytes(const Geometry&, int B, int S, int T_cap, int sparse_topk) {
  return make_plan(B, S, T_cap, sparse_topk).total;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, void* ws, size_t, cudaStream_t st) {
  return run(a, ws, false, st);
}

cudaError_t launch_sparse_decode_tc(const DecodeArgs& a, void* ws, size_t, cudaStream_t st) {
  return run(a, ws, true, st);
}

}  // namespace mla
