// attn_core.cuh -- the absorbed-attention pass over the latent cache on the
// tensor cores (page "MLA 注意力与 KV 缓存", §2.3: scores qabs . Lc + q_rot . Rc,
// softmax, latent context sum p Lc), as used by the attention kernel.
//
// Per key tile the tensor pipe runs two products,
//   S^T[128 keys x 64 rows]   = [Lc | Rc] tile x qcat^T              (K = 576)
//   O^T[512 x 64 rows]       += Lc tile^T x P^T                      (K = keys)
// with the softmax warps turning S^T into P^T in between.  The tile is read
// from memory once: shared memory holds the query block and the nine atoms of
// one tile (eight latent, one rope-key atom that P^T reuses once the score
// product is done).  The value product releases the latent atoms pairwise, so
// the next tile's loads start while it still runs, and the next score product
// accumulates atom by atom as they land.
//
// Warp roles (kAttnThreads = 320): warp 0 streams the tile's nine 64-column
// atoms with TMA (attn_producer), warp 1 issues the MMAs (attn_mma), warps 2-9
// run the online softmax, one key row and 32 heads per thread, and write the
// per-split (m, l, O) partials (attn_softmax).
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kH = 64, kDl = 512, kDr = 64, kDc = 576;  // kDc = kv_lora + qk_rope
constexpr int kTile = 128;
constexpr int kSlots = 9;                      // 8 latent atoms + 1 rope atom per key tile
constexpr uint32_t kSlotBytes = 16384;         // 128 keys x 64 bf16
constexpr uint32_t kQAtomBytes = 8192;         // 64 rows x 64 bf16
constexpr uint32_t kQBytes = 9 * kQAtomBytes;  // 73728
constexpr uint32_t kKVBytes = 9 * kSlotBytes;  // 147456
constexpr uint32_t kAttnDynSmem = kQBytes + kKVBytes + 1024;
// FP8 latent cache (attn8_kernel): a key tile is four latent atoms of 128
// keys x 128 E4M3 codes and the bf16 rope atom, 16 KB each, and two tiles are
// resident; the query block is four 8 KB atoms of 64 rows x 128 codes and the
// bf16 rope atom, loaded from the quantised query rows (640 bytes each: 512
// codes, then 64 bf16).
constexpr int kAtoms8 = 5;
constexpr uint32_t kQ8Bytes = 5 * kQAtomBytes;     // 40960
constexpr uint32_t kTile8Bytes = 5 * kSlotBytes;   // 81920
constexpr uint32_t kAttn8DynSmem = kQ8Bytes + 2 * kTile8Bytes + 1024;
constexpr int kQ8Row = kDl + 2 * kDr;              // 640 bytes
constexpr uint32_t kTmemO8 = 128;  // FP8: S^T double-buffered (cols 0..127), then O^T
constexpr int kSoftWarps = 8;
constexpr int kSoftThreads = 32 * kSoftWarps;
constexpr int kAttnThreads = 64 + kSoftThreads;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;    // S^T: 64 columns
constexpr uint32_t kTmemO = 128;  // O^T: 4 M-blocks x 64 columns
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTau = 8.f;       // lazy rescale threshold (log2 units)
constexpr int kPlanMax = 1024;    // tile-list rows whose plan the attention CTA builds itself
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
  int kv_rows;    // rows of the key source per tile-list row: T_cap (dense) or Kpad (sparse)
  int read_once;  // every key tile is loaded by exactly one CTA: mark its lines evict-first in L2
  int qsplit;     // CTAs per piece (1, 2 or 4): each repeats the score product and owns 4/qsplit
                  // of the four 128-row blocks of O^T (the value product and its partial)
  float c;        // softmax scale * log2(e)
  float lat_scale;  // FP8 cache: latent row = lat_scale * E4M3 codes
  const float* fh;  // FP8 cache: per query row, c * lat_scale * the row's quantisation scale
  const __nv_bfloat16* qcat;  // FP8 cache, few rows: the unquantised query rows [R*64, 576]
  float* o_part;
  float* ml_part;
  unsigned int* flags;
  long long wait_ns;
  PageTable pages;  // dense path: key tiles come from pages (page_size a multiple of kTile)
};

// One arrival per warp on a barrier initialised with the number of arriving
// warps: after the warp syncs, lane 0's release-arrive publishes what every
// lane wrote before it (ordered by the fences each lane issued first).  All
// 32 lanes call it.
__device__ __forceinline__ void mbar_arrive_warp(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
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

// a / d for a >= 0, d > 0: a 32-bit division whenever a fits in 32 bits
// (always, for tile counts below 2^23), the 64-bit one otherwise.
__device__ __forceinline__ long long div_nonneg(long long a, long long d) {
  if (((unsigned long long)a >> 32) == 0 && ((unsigned long long)d >> 32) == 0)
    return (long long)((unsigned)a / (unsigned)d);
  return a / d;
}

// Chunk g of the flattened tile list covers tiles [N*g/G, N*(g+1)/G).
__device__ __forceinline__ long long chunk_begin(long long N, int g, int G) { return div_nonneg(N * g, G); }

__device__ __forceinline__ int chunk_of(long long x, long long N, int G) {
  int g = (int)div_nonneg(x * G, N);
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

// Reduce 32 per-lane values over the 32 lanes of a warp; afterwards lane L
// holds the result for entry L in v[0].
template <bool kMax>
__device__ __forceinline__ void transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int o = 16 >> step;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? v[i] : v[i + o];
      const float keep = upper ? v[i + o] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
}

// Walks the key tiles of one attention CTA in processing order: the pieces
// (tile-list rows) of chunk g, and within a piece its tiles lo..hi-1.
template <bool kSparse>
struct TileCursor {
  int row, lo, hi, k;
  bool live;
  __device__ __forceinline__ void start(const AttnParams& p, const int32_t* ts, int NR, long long N, int g, int s,
                                        int row0) {
    row = row0;
    live = next_piece<kSparse>(p, ts, NR, N, g, s, &row, &lo, &hi);
    k = lo;
  }
  __device__ __forceinline__ void next(const AttnParams& p, const int32_t* ts, int NR, long long N, int g, int s) {
    if (++k < hi) return;
    ++row;
    live = next_piece<kSparse>(p, ts, NR, N, g, s, &row, &lo, &hi);
    k = lo;
  }
  __device__ __forceinline__ bool first() const { return k == lo; }
  __device__ __forceinline__ bool last() const { return k == hi - 1; }
};

// Keys of tile k of tile-list row `row` that the query attends to (>= 1 for a
// tile inside a piece).
template <bool kSparse>
__device__ __forceinline__ int tile_keys(const AttnParams& p, int row, int s, int k) {
  const int nk = kSparse ? p.nsel[row] : p.T[row] - p.S + s + 1;
  const int n = nk - k * kTile;
  return n < kTile ? n : kTile;
}

// Shared-memory state of one attention CTA (static shared; the query block
// and the key tile live in dynamic shared memory).
struct AttnShared {
  uint64_t full_bar[kSlots], empty_bar[kSlots];
  uint64_t q_full, q_empty, s_full, s_free, p_full, mma_done, o_blk[4];
  uint32_t tmem_base;
  int abort_flag;
  __align__(16) float red_max[4][kH];
  __align__(16) float red_sum[4][kH];
  __align__(16) float m_sh[kH];
  __align__(16) float alpha_sh[kH];
};

// Where one CTA's share of the tile list starts, and its place in the grid.
struct AttnCtx {
  const int32_t* ts;  // tile-start prefix over the tile-list rows [NR + 1]
  int NR;
  long long N;        // ts[NR]
  int g, s;           // chunk, query position
  int part, mb0, mb1; // latent part (value-product blocks [mb0, mb1))
  int row0;           // first tile-list row of chunk g
  unsigned char* sQ;  // query block (9 atoms of 64 rows x 64 bf16)
  unsigned char* sKV; // key tile (9 atoms of 128 keys x 64 bf16)
  uint32_t tmem;
};

// Barrier initialisation (one thread).
__device__ __forceinline__ void attn_init_barriers(AttnShared& sh) {
  for (int i = 0; i < kSlots; ++i) {
    mbar_init(&sh.full_bar[i], 1);
    mbar_init(&sh.empty_bar[i], 1);
  }
  mbar_init(&sh.q_full, 1);
  mbar_init(&sh.q_empty, 1);
  mbar_init(&sh.s_full, 1);
  mbar_init(&sh.s_free, kSoftWarps);
  mbar_init(&sh.p_full, kSoftWarps);
  for (int m = 0; m < 4; ++m) mbar_init(&sh.o_blk[m], 1);
  mbar_init(&sh.mma_done, 1);
  sh.abort_flag = 0;
}

// Tile-start prefix over NR <= nthreads-bounded rows, built by every thread of
// the block from T / nsel (kernel inputs): plan_ts[0..NR], plan_wsum scratch
// of one int per warp.
template <bool kSparse>
__device__ __forceinline__ void attn_local_plan(const AttnParams& p, int NR, int* plan_ts, int* plan_wsum) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nthr = blockDim.x, nwarp = nthr >> 5;
  int carry = 0;
  for (int base = 0; base < NR; base += nthr) {
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
    for (int i = 0; i < nwarp; ++i) tot += plan_wsum[i];
    carry += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) plan_ts[0] = 0;
  __syncthreads();
}

// ------------------------------------------------------------ producer (lane 0 of warp 0)
// qwait() is called once, right before the first query-block load: it returns
// false when the query block will never be ready (the wait gave up).
template <bool kSparse, bool kPaged, class QWait>
__device__ __forceinline__ void attn_producer(const AttnParams& p, AttnShared& sh, const AttnCtx& cx, QWait&& qwait) {
  volatile int* abort = &sh.abort_flag;
  const int S = p.S;
  const uint64_t pol_once = l2_policy_evict_first();
  TileCursor<kSparse> c;
  c.start(p, cx.ts, cx.NR, cx.N, cx.g, cx.s, cx.row0);
  int it = 0, pc = -1, last_it[kSlots], last_q = -1;
  for (int a = 0; a < kSlots; ++a) last_it[a] = -1;
  bool ok = true, q_waited = false;
  while (ok && c.live) {
    const bool first = c.first();
    if (first) ++pc;
    int y = c.row * p.kv_rows + c.k * kTile;  // tile-list row = block of key-source rows
    if (kPaged) {  // the tile's 128 rows lie in one page
      bool bad_page = false;
      y = (int)cache_row(p.pages, c.row, p.T_cap, c.k * kTile, &bad_page);
      if (bad_page) raise_flag(p.flags, MLA_DEV_BAD_INDEX);
    }
    const uint32_t par = (it & 1) ^ 1;
    for (int a = 0; a < kSlots && ok; ++a) {
      // latent atoms 2m and 2m + 1 are released together (empty_bar[2m]),
      // the rope slot on its own
      if (a == 8 || (a & 1) == 0) ok = mbar_wait(&sh.empty_bar[a], par, abort, p.flags, p.wait_ns);
      if (!ok) break;
      mbar_arrive_expect_tx(&sh.full_bar[a], kSlotBytes);
      const CUtensorMap* map = a < 8 ? &p.mL : &p.mR;
      const int x = a < 8 ? 64 * a : 0;
      if (p.read_once) tma_load_2d_hint(cx.sKV + a * kSlotBytes, map, x, y, &sh.full_bar[a], pol_once);
      else tma_load_2d(cx.sKV + a * kSlotBytes, map, x, y, &sh.full_bar[a]);
      last_it[a] = it;
    }
    if (ok && first) {  // the piece's query block, once its first key tile is on its way
      if (!q_waited) {
        q_waited = true;
        if (!qwait()) {
          *abort = 1;
          ok = false;
          break;
        }
      }
      ok = mbar_wait(&sh.q_empty, (pc & 1) ^ 1, abort, p.flags, p.wait_ns);
      if (ok) {
        mbar_arrive_expect_tx(&sh.q_full, kQBytes);
        const int qrow = kSparse ? c.row : c.row * S + cx.s;
        for (int a = 0; a < kSlots; ++a) tma_load_2d(cx.sQ + a * kQAtomBytes, &p.mQ, 64 * a, qrow * kH, &sh.q_full);
        last_q = pc;
      }
    }
    ++it;
    c.next(p, cx.ts, cx.NR, cx.N, cx.g, cx.s);
  }
  // Never leave with copies in flight: wait for the last load of each slot.
  volatile int no_abort = 0;
  const long long drain_ns = p.wait_ns > kDrainNs ? p.wait_ns : kDrainNs;
  for (int a = 0; a < kSlots; ++a)
    if (last_it[a] >= 0) mbar_wait(&sh.full_bar[a], last_it[a] & 1, &no_abort, p.flags, drain_ns);
  if (last_q >= 0) mbar_wait(&sh.q_full, last_q & 1, &no_abort, p.flags, drain_ns);
}

// ------------------------------------------------------------ MMA issuer (warp 1; lane 0 issues)
// kStream: the CTA streams several tiles; the score product then runs from one
// lane's unrolled loop (less per-atom overhead), else from a compact
// warp-wide loop whose smaller code costs less in a launch that runs it once.
template <bool kSparse, bool kStream>
__device__ __forceinline__ void attn_mma(const AttnParams& p, AttnShared& sh, const AttnCtx& cx) {
  volatile int* abort = &sh.abort_flag;
  const int lane = threadIdx.x & 31;
  const int mb0 = cx.mb0, mb1 = cx.mb1;
  const uint32_t tmem = cx.tmem;
  const uint32_t idS = idesc_bf16_f32(128, 64, 0, 0);
  const uint32_t idO = idesc_bf16_f32(128, 64, 1, 1);
  const uint32_t kv0 = smem_u32(cx.sKV), q0 = smem_u32(cx.sQ);
  // Operand descriptors of the first K step; a later step or atom adds its
  // byte offset / 16 to the start-address field (shared-memory addresses stay
  // below 256 KB, so the 14-bit field never carries).  The issuing thread then
  // spends a few instructions per MMA.
  const uint64_t dS0 = smem_desc_sw128(kv0, 16, 1024);                     // score A: key atoms, K-major
  const uint64_t dQ0 = smem_desc_sw128(q0, 16, 1024);                      // score B: query atoms
  const uint64_t dO0 = smem_desc_sw128(kv0, kSlotBytes, 1024);             // value A: latent atoms, MN-major
  const uint64_t dP0 = smem_desc_sw128(kv0 + 8 * kSlotBytes, kSlotBytes, 1024);  // value B: P^T, MN-major
  TileCursor<kSparse> c;
  c.start(p, cx.ts, cx.NR, cx.N, cx.g, cx.s, cx.row0);
  int it = 0, pc = -1;
  bool ok = true, issued = false;
  auto wait = [&](uint64_t* bar, uint32_t par) -> bool {
    const bool r = mbar_wait(bar, par, abort, p.flags, p.wait_ns);
    return __all_sync(0xffffffffu, r);
  };
  while (ok && c.live) {
    const bool first = c.first();
    // keys of this tile, read now so that the load overlaps the waits below
    const int ksteps = (tile_keys<kSparse>(p, c.row, cx.s, c.k) + 15) >> 4;
    if (first) {
      ++pc;
      ok = wait(&sh.q_full, pc & 1);
    }
    ok = ok && wait(&sh.s_free, (it & 1) ^ 1);
    if (!ok) break;
    tc_fence_after();
    // The score product.
    if constexpr (!kStream) {  // the whole warp waits for each atom, lane 0 issues
      for (int a = 0; a < kSlots && ok; ++a) {
        ok = wait(&sh.full_bar[a], it & 1);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint64_t da = dS0 + (uint64_t)(a * (kSlotBytes >> 4));
          const uint64_t db = dQ0 + (uint64_t)(a * (kQAtomBytes >> 4));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_bf16(tmem + kTmemS, da + 2 * kk, db + 2 * kk, idS, (a | kk) != 0 ? 1u : 0u);
        }
        __syncwarp();
        issued = true;
      }
    } else {
      // Lane 0 alone waits for each atom and issues its MMAs (the other lanes
      // wait at the warp sync), then shares the outcome.  The atom loop is
      // unrolled; the descriptors advance atom by atom from a base the
      // compiler cannot see through, so that it does not keep all nine atoms'
      // descriptors live (in registers or spilled) across tiles.
      int sok = 1;
      if (lane == 0) {
        uint64_t da = dS0, db = dQ0;
        asm volatile("" : "+l"(da), "+l"(db));
#pragma unroll
        for (int a = 0; a < kSlots; ++a) {
          if (!mbar_wait(&sh.full_bar[a], it & 1, abort, p.flags, p.wait_ns)) {
            sok = 0;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_bf16(tmem + kTmemS, da + 2 * kk, db + 2 * kk, idS, (a | kk) != 0 ? 1u : 0u);
          da += kSlotBytes >> 4;
          db += kQAtomBytes >> 4;
          issued = true;
        }
      }
      ok = __shfl_sync(0xffffffffu, sok, 0) != 0;
      issued = __shfl_sync(0xffffffffu, issued ? 1 : 0, 0) != 0;
    }
    if (!ok) break;
    if (lane == 0) {
      mma_commit(&sh.s_full);
      if (c.last()) mma_commit(&sh.q_empty);
    }
    __syncwarp();
    ok = wait(&sh.p_full, it & 1);
    if (!ok) break;
    tc_fence_after();
    if (lane == 0) {
      // latent atoms of the blocks another part owns: free once the score product retired
      for (int m = 0; m < 4; ++m)
        if (m < mb0 || m >= mb1) mma_commit(&sh.empty_bar[2 * m]);
      for (int m = mb0; m < mb1; ++m) {
        const uint64_t da = dO0 + (uint64_t)(2 * m * (kSlotBytes >> 4));
        const uint32_t dt = tmem + kTmemO + 64 * m;
        if (ksteps == kTile / 16) {  // a full tile: the issue loop unrolled
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_bf16(dt, da + 128 * kk, dP0 + 128 * kk, idO, (kk > 0 || !first) ? 1u : 0u);
        } else {
          for (int kk = 0; kk < ksteps; ++kk)
            mma_bf16(dt, da + 128 * kk, dP0 + 128 * kk, idO, (kk > 0 || !first) ? 1u : 0u);
        }
        mma_commit(&sh.empty_bar[2 * m]);  // latent atoms 2m, 2m + 1
        // a piece's last tile: the epilogue may read this block while the next ones run
        if (c.last()) mma_commit(&sh.o_blk[m]);
      }
      mma_commit(&sh.empty_bar[8]);
    }
    __syncwarp();
    ++it;
    c.next(p, cx.ts, cx.NR, cx.N, cx.g, cx.s);
  }
  if (issued) {  // all MMAs retired before TMEM is released
    if (lane == 0) mma_commit(&sh.mma_done);
    __syncwarp();
    volatile int no_abort = 0;
    mbar_wait(&sh.mma_done, 0, &no_abort, p.flags, p.wait_ns > kDrainNs ? p.wait_ns : kDrainNs);
  }
  __syncwarp();
}

// ------------------------------------------------------------ softmax warps 2..9
template <bool kSparse>
__device__ __forceinline__ void attn_softmax(const AttnParams& p, AttnShared& sh, const AttnCtx& cx) {
  volatile int* abort = &sh.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.S;
  const int g = cx.g, s = cx.s, part = cx.part, mb0 = cx.mb0, mb1 = cx.mb1;
  const uint32_t tmem = cx.tmem;
  unsigned char* sKV = cx.sKV;
  const int tsm = threadIdx.x - 64;         // 0..255
  const int qd = warp & 3;                  // TMEM lane quadrant of this warp
  const int half = (warp - 2) >> 2;         // which 32 of the 64 query rows (heads) this warp covers
  const int col0 = 32 * half;
  const int trow = 32 * qd + lane;          // key row of the tile / latent row of an O^T block
  const uint32_t t_lane = (uint32_t)(32 * qd) << 16;
  const float c = p.c;
  TileCursor<kSparse> cur;
  cur.start(p, cx.ts, cx.NR, cx.N, g, s, cx.row0);
  int it = 0, slot = 0, pos = 0, nkeys = 0;
  const int32_t* srow = nullptr;
  bool ok = true, bad_idx = false;
  float lp[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) lp[i] = 0.f;

  // Partials of the CTA's piece number `pcs`: each 128-row block of O^T as
  // soon as its part of the piece's last value product retired (o_blk[m]
  // completes once per piece).
  int pcs = 0;
  auto epilogue = [&]() -> bool {
    float* op = p.o_part + (size_t)slot * kH * kDl;
    const uint32_t par = (uint32_t)(pcs++ & 1);
#pragma unroll 1
    for (int m = mb0; m < mb1; ++m) {
      const bool fail = !mbar_wait(&sh.o_blk[m], par, abort, p.flags, p.wait_ns);
      if (bar_red_or(1, kSoftThreads, fail)) return false;
      tc_fence_after();
      float w[32];
      tmem_ld32(tmem + t_lane + kTmemO + 64 * m + col0, w);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) op[(size_t)(col0 + i) * kDl + 128 * m + trow] = w[i];
    }
    tc_fence_before();
    transpose_reduce32<false>(lp, lane);
    sh.red_sum[qd][col0 + lane] = lp[0];
    const bool bad = bar_red_or(1, kSoftThreads, bad_idx);
    if (tsm < kH && part == 0) {  // every part holds the same m and l
      const float l = sh.red_sum[0][tsm] + sh.red_sum[1][tsm] + sh.red_sum[2][tsm] + sh.red_sum[3][tsm];
      float* ml = p.ml_part + ((size_t)slot * kH + tsm) * 2;
      ml[0] = sh.m_sh[tsm];
      ml[1] = bad ? __int_as_float(0x7fc00000) : l;
    }
    if (bad && tsm == 0 && part == 0) raise_flag(p.flags, MLA_DEV_BAD_INDEX);
    return true;
  };

  while (ok && cur.live) {
    const bool first = cur.first();
    if (first) {
      if (it > 0 && !epilogue()) {
        ok = false;
        break;
      }
      const int b = kSparse ? cur.row / S : cur.row;
      const int qs = kSparse ? cur.row % S : s;
      pos = p.T[b] - S + qs;
      nkeys = kSparse ? p.nsel[cur.row] : pos + 1;
      srow = kSparse ? p.sel + (size_t)cur.row * p.topk : nullptr;
      slot = kSparse ? g + cur.row : (g + cur.row) * S + s;
      bad_idx = false;
#pragma unroll
      for (int i = 0; i < 32; ++i) lp[i] = 0.f;
    }
    // A failed wait is decided jointly by the softmax threads (bar.red), so
    // that no thread is left waiting at a barrier the others quit.
    bool fail = !mbar_wait(&sh.s_full, it & 1, abort, p.flags, p.wait_ns);
    if (bar_red_or(1, kSoftThreads, fail)) {
      ok = false;
      break;
    }
    tc_fence_after();
    float v[32];
    tmem_ld32(tmem + t_lane + kTmemS + col0, v);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive_warp(&sh.s_free);
    const int j = cur.k * kTile + trow;
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
      for (int i = 0; i < 32; ++i) v[i] = -INFINITY;
    }
    // The running max of a head moves only when the tile's max exceeds it by
    // more than kTau (lazy rescale).  Past a piece's first tile that is rare,
    // and one OR over the threads tells whether any head's does: only then is
    // the tile max reduced and the running max updated.
    bool slow = first;
    if (!first) {
      bool ex = false;
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 mo = *reinterpret_cast<const float4*>(&sh.m_sh[col0 + i]);
        ex = ex || v[i] * c > mo.x + kTau || v[i + 1] * c > mo.y + kTau || v[i + 2] * c > mo.z + kTau ||
             v[i + 3] * c > mo.w + kTau;
      }
      slow = bar_red_or(2, kSoftThreads, ex);
    }
    bool rescale = false;
    if (slow) {
      float mx[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) mx[i] = v[i];
      transpose_reduce32<true>(mx, lane);
      sh.red_max[qd][col0 + lane] = mx[0];
      named_barrier(1, kSoftThreads);
      bool need = false;
      if (tsm < kH) {
        const float tmax =
            fmaxf(fmaxf(sh.red_max[0][tsm], sh.red_max[1][tsm]), fmaxf(sh.red_max[2][tsm], sh.red_max[3][tsm]));
        const float cand = tmax * c;
        const float mo = first ? -INFINITY : sh.m_sh[tsm];
        float mn = mo, al = 1.f;
        if (cand > mo + kTau) {
          mn = cand;
          al = exp2f(mo - mn);
        }
        sh.m_sh[tsm] = mn;
        sh.alpha_sh[tsm] = al;
        need = !first && al != 1.f;
      }
      rescale = bar_red_or(2, kSoftThreads, need);
    }
    // probabilities (bf16, the value-product operand) and their row sums
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const float4 mu = *reinterpret_cast<const float4*>(&sh.m_sh[col0 + i]);
      pk[i / 2] = pack_bf16(exp2f(fmaf(v[i + 0], c, -mu.x)), exp2f(fmaf(v[i + 1], c, -mu.y)));
      pk[i / 2 + 1] = pack_bf16(exp2f(fmaf(v[i + 2], c, -mu.z)), exp2f(fmaf(v[i + 3], c, -mu.w)));
    }
    if (rescale) {
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 al = *reinterpret_cast<const float4*>(&sh.alpha_sh[col0 + i]);
        lp[i + 0] *= al.x;
        lp[i + 1] *= al.y;
        lp[i + 2] *= al.z;
        lp[i + 3] *= al.w;
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      __nv_bfloat162 t = *reinterpret_cast<__nv_bfloat162*>(&pk[i]);
      const float2 f = __bfloat1622float2(t);
      lp[2 * i] += f.x;
      lp[2 * i + 1] += f.y;
    }
    // P^T row into the rope atom's slot (its score product is done): a
    // 128-byte row per key, 16-byte chunks XOR-swizzled by row
    unsigned char* prow = sKV + 8 * kSlotBytes + trow * 128;
    const int cbase = col0 >> 3;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const uint4 val = make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      *reinterpret_cast<uint4*>(prow + (((cbase + cc) ^ (trow & 7)) << 4)) = val;
    }
    // Masked key rows inside the value product's last 16-key step: their
    // probability is 0, but the latent row must be finite too.
    const int z1 = (cur.k * kTile + kTile <= nkeys) ? kTile : (((nkeys - cur.k * kTile) + 15) & ~15);
    if (!valid && trow < z1) {
#pragma unroll
      for (int a = 4 * half; a < 4 * half + 4; ++a) {
        unsigned char* lr = sKV + a * kSlotBytes + trow * 128;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) *reinterpret_cast<uint4*>(lr + 16 * cc) = make_uint4(0, 0, 0, 0);
      }
    }
    if (rescale) {  // (never on a piece's first tile)
      // O^T is stable here: the MMA thread committed s_full for this tile
      // after it issued the previous value product, and a commit tracks every
      // MMA that thread issued before it; this tile's value product waits for
      // p_full.
#pragma unroll 1
      for (int m = mb0; m < mb1; ++m) {
        float w[32];
        tmem_ld32(tmem + t_lane + kTmemO + 64 * m + col0, w);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 al = *reinterpret_cast<const float4*>(&sh.alpha_sh[col0 + i]);
          w[i] *= al.x;
          w[i + 1] *= al.y;
          w[i + 2] *= al.z;
          w[i + 3] *= al.w;
        }
        tmem_st32(tmem + t_lane + kTmemO + 64 * m + col0, w);
      }
      tmem_wait_st();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive_warp(&sh.p_full);
    ++it;
    cur.next(p, cx.ts, cx.NR, cx.N, g, s);
  }
  if (ok && it > 0) epilogue();
}

}  // namespace
}  // namespace mla
