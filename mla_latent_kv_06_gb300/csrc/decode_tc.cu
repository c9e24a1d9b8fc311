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
//                warp 1 issues the MMAs, warps 2-9 run the online softmax
//                (one key row and 32 heads per thread) and write the
//                per-split (m, l, O) partials.
//  3. combine  : log-sum-exp merge of the splits, then out = W_UV clat / l.
// More than 8 query rows: the absorb and the W_UV lift run as tcgen05 GEMMs
// (gemm_tc.cu) and merge_kernel replaces the combine's merge.
// The sparse variant first gathers each query's selected [Lc | Rc] rows into
// a contiguous staging buffer (row-major, 576 values per key, zero past nsel),
// so that its attention pass uses the same 1024-byte-aligned tile loads.
// The FP8 latent cache (E4M3 codes, one scale) adds quant_q_kernel, which
// quantises the query rows, and attn8_kernel, the attention on kind::f8f6f4
// MMAs with two resident key tiles.
#include <cuda_fp8.h>

#include <atomic>
#include <cmath>

#include "attn_core.cuh"
#include "decode_tc.h"
#include "gemm_tc.h"
#include "sm100.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace sm100;


// Two E4M3 codes of (lo, hi), lo in the low byte (the lower address).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// ===========================================================================
// Attention kernel: the pass of attn_core.cuh as its own launch, chained by
// programmatic dependent launch behind the absorb kernel (only the query-block
// loads wait for it; the key tiles stream in meanwhile).
// ===========================================================================
template <bool kSparse, bool kPaged = false, bool kStream = false>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  __shared__ AttnShared sh;
  __shared__ int plan_ts[kPlanMax + 1];
  __shared__ int plan_wsum[kAttnThreads / 32];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.S;
  // blockIdx.x = piece row * qsplit + latent part; the part owns O^T blocks [mb0, mb1)
  const int part = (int)blockIdx.x % p.qsplit, brow = (int)blockIdx.x / p.qsplit;

  if (threadIdx.x == 0) {
    attn_init_barriers(sh);
    fence_mbar_init();
    prefetch_tensormap(&p.mQ);
    prefetch_tensormap(&p.mL);
    prefetch_tensormap(&p.mR);
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // The combine kernel may start now: it only prefetches W_UV before waiting
  // for this grid to finish.
  grid_dep_launch();

  // Tile plan.  Built here from T / nsel (kernel inputs, ready at launch)
  // so that the key tiles can stream in while the absorb kernel still runs;
  // only the qcat loads wait for it.  Very long batches use the absorb
  // kernel's copy of the same plan.
  AttnCtx cx;
  cx.NR = kSparse ? p.B * S : p.B;
  const bool local_plan = cx.NR <= kPlanMax;
  cx.ts = p.tile_start;
  if (local_plan) {
    attn_local_plan<kSparse>(p, cx.NR, plan_ts, plan_wsum);
    cx.ts = plan_ts;
  } else {
    grid_dep_wait();
  }
  cx.N = cx.ts[cx.NR];
  cx.g = kSparse ? brow : brow / S;
  cx.s = kSparse ? 0 : brow % S;
  cx.part = part;
  cx.mb0 = part * (4 / p.qsplit);
  cx.mb1 = cx.mb0 + 4 / p.qsplit;
  cx.row0 = first_row(cx.ts, cx.NR, chunk_begin(cx.N, cx.g, p.G));
  cx.sQ = smem;
  cx.sKV = smem + kQBytes;
  cx.tmem = sh.tmem_base;

  if (warp == 0) {
    if (lane == 0)
      attn_producer<kSparse, kPaged>(p, sh, cx, [&]() -> bool {
        if (local_plan) grid_dep_wait();  // qcat comes from the absorb kernel
        return true;
      });
    __syncwarp();
  } else if (warp == 1) {
    attn_mma<kSparse, kStream>(p, sh, cx);
  } else {
    attn_softmax<kSparse>(p, sh, cx);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(cx.tmem, kTmemCols);
  }
}

// ===========================================================================
// FP8 query quantiser: one warp per query row (r, h) of qcat.  The 512
// absorbed values become E4M3 codes with the row's scale sq = amax / 448; the
// 64 rope values become bf16 divided by lat_scale * sq, so that one fp32
// accumulator of the FP8 attention holds (qabs . Lc + q_rot . Rc) / (lat_scale
// * sq); fh[row] = c * lat_scale * sq turns it back into the score in log2
// units.  Output rows of 640 bytes: the codes, then the rope values.
// ===========================================================================
struct QuantParams {
  const __nv_bfloat16* qcat;  // [rows, 576]
  unsigned char* q8;          // [rows, 640]
  float* fh;                  // [rows]
  int rows;
  float c, lat_scale;
};

__global__ void __launch_bounds__(256) quant_q_kernel(const QuantParams p) {
  grid_dep_wait();  // qcat comes from the absorb kernels
  grid_dep_launch();
  const int w = (int)((blockIdx.x * 256u + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  if (w >= p.rows) return;
  const __nv_bfloat16* src = p.qcat + (size_t)w * kDc;
  uint4 raw[2];
  raw[0] = *reinterpret_cast<const uint4*>(src + 16 * lane);
  raw[1] = *reinterpret_cast<const uint4*>(src + 16 * lane + 8);
  const uint32_t rp = *reinterpret_cast<const uint32_t*>(src + kDl + 2 * lane);
  float v[16];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw[h]);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 f = __bfloat1622float2(b2[t]);
      v[8 * h + 2 * t] = f.x;
      v[8 * h + 2 * t + 1] = f.y;
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sq = amax > 0.f ? amax * (1.f / 448.f) : 1.f;
  const float inv = amax > 0.f ? 448.f / amax : 1.f;
  uint32_t code[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    code[i] = e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv) | (e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv) << 16);
  unsigned char* dst = p.q8 + (size_t)w * kQ8Row;
  *reinterpret_cast<uint4*>(dst + 16 * lane) = make_uint4(code[0], code[1], code[2], code[3]);
  const float rs = 1.f / (p.lat_scale * sq);
  __nv_bfloat162 r2 = *reinterpret_cast<const __nv_bfloat162*>(&rp);
  const float2 rf = __bfloat1622float2(r2);
  r2 = __floats2bfloat162_rn(rf.x * rs, rf.y * rs);
  *reinterpret_cast<__nv_bfloat162*>(dst + kDl + 4 * lane) = r2;  // bytes 512.. : the rope values
  if (lane == 0) p.fh[w] = p.c * p.lat_scale * sq;
}

// ===========================================================================
// FP8 attention kernel (latent cache of E4M3 codes with one cache scale).
//
// The products of attn_kernel on kind::f8f6f4 MMAs (32 codes of K per
// instruction: half the instructions per tile):
//   S^T[128 keys x 64 rows]  = [Lc codes | Rc] tile x q8^T   (K = 512 codes, then 64 bf16)
//   O^T[512 x 64 rows]      += Lc codes^T x P^T                (K = keys, P as E4M3 codes)
// Half-size tiles leave room for two key-tile buffers, and TMEM holds two score
// accumulators: the MMA warp issues the score product of tile j before the
// value product of tile j - 1, so the tensor pipe computes the next scores
// while the softmax warps turn the current ones into probabilities, and tile
// j + 1 loads while tile j is in use.  The row sum l stays fp32; the partial's
// l is divided by lat_scale, which puts the cache scale back.
// ===========================================================================
// Query rows row0 .. row0 + 63 of qcat (one piece: 64 heads) into the FP8
// query atoms: softmax warp w (0..7) takes heads 8w .. 8w + 7, lane L the 16
// absorbed values 16L .. 16L + 15 and the rope pair 2L, 2L + 1 of each.  The
// arithmetic is quant_q_kernel's; the bytes land where a 128-byte-swizzled TMA
// load of the 640-byte quantised rows puts them (16-byte chunk c of row r at
// chunk c ^ (r & 7)).
// All eight rows are loaded before the first store: the stores go through
// generic pointers, which the compiler cannot separate from the loads, so
// loads placed after them would each wait a full L2 round trip.
__device__ __forceinline__ void quantise_query_rows(const AttnParams& p, size_t row0, int w, int lane,
                                                    unsigned char* sQ8, float* fh) {
  uint4 raw8[8][2];
  uint32_t rp8[8];
#pragma unroll
  for (int hh = 0; hh < 8; ++hh) {
    const __nv_bfloat16* src = p.qcat + (row0 + 8 * w + hh) * kDc;
    raw8[hh][0] = *reinterpret_cast<const uint4*>(src + 16 * lane);
    raw8[hh][1] = *reinterpret_cast<const uint4*>(src + 16 * lane + 8);
    rp8[hh] = *reinterpret_cast<const uint32_t*>(src + kDl + 2 * lane);
  }
#pragma unroll
  for (int hh = 0; hh < 8; ++hh) {
    const int h = 8 * w + hh;
    const uint32_t rp = rp8[hh];
    float v[16];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw8[hh][k]);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 f = __bfloat1622float2(b2[t]);
        v[8 * k + 2 * t] = f.x;
        v[8 * k + 2 * t + 1] = f.y;
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sq = amax > 0.f ? amax * (1.f / 448.f) : 1.f;
    const float inv = amax > 0.f ? 448.f / amax : 1.f;
    uint32_t code[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      code[i] = e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv) | (e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv) << 16);
    // codes 16L .. 16L+15: atom L / 8, chunk L % 8 of row h
    const int c = lane & 7;
    *reinterpret_cast<uint4*>(sQ8 + (lane >> 3) * kQAtomBytes + h * 128 + ((c ^ (h & 7)) << 4)) =
        make_uint4(code[0], code[1], code[2], code[3]);
    // rope pair: bytes 4L .. 4L+3 of row h of the bf16 atom (chunk L / 4)
    const float rs = 1.f / (p.lat_scale * sq);
    __nv_bfloat162 r2 = *reinterpret_cast<const __nv_bfloat162*>(&rp);
    const float2 rf = __bfloat1622float2(r2);
    r2 = __floats2bfloat162_rn(rf.x * rs, rf.y * rs);
    const int rc = lane >> 2;
    *reinterpret_cast<__nv_bfloat162*>(sQ8 + 4 * kQAtomBytes + h * 128 + ((rc ^ (h & 7)) << 4) + 4 * (lane & 3)) = r2;
    if (lane == 0) fh[h] = p.c * p.lat_scale * sq;
  }
}

// kQuantIn: the softmax warps quantise each piece's query rows from qcat
// themselves (as quant_q_kernel does, one warp per head) and write the codes
// and rope values into the query atoms, in the layout a 128-byte-swizzled TMA
// load of the quantised rows would give; the few-row path takes this form,
// which saves the quantiser's launch and hand-over.
template <bool kQuantIn, bool kStream = false>
__global__ void __launch_bounds__(kAttnThreads, 1) attn8_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  unsigned char* sQ8 = smem;
  unsigned char* sKV = smem + kQ8Bytes;  // buffer u at sKV + u * kTile8Bytes

  __shared__ uint64_t full_bar[2][kAtoms8], empty_bar[2][kAtoms8];
  __shared__ uint64_t q_full, q_empty, s_full[2], s_free[2], p_full, o_done, mma_done, o_blk[4];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ __align__(16) float red_max[4][kH];
  __shared__ __align__(16) float red_sum[4][kH];
  __shared__ __align__(16) float m_sh[kH];
  __shared__ __align__(16) float alpha_sh[kH];
  __shared__ __align__(16) float fh_sh[2][kH];
  __shared__ int plan_ts[kPlanMax + 1];
  __shared__ int plan_wsum[kAttnThreads / 32];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.S;
  const int part = (int)blockIdx.x % p.qsplit, brow = (int)blockIdx.x / p.qsplit;
  const int g = brow / S, s = brow % S;
  const int mb0 = part * (4 / p.qsplit), mb1 = mb0 + 4 / p.qsplit;

  if (threadIdx.x == 0) {
    for (int u = 0; u < 2; ++u)
      for (int a = 0; a < kAtoms8; ++a) {
        mbar_init(&full_bar[u][a], 1);
        mbar_init(&empty_bar[u][a], 1);
      }
    mbar_init(&q_full, kQuantIn ? kSoftWarps : 1);
    mbar_init(&q_empty, 1);
    for (int u = 0; u < 2; ++u) {
      mbar_init(&s_full[u], 1);
      mbar_init(&s_free[u], kSoftWarps);
    }
    mbar_init(&p_full, kSoftWarps);
    mbar_init(&o_done, 1);
    for (int m = 0; m < 4; ++m) mbar_init(&o_blk[m], 1);
    mbar_init(&mma_done, 1);
    abort_flag = 0;
    fence_mbar_init();
    if (!kQuantIn) prefetch_tensormap(&p.mQ);
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
  grid_dep_launch();

  // Tile plan, as in attn_kernel.
  const int NR = p.B;
  const bool local_plan = NR <= kPlanMax;
  const int32_t* ts = p.tile_start;
  if (local_plan) {
    int carry = 0;
    for (int base = 0; base < NR; base += kAttnThreads) {
      const int r = base + threadIdx.x;
      int x = r < NR ? row_tiles<false>(p, r) : 0;
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
    if (lane == 0) {
      const uint64_t pol_once = l2_policy_evict_first();
      TileCursor<false> c;
      c.start(p, ts, NR, N, g, s, row0);
      int it = 0, pc = -1, last_it[2][kAtoms8], last_q = -1;
      for (int u = 0; u < 2; ++u)
        for (int a = 0; a < kAtoms8; ++a) last_it[u][a] = -1;
      bool ok = true, dep_waited = !local_plan;
      // First cache row of a tile (the tile's 128 rows lie in one page).
      auto tile_y = [&](const TileCursor<false>& t, bool* bad_page) -> int {
        *bad_page = false;
        if (!p.pages.table) return t.row * p.kv_rows + t.k * kTile;
        return (int)cache_row(p.pages, t.row, p.T_cap, t.k * kTile, bad_page);
      };
      while (ok && c.live) {
        const bool first = c.first();
        if (first) ++pc;
        bool bad_page;
        const int y = tile_y(c, &bad_page);
        if (bad_page) raise_flag(p.flags, MLA_DEV_BAD_INDEX);
        const int u = it & 1;
        const uint32_t par = ((it >> 1) & 1) ^ 1;
        unsigned char* tile = sKV + u * kTile8Bytes;
        for (int a = 0; a < kAtoms8 && ok; ++a) {
          ok = mbar_wait(&empty_bar[u][a], par, abort, p.flags, p.wait_ns);
          if (!ok) break;
          mbar_arrive_expect_tx(&full_bar[u][a], kSlotBytes);
          const CUtensorMap* map = a < 4 ? &p.mL : &p.mR;
          const int x = a < 4 ? 128 * a : 0;
          if (p.read_once) tma_load_2d_hint(tile + a * kSlotBytes, map, x, y, &full_bar[u][a], pol_once);
          else tma_load_2d(tile + a * kSlotBytes, map, x, y, &full_bar[u][a]);
          last_it[u][a] = it;
        }
        if (!kQuantIn && ok && first) {  // the piece's quantised query block
          if (!dep_waited) {
            grid_dep_wait();  // q8 comes from the quantiser
            dep_waited = true;
          }
          ok = mbar_wait(&q_empty, (pc & 1) ^ 1, abort, p.flags, p.wait_ns);
          if (ok) {
            mbar_arrive_expect_tx(&q_full, kQ8Bytes);
            const int qrow = c.row * S + s;
            for (int a = 0; a < kAtoms8; ++a) tma_load_2d(sQ8 + a * kQAtomBytes, &p.mQ, 128 * a, qrow * kH, &q_full);
            last_q = pc;
          }
        }
        ++it;
        c.next(p, ts, NR, N, g, s);
      }
      // Never leave with copies in flight: wait for the last load of each slot.
      volatile int no_abort = 0;
      const long long drain_ns = p.wait_ns > kDrainNs ? p.wait_ns : kDrainNs;
      for (int u = 0; u < 2; ++u)
        for (int a = 0; a < kAtoms8; ++a)
          if (last_it[u][a] >= 0)
            mbar_wait(&full_bar[u][a], (last_it[u][a] >> 1) & 1, &no_abort, p.flags, drain_ns);
      if (last_q >= 0) mbar_wait(&q_full, last_q & 1, &no_abort, p.flags, drain_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (whole warp waits, lane 0 issues)
    const uint32_t idS = idesc_bf16_f32(128, 64, 0, 0);
    const uint32_t idS8 = idesc_e4m3_f32(128, 64, 0, 0);
    const uint32_t idO8 = idesc_e4m3_f32(128, 64, 1, 0);
    const uint32_t kv0 = smem_u32(sKV), q0 = smem_u32(sQ8);
    // First-step operand descriptors; a later step, atom or buffer adds its
    // byte offset / 16 (addresses stay below 256 KB: no carry out of the field).
    const uint64_t dS0 = smem_desc_sw128(kv0, 16, 1024);                    // score A, K-major
    const uint64_t dQ0 = smem_desc_sw128(q0, 16, 1024);                     // score B
    const uint64_t dV0 = smem_desc_sw128(kv0, kSlotBytes, 1024);            // value A, MN-major codes
    const uint64_t dP0 = smem_desc_sw128(kv0 + 4 * kSlotBytes, 16, 1024);   // value B: P^T codes, K-major
    TileCursor<false> c;
    c.start(p, ts, NR, N, g, s, row0);
    int it = 0, pc = -1;
    bool ok = true, issued = false;
    auto wait = [&](uint64_t* bar, uint32_t par) -> bool {
      const bool r = mbar_wait(bar, par, abort, p.flags, p.wait_ns);
      return __all_sync(0xffffffffu, r);
    };
    // Value product of tile j: O^T block m = latent atom m (MN-major, 32 keys =
    // 4 KB per step) x P^T (K-major codes in the tile's rope slot).
    auto value = [&](int j, int ksteps, bool firstj, bool lastj) -> bool {
      if (!wait(&p_full, j & 1)) return false;
      tc_fence_after();
      if (lane == 0) {
        const int u = j & 1;
        const uint64_t ub = (uint64_t)(u * (kTile8Bytes >> 4));
        for (int m = 0; m < 4; ++m)
          if (m < mb0 || m >= mb1) mma_commit(&empty_bar[u][m]);  // another part's block: free now
        for (int m = mb0; m < mb1; ++m) {
          const uint64_t da = dV0 + ub + (uint64_t)(m * (kSlotBytes >> 4));
          const uint64_t db = dP0 + ub;
          const uint32_t dt = tmem + kTmemO8 + 64 * m;
          if (ksteps == kTile / 32) {  // a full tile: the issue loop unrolled
#pragma unroll
            for (int kk = 0; kk < kTile / 32; ++kk)
              mma_f8(dt, da + 256 * kk, db + 2 * kk, idO8, (kk > 0 || !firstj) ? 1u : 0u);
          } else {
            for (int kk = 0; kk < ksteps; ++kk) mma_f8(dt, da + 256 * kk, db + 2 * kk, idO8, (kk > 0 || !firstj) ? 1u : 0u);
          }
          mma_commit(&empty_bar[u][m]);
          // a piece's last tile: the epilogue may read this block while the next ones run
          if (lastj) mma_commit(&o_blk[m]);
        }
        mma_commit(&empty_bar[u][4]);
        mma_commit(&o_done);
      }
      __syncwarp();
      return true;
    };
    bool pend = false, pend_first = false, pend_last = false;
    int pend_it = 0, pend_ks = 0;
    while (ok && c.live) {
      const bool first = c.first();
      const int ksteps = (tile_keys<false>(p, c.row, s, c.k) + 31) >> 5;
      const int u = it & 1;
      if (first) {
        ++pc;
        ok = wait(&q_full, pc & 1);
      }
      ok = ok && wait(&s_free[u], ((it >> 1) & 1) ^ 1);
      if (!ok) break;
      tc_fence_after();
      const uint64_t ub = (uint64_t)(u * (kTile8Bytes >> 4));
      if constexpr (!kStream) {  // the whole warp waits for each atom, lane 0 issues
        for (int a = 0; a < kAtoms8 && ok; ++a) {
          ok = wait(&full_bar[u][a], (it >> 1) & 1);
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            // 32 bytes of K per instruction: 32 codes, or 16 bf16 for the rope atom
            const uint64_t da = dS0 + ub + (uint64_t)(a * (kSlotBytes >> 4));
            const uint64_t db = dQ0 + (uint64_t)(a * (kQAtomBytes >> 4));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              if (a < 4) mma_f8(tmem + kTmemS + 64 * u, da + 2 * kk, db + 2 * kk, idS8, (a | kk) != 0 ? 1u : 0u);
              else mma_bf16(tmem + kTmemS + 64 * u, da + 2 * kk, db + 2 * kk, idS, 1u);
            }
          }
          __syncwarp();
          issued = true;
        }
      } else {
        // Streaming CTAs: lane 0 alone waits for each atom and issues its MMAs
        // from an unrolled loop, then shares the outcome; the descriptors
        // advance from a base the compiler cannot see through.
        int sok = 1;
        if (lane == 0) {
          uint64_t da = dS0 + ub, db = dQ0;
          asm volatile("" : "+l"(da), "+l"(db));
#pragma unroll
          for (int a = 0; a < kAtoms8; ++a) {
            if (!mbar_wait(&full_bar[u][a], (it >> 1) & 1, abort, p.flags, p.wait_ns)) {
              sok = 0;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              if (a < 4) mma_f8(tmem + kTmemS + 64 * u, da + 2 * kk, db + 2 * kk, idS8, (a | kk) != 0 ? 1u : 0u);
              else mma_bf16(tmem + kTmemS + 64 * u, da + 2 * kk, db + 2 * kk, idS, 1u);
            }
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
        mma_commit(&s_full[u]);
        if (c.last()) mma_commit(&q_empty);
      }
      __syncwarp();
      // the previous tile's value product, queued behind this tile's scores
      if (pend && !(ok = value(pend_it, pend_ks, pend_first, pend_last))) break;
      pend = true;
      pend_it = it;
      pend_ks = ksteps;
      pend_first = first;
      pend_last = c.last();
      ++it;
      c.next(p, ts, NR, N, g, s);
    }
    if (ok && pend) value(pend_it, pend_ks, pend_first, pend_last);
    if (issued) {  // all MMAs retired before TMEM is released
      if (lane == 0) mma_commit(&mma_done);
      __syncwarp();
      volatile int no_abort = 0;
      mbar_wait(&mma_done, 0, &no_abort, p.flags, p.wait_ns > kDrainNs ? p.wait_ns : kDrainNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps 2..9
    const int tsm = threadIdx.x - 64;         // 0..255
    const int qd = warp & 3;                  // TMEM lane quadrant of this warp
    const int half = (warp - 2) >> 2;         // which 32 of the 64 query rows this warp covers
    const int col0 = 32 * half;
    const int trow = 32 * qd + lane;          // key row of the tile / latent row of an O^T block
    const uint32_t t_lane = (uint32_t)(32 * qd) << 16;
    TileCursor<false> cur;
    cur.start(p, ts, NR, N, g, s, row0);
    int it = 0, slot = 0, nkeys = 0, spc = -1;
    bool ok = true, dep_waited = false;
    float lp[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) lp[i] = 0.f;

    // o_blk[m] completes once per piece, with the piece's last value product:
    // the epilogue of piece pcs waits for phase pcs.  The next piece's cannot
    // complete before this epilogue ends (its value products wait for P).
    int pcs = 0;
    auto epilogue = [&]() -> bool {
      float* op = p.o_part + (size_t)slot * kH * kDl;
      const uint32_t par = (uint32_t)(pcs++ & 1);
#pragma unroll 1
      for (int m = mb0; m < mb1; ++m) {
        const bool fail = !mbar_wait(&o_blk[m], par, abort, p.flags, p.wait_ns);
        if (bar_red_or(1, kSoftThreads, fail)) return false;
        tc_fence_after();
        float w[32];
        tmem_ld32(tmem + t_lane + kTmemO8 + 64 * m + col0, w);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) op[(size_t)(col0 + i) * kDl + 128 * m + trow] = w[i];
      }
      tc_fence_before();
      transpose_reduce32<false>(lp, lane);
      red_sum[qd][col0 + lane] = lp[0];
      named_barrier(1, kSoftThreads);
      if (tsm < kH && part == 0) {  // every part holds the same m and l
        const float l = red_sum[0][tsm] + red_sum[1][tsm] + red_sum[2][tsm] + red_sum[3][tsm];
        float* ml = p.ml_part + ((size_t)slot * kH + tsm) * 2;
        ml[0] = m_sh[tsm];
        ml[1] = l / p.lat_scale;  // O^T sums codes: dividing l by lat_scale puts the scale back
      }
      return true;
    };

    while (ok && cur.live) {
      const bool first = cur.first();
      const int u = it & 1;
      if (first) {
        ++spc;
        if (kQuantIn) {
          // the piece's query block, once the previous piece's score products are done
          if (!dep_waited) {
            grid_dep_wait();  // qcat comes from the absorb kernel
            dep_waited = true;
          }
          const bool qfail = !mbar_wait(&q_empty, (spc & 1) ^ 1, abort, p.flags, p.wait_ns);
          if (bar_red_or(1, kSoftThreads, qfail)) {
            ok = false;
            break;
          }
          quantise_query_rows(p, (size_t)(cur.row * S + s) * kH, warp - 2, lane, sQ8, fh_sh[spc & 1]);
          fence_proxy_async_smem();
          mbar_arrive_warp(&q_full);
        }
        if (it > 0 && !epilogue()) {
          ok = false;
          break;
        }
        nkeys = p.T[cur.row] - S + s + 1;
        slot = (g + cur.row) * S + s;
#pragma unroll
        for (int i = 0; i < 32; ++i) lp[i] = 0.f;
        if (!kQuantIn) {
          if (!dep_waited) {
            grid_dep_wait();  // fh comes from the quantiser
            dep_waited = true;
          }
          if (tsm < kH) fh_sh[spc & 1][tsm] = p.fh[(size_t)(cur.row * S + s) * kH + tsm];
        }
      }
      bool fail = !mbar_wait(&s_full[u], (it >> 1) & 1, abort, p.flags, p.wait_ns);
      if (bar_red_or(1, kSoftThreads, fail)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float v[32];
      tmem_ld32(tmem + t_lane + kTmemS + 64 * u + col0, v);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive_warp(&s_free[u]);
      const int j = cur.k * kTile + trow;
      const bool valid = j < nkeys;
      if (!valid) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = -INFINITY;
      }
      const float* fh = fh_sh[spc & 1];
      // lazy rescale: past a piece's first tile, the tile max is reduced only
      // when some head's scores exceed its running max by more than kTau
      bool slow = first;
      if (!first) {
        bool ex = false;
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 mo = *reinterpret_cast<const float4*>(&m_sh[col0 + i]);
          const float4 f = *reinterpret_cast<const float4*>(&fh[col0 + i]);
          ex = ex || v[i] * f.x > mo.x + kTau || v[i + 1] * f.y > mo.y + kTau || v[i + 2] * f.z > mo.z + kTau ||
               v[i + 3] * f.w > mo.w + kTau;
        }
        slow = bar_red_or(2, kSoftThreads, ex);
      }
      bool rescale = false;
      if (slow) {
        float mx[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) mx[i] = v[i];
        transpose_reduce32<true>(mx, lane);
        red_max[qd][col0 + lane] = mx[0];
        named_barrier(1, kSoftThreads);
        bool need = false;
        if (tsm < kH) {
          const float tmax =
              fmaxf(fmaxf(red_max[0][tsm], red_max[1][tsm]), fmaxf(red_max[2][tsm], red_max[3][tsm]));
          const float cand = tmax * fh[tsm];
          const float mo = first ? -INFINITY : m_sh[tsm];
          float mn = mo, al = 1.f;
          if (cand > mo + kTau) {
            mn = cand;
            al = exp2f(mo - mn);
          }
          m_sh[tsm] = mn;
          alpha_sh[tsm] = al;
          need = !first && al != 1.f;
        }
        rescale = bar_red_or(2, kSoftThreads, need);
      }
      if (rescale) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 al = *reinterpret_cast<const float4*>(&alpha_sh[col0 + i]);
          lp[i + 0] *= al.x;
          lp[i + 1] *= al.y;
          lp[i + 2] *= al.z;
          lp[i + 3] *= al.w;
        }
      }
      // probabilities: fp32 row sums, E4M3 codes for the value product.  P^T
      // is K-major in the tile's rope slot: query row n holds the codes of
      // the 128 keys in one 128-byte row (rows in 1 KB groups of 8, 16-byte
      // chunks XOR-swizzled by n % 8); this thread writes byte trow of rows
      // col0 .. col0 + 31.
      unsigned char* tile = sKV + u * kTile8Bytes;
      unsigned char* pt = tile + 4 * kSlotBytes;
      const int kc = trow >> 4, kb = trow & 15;
      auto put = [&](int n, uint32_t code) {
        pt[(n >> 3) * 1024 + (n & 7) * 128 + ((kc ^ (n & 7)) << 4) + kb] = (unsigned char)code;
      };
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 mu = *reinterpret_cast<const float4*>(&m_sh[col0 + i]);
        const float4 f = *reinterpret_cast<const float4*>(&fh[col0 + i]);
        const float p0 = exp2f(fmaf(v[i], f.x, -mu.x)), p1 = exp2f(fmaf(v[i + 1], f.y, -mu.y));
        const float p2 = exp2f(fmaf(v[i + 2], f.z, -mu.z)), p3 = exp2f(fmaf(v[i + 3], f.w, -mu.w));
        lp[i] += p0;
        lp[i + 1] += p1;
        lp[i + 2] += p2;
        lp[i + 3] += p3;
        const uint32_t c01 = e4m3x2(p0, p1), c23 = e4m3x2(p2, p3);
        put(col0 + i, c01 & 0xFFu);
        put(col0 + i + 1, c01 >> 8);
        put(col0 + i + 2, c23 & 0xFFu);
        put(col0 + i + 3, c23 >> 8);
      }
      // Masked key rows inside the value product's last 32-key step: their
      // probability is 0, but the latent codes must be finite too.
      const int z1 = (cur.k * kTile + kTile <= nkeys) ? kTile : (((nkeys - cur.k * kTile) + 31) & ~31);
      if (!valid && trow < z1) {
#pragma unroll
        for (int a = 2 * half; a < 2 * half + 2; ++a) {
          unsigned char* lr = tile + a * kSlotBytes + trow * 128;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) *reinterpret_cast<uint4*>(lr + 16 * cc) = make_uint4(0, 0, 0, 0);
        }
      }
      if (rescale) {
        // O^T is stable once the previous value product retired.  Without a
        // rescale nothing here touches O^T, and the tensor pipe orders this
        // tile's value product after the previous one by itself.
        fail = !mbar_wait(&o_done, (it - 1) & 1, abort, p.flags, p.wait_ns);
        if (bar_red_or(2, kSoftThreads, fail)) {
          ok = false;
          break;
        }
        tc_fence_after();
        {
#pragma unroll 1
          for (int m = mb0; m < mb1; ++m) {
            float w[32];
            tmem_ld32(tmem + t_lane + kTmemO8 + 64 * m + col0, w);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float4 al = *reinterpret_cast<const float4*>(&alpha_sh[col0 + i]);
              w[i] *= al.x;
              w[i + 1] *= al.y;
              w[i + 2] *= al.z;
              w[i + 3] *= al.w;
            }
            tmem_st32(tmem + t_lane + kTmemO8 + 64 * m + col0, w);
          }
          tmem_wait_st();
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive_warp(&p_full);
      ++it;
      cur.next(p, ts, NR, N, g, s);
    }
    if (ok && it > 0) epilogue();
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
constexpr int kAbsCols = 128;     // W_UK columns per CTA
constexpr int kAbsRows = 8;       // query rows of the GEMV path (larger batches use the GEMM)
constexpr int kAbsGroups = kAbsThreads / (kAbsCols / 8);  // 16 row groups of 8-column threads

struct AbsorbParams {
  const __nv_bfloat16* q;     // [R, 64, Dn+64]
  const __nv_bfloat16* kv_b;  // [64, Dn+Dv, 512]
  const int32_t* T;
  const int32_t* nsel;
  __nv_bfloat16* qcat;  // [R, 64, 576]
  int32_t* tile_start;  // [NR + 1]
  int32_t* bad;         // [NR]
  int B, S, T_cap, Dn, Dv, topk, sparse;
  // L2 prefetch (small batches): the latent cache rows [0, T[b]) of every
  // sequence and the W_UV rows this CTA's combine counterpart will read
  const unsigned char* Lc;  // latent rows of lat_row_bytes bytes (bf16 or E4M3)
  const __nv_bfloat16* Rc;
  int lat_row_bytes;
  int prefetch;
  uint64_t turn[kDr / 2];  // rope_turns(rope_base^(-2j/qk_rope)), from the host
  unsigned int* flags;
  PageTable pages;
};

// Rotary part of query row r of head h, rotated to the row's own position.
__device__ __forceinline__ void rope_row(const AbsorbParams& p, int r, int h, int j) {
  const int Dq = p.Dn + kDr;
  const int b = r / p.S, s = r % p.S;
  const int Tb = p.T[b];
  const int pos = (Tb < p.S || Tb > p.T_cap) ? 0 : Tb - p.S + s;
  float sn, cs;
  rope_cs_turns(pos, p.turn[j], &cs, &sn);
  const __nv_bfloat16* qr = p.q + ((size_t)r * kH + h) * Dq + p.Dn;
  const float x0 = __bfloat162float(qr[2 * j]), x1 = __bfloat162float(qr[2 * j + 1]);
  __nv_bfloat16* dst = p.qcat + ((size_t)r * kH + h) * kDc + kDl;
  dst[j] = __float2bfloat16_rn(x0 * cs - x1 * sn);
  dst[kDr / 2 + j] = __float2bfloat16_rn(x1 * cs + x0 * sn);
}

// Rotary parts of rows x pairs e = tid, tid + nthr, ... (row e / 32, pair e % 32):
// eight pairs per thread at a time, their loads (T[b] and the two bf16 values)
// all in flight before the first rotation.
__device__ __forceinline__ void rope_rows(const AbsorbParams& p, int h, int tid, int nthr) {
  const int R = p.B * p.S, Dq = p.Dn + kDr, n = R * (kDr / 2);
  for (int e0 = tid; e0 < n; e0 += 8 * nthr) {
    uint32_t raw[8];
    int Tb[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + u * nthr;
      if (e < n) {
        const int r = e / (kDr / 2), j = e % (kDr / 2);
        raw[u] = *reinterpret_cast<const uint32_t*>(p.q + ((size_t)r * kH + h) * Dq + p.Dn + 2 * j);
        Tb[u] = p.T[r / p.S];
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + u * nthr;
      if (e < n) {
        const int r = e / (kDr / 2), j = e % (kDr / 2), s = r % p.S;
        const int pos = (Tb[u] < p.S || Tb[u] > p.T_cap) ? 0 : Tb[u] - p.S + s;
        float sn, cs;
        rope_cs_turns(pos, p.turn[j], &cs, &sn);
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[u]));
        __nv_bfloat16* dst = p.qcat + ((size_t)r * kH + h) * kDc + kDl;
        dst[j] = __float2bfloat16_rn(x.x * cs - x.y * sn);
        dst[kDr / 2 + j] = __float2bfloat16_rn(x.y * cs + x.x * sn);
      }
    }
  }
}

// Partial products of every query row with the thread's W_UK registers
// (rows grp + 16u, columns c8*8 .. c8*8+7), one row at a time.
template <int NV>
__device__ __forceinline__ void absorb_regs(const uint4 (&wv)[NV], const float* qn, int Dn, int grp, int nr,
                                            float* part, int c8) {
  for (int r = 0; r < nr; ++r) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      const float qv = qn[r * Dn + grp + kAbsGroups * u];
      const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&wv[u]);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 f = __bfloat1622float2(w2[t]);
        acc[2 * t] = fmaf(qv, f.x, acc[2 * t]);
        acc[2 * t + 1] = fmaf(qv, f.y, acc[2 * t + 1]);
      }
    }
    float4* d = reinterpret_cast<float4*>(part + ((size_t)grp * kAbsRows + r) * kAbsCols + c8 * 8);
    d[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    d[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// NV = qk_nope / 16: W_UK registers (16-byte vectors) per thread.  kQabs =
// false: the plan and the rotary part only (the GEMM forms qabs); a separate
// instantiation, so that the small-batch kernel carries only its own code.
template <int NV, bool kQabs = true, bool kPaged = false>
__global__ void __launch_bounds__(kAbsThreads, 2) absorb_kernel(const AbsorbParams p) {
  extern __shared__ __align__(128) unsigned char sm[];
  const int cb = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int Dn = p.Dn, Dq = Dn + kDr;
  const int R = p.B * p.S;
  // W_UK[h][:, cb*128 : cb*128+128] straight into registers: thread (grp, c8)
  // holds rows grp, grp+16, ... of columns c8*8 .. c8*8+7.  Under programmatic
  // serialization this kernel may start before the previous kernel of the
  // stream retires (for example the combine of an earlier call): the weights
  // are an input no kernel of this library writes, so their loads go out
  // first; everything else waits for that kernel.
  const int c8 = tid % (kAbsCols / 8), grp = tid / (kAbsCols / 8);
  uint4 wv[NV];
  if (kQabs) {
    const __nv_bfloat16* W = p.kv_b + (size_t)h * (Dn + p.Dv) * kDl + cb * kAbsCols + c8 * 8;
#pragma unroll
    for (int u = 0; u < NV; ++u) wv[u] = __ldg(reinterpret_cast<const uint4*>(W + (size_t)(grp + kAbsGroups * u) * kDl));
  }
  if (p.prefetch && tid == 0) {
    // Everything the later kernels of this call read streams from HBM now,
    // behind W_UK, in the order it is needed: 1/nblk of every sequence's
    // cache rows (the attention kernel), then W_UV rows (the combine).  It is
    // issued before the dependency wait: the kernel completes only once its
    // prefetches have landed, and the wait is time they can use.  A
    // prefetch changes no data; T and the page table are read here only to
    // place it (lengths clamped to [0, T_cap], pages checked against the
    // pool), so values an earlier kernel is still writing can at worst
    // prefetch the wrong rows.
    const int nblk = gridDim.x * gridDim.y, me = h * gridDim.x + cb;
    // Paged caches: units of 16 KB, nine per key tile (eight 16-row blocks of
    // latent rows, then the tile's rope rows), dealt round-robin to the CTAs.
    for (int b = 0, base = 0; kPaged && b < p.B; ++b) {
      const int Tb = min(max(p.T[b], 0), p.T_cap);
      const int units = (Tb + kTile - 1) / kTile * 9;
      for (int u = ((me - base) % nblk + nblk) % nblk; u < units; u += nblk) {
        bool bad_page = false;
        const long long row = cache_row(p.pages, b, p.T_cap, (u / 9) * kTile, &bad_page);
        if (bad_page) continue;
        const int part = u % 9;
        if (part < 8) l2_prefetch(p.Lc + (size_t)(row + 16 * part) * p.lat_row_bytes, 16 * p.lat_row_bytes);
        else l2_prefetch(p.Rc + (size_t)row * kDr, kTile * kDr * 2);
      }
      base += units;
    }
    for (int b = 0; !kPaged && b < p.B; ++b) {
      const int Tb = min(max(p.T[b], 0), p.T_cap);
      const size_t lb = (size_t)Tb * p.lat_row_bytes, rb = (size_t)Tb * kDr * 2;
      const size_t l0 = (lb * me / nblk) & ~(size_t)15, l1 = (lb * (me + 1) / nblk) & ~(size_t)15;
      const size_t r0 = (rb * me / nblk) & ~(size_t)15, r1 = (rb * (me + 1) / nblk) & ~(size_t)15;
      const unsigned char* lbase = p.Lc + (size_t)b * p.T_cap * p.lat_row_bytes;
      const unsigned char* rbase = reinterpret_cast<const unsigned char*>(p.Rc + (size_t)b * p.T_cap * kDr);
      if (l1 > l0) l2_prefetch(lbase + l0, (uint32_t)(l1 - l0));
      if (r1 > r0) l2_prefetch(rbase + r0, (uint32_t)(r1 - r0));
    }
    const __nv_bfloat16* wuv = p.kv_b + ((size_t)h * (p.Dn + p.Dv) + p.Dn + (size_t)cb * (p.Dv / gridDim.x)) * kDl;
    l2_prefetch(wuv, (uint32_t)(p.Dv / gridDim.x) * kDl * 2);
  }
  grid_dep_wait();
  grid_dep_launch();

  float* qn = reinterpret_cast<float*>(sm);      // [kAbsRows][Dn]
  float* part = qn + kAbsRows * Dn;               // [kAbsGroups][kAbsRows][kAbsCols]

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

  if constexpr (!kQabs) {  // rotary part only, every (row, pair) in parallel over the head's CTAs
    rope_rows(p, h, cb * kAbsThreads + tid, gridDim.x * kAbsThreads);
    return;
  }
  // R <= kAbsRows here (larger batches take the GEMM path)
  for (int e = tid; e < R * Dn; e += kAbsThreads) {
    const int rr = e / Dn, i = e % Dn;
    qn[rr * Dn + i] = __bfloat162float(p.q[((size_t)rr * kH + h) * Dq + i]);
  }
  __syncthreads();
  absorb_regs<NV>(wv, qn, Dn, grp, R, part, c8);
  __syncthreads();
  for (int e = tid; e < R * kAbsCols; e += kAbsThreads) {
    const int r = e / kAbsCols, col = e % kAbsCols;
    float v = 0.f;
#pragma unroll
    for (int k = 0; k < kAbsGroups; ++k) v += part[((size_t)k * kAbsRows + r) * kAbsCols + col];
    p.qcat[((size_t)r * kH + h) * kDc + cb * kAbsCols + col] = __float2bfloat16_rn(v);
  }
  if (cb == 0)
    for (int e = tid; e < R * (kDr / 2); e += kAbsThreads) rope_row(p, e / (kDr / 2), h, e % (kDr / 2));
}

// ===========================================================================
// Combine kernel: merge the splits of every (row, head) and lift with W_UV.
// CTA = (128 output columns j, head h).  W_UV[h][j0:j0+128][:] is one
// contiguous 128 KiB block, fetched with a single bulk async copy that runs
// while the kernel waits for the attention grid.
// ===========================================================================
constexpr int kCmbThreads = 256;
constexpr int kCmbJ = 128;
constexpr int kCmbRows = 8;
constexpr int kCPitch = kDl + 4;   // floats per clat row in smem
constexpr int kMaxPieces = 256;    // splits per row (<= CTAs of the attention grid)
constexpr uint32_t kCmbWBytes = kCmbJ * kDl * 2;
constexpr int kCmbPre = 4;         // splits per warp whose partials load before the weights are formed

struct CombineParams {
  const __nv_bfloat16* kv_b;
  const float* o_part;
  const float* ml_part;
  const int32_t* T;
  const int32_t* nsel;
  float* out;  // [R, 64, Dv], R <= kCmbRows
  int B, S, G, Dn, Dv, sparse, T_cap, topk;
  unsigned int* flags;
};


__global__ void __launch_bounds__(kCmbThreads) combine_kernel(const CombineParams p) {
  extern __shared__ __align__(128) unsigned char sm[];
  const __nv_bfloat16* Ws = reinterpret_cast<const __nv_bfloat16*>(sm);   // [64][512]
  float* clat = reinterpret_cast<float*>(sm + kCmbWBytes);                 // [kCmbRows][kCPitch]
  float* inv_l = clat + kCmbRows * kCPitch;                                // [kCmbRows]
  int* pcnt = reinterpret_cast<int*>(inv_l + kCmbRows);                    // [kCmbRows]
  int* pslot = pcnt + kCmbRows;                                            // [kCmbRows][kMaxPieces]
  float* pm = reinterpret_cast<float*>(pslot + kCmbRows * kMaxPieces);     // split weights
  float* pw = pm + kCmbRows * kMaxPieces;                                  // split row sums
  float4* red = reinterpret_cast<float4*>(pw + kCmbRows * kMaxPieces);     // [8 warps][128] partial clat
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
  // The call's rows (R <= kCmbRows) and their tile plan come from the kernel
  // inputs alone -- the same tile counts as the absorb kernel's plan -- so
  // the list of each row's splits is ready before the attention grid ends.
  const int R = p.B * p.S;
  const int NR = p.sparse ? R : p.B;
  __shared__ int cts[kCmbRows + 1], cbad[kCmbRows];
  if (tid < NR) {
    const int b = p.sparse ? tid / p.S : tid;
    const int Tb = p.T[b];
    int bad = (Tb < p.S || Tb > p.T_cap) ? 1 : 0, nk = Tb;
    if (!bad && p.sparse) {
      nk = p.nsel[tid];
      bad = (nk < 1 || nk > p.topk) ? 1 : 0;
    }
    cbad[tid] = bad;
    cts[tid + 1] = bad ? 0 : (nk + kTile - 1) / kTile;
  }
  __syncthreads();
  if (tid == 0) {
    cts[0] = 0;
    for (int r = 0; r < NR; ++r) cts[r + 1] += cts[r];
  }
  __syncthreads();
  const long long N = cts[NR];
  const int nr = R;
  const int r0 = 0;
  // (a) warp w lists the splits of row w ...
  if (warp < nr) {
    const int r = warp, b = r / p.S, s = r % p.S;
    const int row = p.sparse ? r : b;
    int cnt = 0;
    if (!cbad[row] && N > 0) {
      const long long a = cts[row], e = cts[row + 1];
      const int glo = chunk_of(a, N, p.G), ghi = chunk_of(e - 1, N, p.G);
      for (int g0 = glo; g0 <= ghi; g0 += 32) {
        const int gg = g0 + lane;
        int lo = 0, hi = 0;
        if (gg <= ghi) {
          if (p.sparse) piece_range<true>(cts, p.T, p.S, s, row, gg, p.G, N, &lo, &hi);
          else piece_range<false>(cts, p.T, p.S, s, row, gg, p.G, N, &lo, &hi);
        }
        const bool has = lo < hi;
        const unsigned m = __ballot_sync(0xffffffffu, has);
        if (has) pslot[warp * kMaxPieces + cnt + __popc(m & ((1u << lane) - 1))] = p.sparse ? gg + row : (gg + row) * p.S + s;
        cnt += __popc(m);
      }
    }
    if (lane == 0) {
      pcnt[warp] = cnt;
      inv_l[warp] = (cbad[row] || N <= 0) ? __int_as_float(0x7fc00000) : 1.f;
    }
  }
  __syncthreads();  // every warp reads the lists below
  grid_dep_wait();   // partials come from the attention kernel
  bool w_ready = false;
  // (b) deals the 8 warps to the rows (wpr each); warp k takes every wpr-th
  // split of its row.  The partials of its first kCmbPre splits are loaded
  // now, so that they are in flight together with the (m, l) loads of (a)
  // instead of waiting for the weights.
  const int wpr = (kCmbThreads / 32) / nr;  // nr <= kCmbRows = 8
  const int bw = warp / wpr, sk = warp % wpr;
  float4 pre[kCmbPre][4];
  if (bw < nr) {
    const int cnt = pcnt[bw];
#pragma unroll
    for (int u = 0; u < kCmbPre; ++u) {
      const int i = sk + u * wpr;
      if (i < cnt) {
        const float4* src =
            reinterpret_cast<const float4*>(p.o_part + ((size_t)pslot[bw * kMaxPieces + i] * kH + h) * kDl);
#pragma unroll
        for (int q = 0; q < 4; ++q) pre[u][q] = src[lane + 32 * q];
      }
    }
  }
  {
    // (a) with the partials complete, their normalised weights
    if (warp < nr) {
      __syncwarp();  // entries were listed by other lanes
      const int cnt = pcnt[warp];
      float M = -INFINITY;
      for (int i = lane; i < cnt; i += 32) {
        const float2 ml = *reinterpret_cast<const float2*>(p.ml_part + ((size_t)pslot[warp * kMaxPieces + i] * kH + h) * 2);
        pm[warp * kMaxPieces + i] = ml.x;
        pw[warp * kMaxPieces + i] = ml.y;
        M = fmaxf(M, ml.x);
      }
      M = warp_max(M);
      float L = 0.f;
      for (int i = lane; i < cnt; i += 32) {
        const float wg = exp2f(pm[warp * kMaxPieces + i] - M);
        pm[warp * kMaxPieces + i] = wg;
        L = fmaf(wg, pw[warp * kMaxPieces + i], L);
      }
      L = warp_sum(L);
      for (int i = lane; i < cnt; i += 32) pm[warp * kMaxPieces + i] /= L;
    }
    __syncthreads();
    // (b) clat[w][l] = sum_i weight_i * O_i[h][l] for every row at once:
    //     lane covers latents 4*lane + 128*q; the warp sums meet in shared
    //     memory.
    {
      const int w = bw;
      if (w < nr) {
        const int cnt = pcnt[w];
        float4 acc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kCmbPre; ++u) {
          const int i = sk + u * wpr;
          if (i < cnt) {
            const float wg = pm[w * kMaxPieces + i];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[q].x = fmaf(wg, pre[u][q].x, acc[q].x);
              acc[q].y = fmaf(wg, pre[u][q].y, acc[q].y);
              acc[q].z = fmaf(wg, pre[u][q].z, acc[q].z);
              acc[q].w = fmaf(wg, pre[u][q].w, acc[q].w);
            }
          }
        }
#pragma unroll 4
        for (int i = sk + kCmbPre * wpr; i < cnt; i += wpr) {
          const float wg = pm[w * kMaxPieces + i];
          const float4* src =
              reinterpret_cast<const float4*>(p.o_part + ((size_t)pslot[w * kMaxPieces + i] * kH + h) * kDl);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 o = src[lane + 32 * q];
            acc[q].x = fmaf(wg, o.x, acc[q].x);
            acc[q].y = fmaf(wg, o.y, acc[q].y);
            acc[q].z = fmaf(wg, o.z, acc[q].z);
            acc[q].w = fmaf(wg, o.w, acc[q].w);
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) red[warp * 128 + lane + 32 * q] = acc[q];
      }
      __syncthreads();
      for (int e = tid; e < nr * 128; e += kCmbThreads) {
        const int rw = e >> 7, idx = e & 127;
        float4 t = red[(rw * wpr) * 128 + idx];
        for (int k = 1; k < wpr; ++k) {
          const float4 u = red[(rw * wpr + k) * 128 + idx];
          t.x += u.x;
          t.y += u.y;
          t.z += u.z;
          t.w += u.w;
        }
        *reinterpret_cast<float4*>(clat + rw * kCPitch + 4 * idx) = t;
      }
      __syncthreads();
    }
    if (!w_ready) {
      volatile int no_abort = 0;
      if (!mbar_wait(&wbar, 0, &no_abort, p.flags, kDrainNs)) raise_flag(p.flags, MLA_DEV_TIMEOUT);
      w_ready = true;
    }
    __syncthreads();
    // (c) out[r][h][j0 + j] = W_UV[j] . clat[r]: warp k owns kCmbJ/8 outputs, eight at a time;
    //     lanes split the latent axis (16 values each), and the eight partial
    //     sums are reduced together by a transposing butterfly.
#pragma unroll 1
    for (int jb8 = 0; jb8 < kCmbJ / 64; ++jb8) {
      const int jw = warp * (kCmbJ / 8) + 8 * jb8;
      uint4 wlo[8], whi[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const __nv_bfloat16* wr = Ws + (size_t)(jw + jj) * kDl;
        wlo[jj] = *reinterpret_cast<const uint4*>(wr + 8 * lane);
        whi[jj] = *reinterpret_cast<const uint4*>(wr + 256 + 8 * lane);
      }
      for (int w = 0; w < nr; ++w) {
        const float* cr = clat + w * kCPitch;
        float cv[16];
        *reinterpret_cast<float4*>(&cv[0]) = *reinterpret_cast<const float4*>(cr + 8 * lane);
        *reinterpret_cast<float4*>(&cv[4]) = *reinterpret_cast<const float4*>(cr + 8 * lane + 4);
        *reinterpret_cast<float4*>(&cv[8]) = *reinterpret_cast<const float4*>(cr + 256 + 8 * lane);
        *reinterpret_cast<float4*>(&cv[12]) = *reinterpret_cast<const float4*>(cr + 256 + 8 * lane + 4);
        float d[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&wlo[jj]);
          const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&whi[jj]);
          float acc = 0.f;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float2 fa = __bfloat1622float2(a2[t]);
            const float2 fb = __bfloat1622float2(b2[t]);
            acc = fmaf(fa.x, cv[2 * t], acc);
            acc = fmaf(fa.y, cv[2 * t + 1], acc);
            acc = fmaf(fb.x, cv[8 + 2 * t], acc);
            acc = fmaf(fb.y, cv[8 + 2 * t + 1], acc);
          }
          d[jj] = acc;
        }
        // butterfly: after offsets 16, 8, 4 lane L holds output jw + ((L >> 2) & 7)'s
        // partial over lanes {L ^ 3 mask}; offsets 2 and 1 finish the sum.
#pragma unroll
        for (int step = 0; step < 3; ++step) {
          const int o = 16 >> step, hh = 4 >> step;
          const bool upper = (lane & o) != 0;
#pragma unroll
          for (int i = 0; i < hh; ++i) {
            const float send = upper ? d[i] : d[i + hh];
            const float keep = upper ? d[i + hh] : d[i];
            d[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        d[0] += __shfl_xor_sync(0xffffffffu, d[0], 2);
        d[0] += __shfl_xor_sync(0xffffffffu, d[0], 1);
        if ((lane & 3) == 0) {
          const int jj = 4 * ((lane >> 4) & 1) + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1);
          p.out[((size_t)(r0 + w) * kH + h) * p.Dv + j0 + jw + jj] = d[0] * inv_l[w];
        }
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

constexpr int kMergeBatch = 2;  // splits whose partials are loaded together

__global__ void __launch_bounds__(256, 3) merge_kernel(const MergeParams p) {
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
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  float L = 0.f;
  auto slot_of = [&](int gg) -> int {  // the split of chunk gg, or -1 when the chunk has no tile of this row
    int lo, hi;
    if (p.sparse) piece_range<true>(p.tile_start, p.T, p.S, s, row, gg, p.G, N, &lo, &hi);
    else piece_range<false>(p.tile_start, p.T, p.S, s, row, gg, p.G, N, &lo, &hi);
    if (lo >= hi) return -1;
    return p.sparse ? gg + row : (gg + row) * p.S + s;
  };
  auto add = [&](float wgt, const float4 (&o)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[4 * i] = fmaf(wgt, o[i].x, acc[4 * i]);
      acc[4 * i + 1] = fmaf(wgt, o[i].y, acc[4 * i + 1]);
      acc[4 * i + 2] = fmaf(wgt, o[i].z, acc[4 * i + 2]);
      acc[4 * i + 3] = fmaf(wgt, o[i].w, acc[4 * i + 3]);
    }
  };
  auto part_of = [&](int slot) -> const float4* {
    return reinterpret_cast<const float4*>(p.o_part + ((size_t)slot * kH + h) * kDl + 16 * lane);
  };
  if (ghi - glo < 32) {
    // One split per lane: each lane reads its split's (m, l), the warp forms
    // the weights, then the partials are read two splits at a time with all
    // their loads in flight (more would cost occupancy when rows are many).
    const int myslot = glo + lane <= ghi ? slot_of(glo + lane) : -1;
    float2 ml = make_float2(-INFINITY, 0.f);
    if (myslot >= 0) ml = *reinterpret_cast<const float2*>(p.ml_part + ((size_t)myslot * kH + h) * 2);
    const float M = warp_max(ml.x);
    const float mw = myslot >= 0 ? exp2f(ml.x - M) : 0.f;
    L = warp_sum(mw * ml.y);
    unsigned live = __ballot_sync(0xffffffffu, myslot >= 0);
    while (live) {
      int src[kMergeBatch];
      float wg[kMergeBatch];
      float4 o[kMergeBatch][4];
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        src[u] = live ? __ffs(live) - 1 : -1;
        if (live) live &= live - 1;
      }
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const int sl = __shfl_sync(0xffffffffu, myslot, src[u] < 0 ? 0 : src[u]);
        wg[u] = __shfl_sync(0xffffffffu, mw, src[u] < 0 ? 0 : src[u]);
        if (src[u] >= 0) {
          const float4* op = part_of(sl);
#pragma unroll
          for (int i = 0; i < 4; ++i) o[u][i] = op[i];
        }
      }
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u)
        if (src[u] >= 0) add(wg[u], o[u]);
    }
  } else {  // more than 32 splits: one at a time
    float M = -INFINITY;
    for (int gg = glo + lane; gg <= ghi; gg += 32) {
      const int slot = slot_of(gg);
      if (slot >= 0) M = fmaxf(M, p.ml_part[((size_t)slot * kH + h) * 2]);
    }
    M = warp_max(M);
    for (int gg = glo; gg <= ghi; ++gg) {
      const int slot = slot_of(gg);
      if (slot < 0) continue;
      const float2 ml = *reinterpret_cast<const float2*>(p.ml_part + ((size_t)slot * kH + h) * 2);
      const float wgt = exp2f(ml.x - M);
      L = fmaf(wgt, ml.y, L);
      float4 o[4];
      const float4* op = part_of(slot);
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = op[i];
      add(wgt, o);
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
  PageTable pages;
};

// Warp = 4 selected keys.  All index loads, then all row loads of the warp
// are issued before the first store, so a warp waits for two memory round
// trips instead of one per 16-byte chunk.
__global__ void __launch_bounds__(256) gather_kernel(const GatherParams p) {
  constexpr int kKeys = 4, kChunks = (kDc / 8 + 31) / 32;  // 72 chunks of 16 B per row: 3 per lane
  grid_dep_launch();  // the absorb kernel may start: it loads W_UK, then waits for this grid
  const int r = blockIdx.y, b = r / p.S, s = r % p.S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Tb = p.T[b];
  const int n = p.nsel[r];
  const bool row_ok = Tb >= p.S && Tb <= p.T_cap && n >= 1 && n <= p.topk;
  const int pos = Tb - p.S + s;
  const int j0 = blockIdx.x * 32 + warp * kKeys;
  int idx[kKeys];
#pragma unroll
  for (int kk = 0; kk < kKeys; ++kk) idx[kk] = (row_ok && j0 + kk < n) ? __ldg(p.sel + (size_t)r * p.topk + j0 + kk) : -1;
  long long row[kKeys];
#pragma unroll
  for (int kk = 0; kk < kKeys; ++kk) {
    row[kk] = 0;
    if (row_ok && j0 + kk < n && (idx[kk] < 0 || idx[kk] > pos)) {
      if (lane == 0) raise_flag(p.flags, MLA_DEV_BAD_INDEX);
      idx[kk] = -1;
    }
    if (idx[kk] >= 0) {
      bool bad_page = false;
      row[kk] = cache_row(p.pages, b, p.T_cap, idx[kk], &bad_page);
      if (bad_page) {
        if (lane == 0) raise_flag(p.flags, MLA_DEV_BAD_INDEX);
        idx[kk] = -1;
        row[kk] = 0;
      }
    }
  }
  uint4 v[kKeys][kChunks];
#pragma unroll
  for (int kk = 0; kk < kKeys; ++kk) {
    const uint4* lsrc = reinterpret_cast<const uint4*>(p.Lc + (size_t)row[kk] * kDl);
    const uint4* rsrc = reinterpret_cast<const uint4*>(p.Rc + (size_t)row[kk] * kDr);
#pragma unroll
    for (int u = 0; u < kChunks; ++u) {
      const int c = lane + 32 * u;
      v[kk][u] = make_uint4(0, 0, 0, 0);
      if (idx[kk] >= 0 && c < kDc / 8) v[kk][u] = c < kDl / 8 ? __ldg(lsrc + c) : __ldg(rsrc + (c - kDl / 8));
    }
  }
#pragma unroll
  for (int kk = 0; kk < kKeys; ++kk) {
    uint4* dst = reinterpret_cast<uint4*>(p.stage + ((size_t)r * p.Kpad + j0 + kk) * kDc);
#pragma unroll
    for (int u = 0; u < kChunks; ++u) {
      const int c = lane + 32 * u;
      if (c < kDc / 8) dst[c] = v[kk][u];
    }
  }
  // Launched as a programmatic dependent, this kernel reads only inputs that
  // no kernel of the call writes; waiting here, after the stores, keeps the
  // chain's order: its completion implies the previous kernel's.
  grid_dep_wait();
}

// ===========================================================================
// Host side
// ===========================================================================
struct Plan {
  int G, NR, P, R, Kpad;
  size_t off_q, off_ts, off_bad, off_o, off_ml, off_stage, off_clat, off_invl, off_q8, off_fh, total;
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

std::atomic<unsigned long long> g_abs_attr[9] = {}, g_attn_attr[10] = {}, g_cmb_attr{0};

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
  pl.off_stage = off;  // two staging buffers: consecutive layers of one call alternate
  off = align256(off + 2 * (size_t)pl.R * pl.Kpad * kDc * 2);
  pl.off_clat = off;
  off = align256(off + (pl.R > kSmallRows ? (size_t)pl.R * kH * kDl * 2 : 0));
  pl.off_invl = off;
  off = align256(off + (pl.R > kSmallRows ? (size_t)pl.R * kH * 4 : 0));
  // FP8 cache (dense only): quantised query rows and their score factors
  pl.off_q8 = off;
  off = align256(off + (sparse_topk ? 0 : (size_t)pl.R * kH * kQ8Row));
  pl.off_fh = off;
  off = align256(off + (sparse_topk ? 0 : (size_t)pl.R * kH * 4));
  pl.total = off;
  return pl;
}

cudaError_t run(const DecodeArgs& a, void* ws, bool sparse, cudaStream_t st) {
  const Geometry& g = a.g;
  const int B = a.B, S = a.S;
  const Plan pl = make_plan(B, S, a.T_cap, sparse ? a.topk : 0);
  const bool paged = a.pages.table != nullptr;
  const long long pool_rows = paged ? (long long)a.pages.num_pages * a.pages.page_size : (long long)B * a.T_cap;
  if (pool_rows >= (1ll << 31) || (long long)B * a.T_cap >= (1ll << 31)) return cudaErrorInvalidValue;
  if (paged && a.pages.page_size % kTile != 0) return cudaErrorInvalidValue;
  unsigned char* w = static_cast<unsigned char*>(ws);
  __nv_bfloat16* qcat = reinterpret_cast<__nv_bfloat16*>(w + pl.off_q);
  int32_t* ts = reinterpret_cast<int32_t*>(w + pl.off_ts);
  int32_t* bad = reinterpret_cast<int32_t*>(w + pl.off_bad);
  float* o_part = reinterpret_cast<float*>(w + pl.off_o);
  float* ml_part = reinterpret_cast<float*>(w + pl.off_ml);
  __nv_bfloat16* stage =
      reinterpret_cast<__nv_bfloat16*>(w + pl.off_stage) + (a.stage_parity & 1) * (size_t)pl.R * pl.Kpad * kDc;
  cudaError_t e;

  // 0. sparse: gather the selected key rows.  A plain launch, except for the
  //    later layers of one mla_sparse_decode_layers call: those alternate
  //    between two staging buffers and launch as programmatic dependents of
  //    the previous layer's last kernel, so their row loads overlap its tail
  //    (the buffer they write was last read two layers back).  The absorb
  //    kernel, launched next with programmatic serialization, starts once
  //    the gather retires.
  if (sparse && a.lat_fp8) return cudaErrorInvalidValue;
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
    gp.pages = a.pages;
    kernel_mark(st, "gather");
    e = launch_pdl(gather_kernel, dim3(pl.Kpad / 32, pl.R), dim3(256), 0, st, gp, a.gather_pdl != 0);
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
  ap.Lc = static_cast<const unsigned char*>(a.Lc);
  ap.Rc = static_cast<const __nv_bfloat16*>(a.Rc);
  ap.lat_row_bytes = a.lat_fp8 ? kDl : kDl * 2;
  // L2 prefetch on the small-batch path while the cache stays well inside L2
  ap.prefetch =
      (!big && !sparse && (long long)B * a.T_cap * (ap.lat_row_bytes + kDr * 2) <= (48ll << 20)) ? 1 : 0;
  ap.pages = sparse ? PageTable{} : a.pages;
  for (int j = 0; j < kDr / 2; ++j) ap.turn[j] = rope_turns(std::pow(g.rope_base, -2.0 * j / kDr));
  ap.flags = a.flags;
  const size_t abs_smem = (size_t)kAbsRows * g.Dn * 4 + (size_t)kAbsGroups * kAbsRows * kAbsCols * 4;
  // one instantiation per case, so that each carries only its own code
  using AbsKern = void (*)(const AbsorbParams);
  static const AbsKern abs_kerns[2][4] = {
      {absorb_kernel<4>, absorb_kernel<8>, absorb_kernel<12>, absorb_kernel<16>},
      {absorb_kernel<4, true, true>, absorb_kernel<8, true, true>, absorb_kernel<12, true, true>,
       absorb_kernel<16, true, true>}};
  const bool paged_abs = ap.prefetch && ap.pages.table;
  const AbsKern akern = big ? absorb_kernel<4, false> : abs_kerns[paged_abs ? 1 : 0][g.Dn / 64 - 1];
  // many rows: the rotary part of each head spread over up to four CTAs
  const int abs_gx = big ? std::min(4, (pl.R * (kDr / 2) + 2047) / 2048) : kDl / kAbsCols;
  e = set_smem_once(akern, (int)abs_smem, &g_abs_attr[big ? 8 : (paged_abs ? 4 : 0) + g.Dn / 64 - 1]);
  if (e != cudaSuccess) return e;
  kernel_mark(st, big ? "plan_rope" : "absorb");
  e = launch_pdl(akern, dim3(abs_gx, kH), dim3(kAbsThreads), abs_smem, st, ap);
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

  // 1b. FP8 cache: quantise the query rows
  unsigned char* q8 = w + pl.off_q8;
  float* fh = reinterpret_cast<float*>(w + pl.off_fh);
  if (a.lat_fp8 && big) {  // few rows: the attention kernel quantises them itself
    QuantParams qp{};
    qp.qcat = qcat;
    qp.q8 = q8;
    qp.fh = fh;
    qp.rows = pl.R * kH;
    qp.c = g.scale * kLog2e;
    qp.lat_scale = a.lat_scale;
    kernel_mark(st, "quant_q");
    e = launch_pdl(quant_q_kernel, dim3((qp.rows * 32 + 255) / 256), dim3(256), 0, st, qp);
    if (e != cudaSuccess) return e;
  }

  // 2. attention
  AttnParams tp{};
  bool maps_ok = a.lat_fp8 ? make_tmap_2d_u8(&tp.mQ, q8, (uint64_t)pl.R * kH, kQ8Row, kQ8Row, kH, 128)
                           : make_tmap_2d_bf16(&tp.mQ, qcat, (uint64_t)pl.R * kH, kDc, kDc, kH, 64);
  if (!sparse) {
    const uint64_t rows = (uint64_t)pool_rows;
    maps_ok = maps_ok &&
              (a.lat_fp8 ? make_tmap_2d_u8(&tp.mL, a.Lc, rows, kDl, kDl, kTile, 128)
                         : make_tmap_2d_bf16(&tp.mL, a.Lc, rows, kDl, kDl, kTile, 64)) &&
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
  // Few pieces leave SMs idle: then 2 or 4 CTAs share a piece, each repeating
  // the score product (the tile comes from L2 after the first) and taking its
  // share of the value product and of the partial's stores.
  const int pieces = sparse ? pl.G : pl.G * S;
  const int sms = sm_count();
  tp.qsplit = pieces * 4 <= sms ? 4 : pieces * 2 <= sms ? 2 : 1;
  tp.read_once = ((sparse || S == 1) && tp.qsplit == 1) ? 1 : 0;
  tp.c = g.scale * kLog2e;
  tp.lat_scale = a.lat_fp8 ? a.lat_scale : 1.f;
  tp.fh = fh;
  tp.qcat = qcat;
  tp.o_part = o_part;
  tp.ml_part = ml_part;
  tp.flags = a.flags;
  tp.wait_ns = a.wait_limit_ns;
  tp.pages = sparse ? PageTable{} : a.pages;
  // Streaming launches (one CTA per piece, at least two tiles a CTA by the
  // T_cap bound) take the instantiation with the single-lane score loop.
  const long long tiles_cap = (long long)B * ((a.T_cap + kTile - 1) / kTile);
  const bool stream = !sparse && tp.qsplit == 1 && tiles_cap >= 2LL * pl.G;
  auto kern = sparse     ? attn_kernel<true>
              : a.lat_fp8 ? (big ? (stream ? attn8_kernel<false, true> : attn8_kernel<false>)
                                 : (stream ? attn8_kernel<true, true> : attn8_kernel<true>))
              : paged     ? (stream ? attn_kernel<false, true, true> : attn_kernel<false, true>)
                          : (stream ? attn_kernel<false, false, true> : attn_kernel<false>);
  const uint32_t attn_smem = a.lat_fp8 ? kAttn8DynSmem : kAttnDynSmem;
  const int attr_slot = (sparse ? 1 : a.lat_fp8 ? (big ? 2 : 4) : paged ? 3 : 0) + (stream ? 5 : 0);
  e = set_smem_once(kern, (int)attn_smem, &g_attn_attr[attr_slot]);
  if (e != cudaSuccess) return e;
  const int nblk = pieces * tp.qsplit;
  kernel_mark(st, "attention");
  e = launch_pdl(kern, dim3(nblk), dim3(kAttnThreads), attn_smem, st, tp);
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
  cp.T = a.T;
  cp.nsel = a.nsel;
  cp.T_cap = a.T_cap;
  cp.topk = a.topk;
  cp.out = a.out;
  cp.B = B;
  cp.S = S;
  cp.G = pl.G;
  cp.Dn = g.Dn;
  cp.Dv = g.Dv;
  cp.sparse = sparse ? 1 : 0;
  cp.flags = a.flags;
  const size_t cmb_smem = (size_t)kCmbWBytes + (size_t)kCmbRows * kCPitch * 4 + kCmbRows * 8 +
                          (size_t)kCmbRows * kMaxPieces * 12 + (size_t)(kCmbThreads / 32) * 128 * 16;
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
