// index_tc.cu -- DSA lightning-indexer scores on the tensor cores.
//
// The page "MLA 注意力与 KV 缓存", §2.2: every past key t of a query gets
// I[t] = sum_h w_h * ReLU(q_h . Ic[t]) over the index heads; keys past the
// query's position are -inf.  The indexer keys Ic are fp32 (page
// "第 7 章 · 03 token 精确前向验证与 faithful DSA", §二).
//
// For 32 index heads of 128 values the dot products are a GEMM per query:
// D[128 keys x 32 heads] = Ic tile [128 x 128] x q^T.  The tensor cores take
// fp32 operands as tf32 (the low 13 mantissa bits dropped), so the product is
// formed as three tf32 products, Ic*q + Ic*q_lo + Ic_lo*q with
// x_lo = x - tf32(x): the omitted Ic_lo*q_lo term and the rounding of the
// split leave an error of a few fp32 ulps of the terms.  Integer-valued inputs
// of magnitude below 2^11 have x_lo = 0 and fp32 partial sums below 2^24, so
// their scores come out exact in any order.  A product whose low operand is
// exactly zero adds exact zeros, so it is skipped: the query's low part when
// the whole query is tf32-exact, a tile's low part (and its rewrite) when the
// tile is -- the check reads the tile once and writes nothing.
//
// CTA = a run of 128-key tiles of one (b, s): warp 0 streams the tiles
// (four 32-column atoms, 128-byte swizzle) into a 3-stage ring with TMA,
// warp 1 issues the MMAs, warps 2-5 rewrite each tile in place as its low
// part for the third product and turn the accumulators into scores.
#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace sm100;

constexpr int kITile = 128;                       // keys per tile
constexpr int kIHd = 128;                         // values per key / per index head
constexpr int kIHeads = 32;                       // index heads
constexpr int kIStages = 3;
constexpr uint32_t kIAtomBytes = kITile * 128;    // 128 keys x 32 fp32
constexpr uint32_t kITileBytes = 4 * kIAtomBytes; // 64 KB
constexpr uint32_t kIQAtomBytes = kIHeads * 128;  // 32 heads x 32 fp32
constexpr uint32_t kIQBytes = 4 * kIQAtomBytes;   // 16 KB
constexpr uint32_t kIDynSmem = kIStages * kITileBytes + 2 * kIQBytes + 1024;
constexpr int kIThreads = 192;
constexpr long long kIDrainNs = 1000000000LL;

struct IdxTcParams {
  CUtensorMap mI;  // Ic as [B*T_cap, 128] fp32
  const float* q;  // [B, S, 32, 128]
  const float* w;  // [B, S, 32]
  const int32_t* T;
  float* scores;   // [B, S, T_cap]
  uint32_t* hpart; // [B*S, gridDim.x, 2048] or null
  int B, S, T_cap, ntiles, tpc;
  unsigned int* flags;
  long long wait_ns;
};

// element (r, k) of a K-major operand of 4-byte values with 128-byte rows, 128-byte swizzle
__device__ __forceinline__ uint32_t swz4(int r, int k) {
  return (uint32_t)(r * 128 + ((((k * 4) >> 4) ^ (r & 7)) << 4) + ((k * 4) & 15));
}

// x - tf32(x): the part the tensor core drops
__device__ __forceinline__ float tf32_lo(float x) { return x - __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

__global__ void __launch_bounds__(kIThreads, 1) index_tc_kernel(const __grid_constant__ IdxTcParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  unsigned char* sTile = smem;                          // kIStages x 64 KB
  unsigned char* sQ = smem + kIStages * kITileBytes;    // q as stored
  unsigned char* sQlo = sQ + kIQBytes;                  // q - tf32(q)
  __shared__ uint64_t full_bar[kIStages], empty_bar[kIStages], hi_done[kIStages], lo_ready[kIStages];
  __shared__ uint64_t acc_full[2], acc_free[2], mma_done;
  __shared__ int lo_needed[kIStages];  // the tile of this stage has a nonzero low part
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ float w_s[kIHeads];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.y, b = blockIdx.z;
  const int tb = blockIdx.x * p.tpc;
  const int te = min(p.ntiles, tb + p.tpc);
  float* srow = p.scores + ((size_t)b * p.S + s) * p.T_cap;
  grid_dep_launch();  // the top-k of a fused selection may launch; it waits for this grid
  // this CTA's slice of the first-pass histogram, filled by the epilogue
  uint32_t* hp = p.hpart ? p.hpart + (((size_t)b * p.S + s) * gridDim.x + blockIdx.x) * 2048 : nullptr;
  if (hp)
    for (int i = threadIdx.x; i < 2048; i += kIThreads) hp[i] = 0u;
  const int Tb = p.T[b];
  if (Tb < p.S || Tb > p.T_cap) {  // whole CTA: NaN scores and the length flag
    if (threadIdx.x == 0 && blockIdx.x == 0 && s == 0) raise_flag(p.flags, MLA_DEV_BAD_LENGTH);
    for (int t = tb * kITile + threadIdx.x; t < min(te * kITile, p.T_cap); t += kIThreads) srow[t] = qnan();
    return;
  }
  const int pos = Tb - p.S + s;
  const int te_act = min(te, pos / kITile + 1);  // tiles holding a key <= pos
  const int na = max(0, te_act - tb);
  // tiles entirely in the future of this query
  for (int t = max(tb, te_act) * kITile + threadIdx.x; t < min(te * kITile, p.T_cap); t += kIThreads)
    srow[t] = -INFINITY;
  if (na == 0) return;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kIStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
      mbar_init(&hi_done[i], 1);
      mbar_init(&lo_ready[i], 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_free[i], 128);
    }
    mbar_init(&mma_done, 1);
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&p.mI);
    // the first tiles stream in while the query block is formed (thread 0 is
    // the producer lane; the ring's stages are free at the start)
    const int y0 = b * p.T_cap + tb * kITile;
    for (int i = 0; i < na && i < kIStages; ++i) {
      mbar_arrive_expect_tx(&full_bar[i], kITileBytes);
      for (int a = 0; a < 4; ++a)
        tma_load_2d(sTile + i * kITileBytes + a * kIAtomBytes, &p.mI, 32 * a, y0 + i * kITile, &full_bar[i]);
    }
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 64);
    tmem_relinquish();
  }
  // query block: stored value and low part, K-major with the 128-byte swizzle
  // All of the thread's query loads are in flight before the first store
  // (one memory round trip, not one per element).
  const float4* qsrc = reinterpret_cast<const float4*>(p.q + ((size_t)b * p.S + s) * kIHeads * kIHd);
  constexpr int kQVec = kIHeads * kIHd / 4, kQPer = (kQVec + kIThreads - 1) / kIThreads;
  float4 qv[kQPer];
#pragma unroll
  for (int u = 0; u < kQPer; ++u) {
    const int e4 = threadIdx.x + u * kIThreads;
    if (e4 < kQVec) qv[u] = qsrc[e4];
  }
  if (threadIdx.x < kIHeads) w_s[threadIdx.x] = p.w[((size_t)b * p.S + s) * kIHeads + threadIdx.x];
  bool qlo_nz = false;
#pragma unroll
  for (int u = 0; u < kQPer; ++u) {
    const int e4 = threadIdx.x + u * kIThreads;
    if (e4 < kQVec) {
      const float xs[4] = {qv[u].x, qv[u].y, qv[u].z, qv[u].w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int e = 4 * e4 + c, h = e / kIHd, d = e % kIHd;
        const uint32_t off = (uint32_t)(d / 32) * kIQAtomBytes + swz4(h, d % 32);
        const float lo = tf32_lo(xs[c]);
        *reinterpret_cast<float*>(sQ + off) = xs[c];
        *reinterpret_cast<float*>(sQlo + off) = lo;
        qlo_nz = qlo_nz || lo != 0.f;
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  const bool q_has_lo = __syncthreads_or(qlo_nz) != 0;
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  volatile int* abort = &abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int y0 = b * p.T_cap + tb * kITile;
      const int i0 = na < kIStages ? na : kIStages;  // issued before the query block
      int last = i0 - 1;
      for (int i = i0; i < na; ++i) {
        const int st = i % kIStages;
        if (!mbar_wait(&empty_bar[st], ((i / kIStages) & 1) ^ 1, abort, p.flags, p.wait_ns)) break;
        mbar_arrive_expect_tx(&full_bar[st], kITileBytes);
        for (int a = 0; a < 4; ++a)
          tma_load_2d(sTile + st * kITileBytes + a * kIAtomBytes, &p.mI, 32 * a, y0 + i * kITile, &full_bar[st]);
        last = i;
      }
      volatile int no_abort = 0;
      const long long drain = p.wait_ns > kIDrainNs ? p.wait_ns : kIDrainNs;
      for (int i = max(0, last - kIStages + 1); i <= last; ++i)
        mbar_wait(&full_bar[i % kIStages], (i / kIStages) & 1, &no_abort, p.flags, drain);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (whole warp waits, lane 0 issues)
    const uint32_t idesc = idesc_tf32_f32(128, kIHeads);
    const uint32_t t0 = smem_u32(sTile), q0 = smem_u32(sQ), ql0 = smem_u32(sQlo);
    bool ok = true, issued = false;
    auto wait = [&](uint64_t* bar, uint32_t par) -> bool {
      const bool r = mbar_wait(bar, par, abort, p.flags, p.wait_ns);
      return __all_sync(0xffffffffu, r);
    };
    // passes 1 and 2 of tile i: tile x q, tile x q_lo
    auto hi_pass = [&](int i) -> bool {
      const int st = i % kIStages, buf = i & 1;
      if (!wait(&full_bar[st], (i / kIStages) & 1)) return false;
      if (!wait(&acc_free[buf], ((i >> 1) & 1) ^ 1)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t tile = t0 + st * kITileBytes;
        for (int pass = 0; pass < (q_has_lo ? 2 : 1); ++pass)
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t da = smem_desc_sw128(tile + a * kIAtomBytes + kk * 32, 16, 1024);
              const uint64_t db = smem_desc_sw128((pass ? ql0 : q0) + a * kIQAtomBytes + kk * 32, 16, 1024);
              mma_tf32(tmem + 32 * buf, da, db, idesc, (pass | a | kk) != 0 ? 1u : 0u);
            }
        mma_commit(&hi_done[st]);
      }
      __syncwarp();
      return true;
    };
    // pass 3 of tile i: tile_lo x q, once the tile holds its low part
    auto lo_pass = [&](int i) -> bool {
      const int st = i % kIStages, buf = i & 1;
      if (!wait(&lo_ready[st], (i / kIStages) & 1)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t tile = t0 + st * kITileBytes;
        if (lo_needed[st]) {  // an exact tile's stage was freed by the warps that checked it
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t da = smem_desc_sw128(tile + a * kIAtomBytes + kk * 32, 16, 1024);
              const uint64_t db = smem_desc_sw128(q0 + a * kIQAtomBytes + kk * 32, 16, 1024);
              mma_tf32(tmem + 32 * buf, da, db, idesc, 1u);
            }
          mma_commit(&empty_bar[st]);
        }
        mma_commit(&acc_full[buf]);
      }
      __syncwarp();
      return true;
    };
    // Tile i+1's first two products go ahead of tile i's third, so that the
    // tensor pipe works while tile i is rewritten as its low part.
    for (int i = 0; ok && i <= na; ++i) {
      if (i < na) {
        ok = hi_pass(i);
        issued = issued || ok;
      }
      if (ok && i > 0) ok = lo_pass(i - 1);
    }
    if (issued) {  // all MMAs retired before TMEM is released
      if (lane == 0) mma_commit(&mma_done);
      __syncwarp();
      volatile int no_abort = 0;
      mbar_wait(&mma_done, 0, &no_abort, p.flags, p.wait_ns > kIDrainNs ? p.wait_ns : kIDrainNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ warps 2-5: low parts and scores
    const int e = threadIdx.x - 64;  // 0..127
    const int qd = warp & 3;         // TMEM lane quadrant: keys 32*qd .. 32*qd+31 of a tile
    const uint32_t t_lane = (uint32_t)(32 * qd) << 16;
    bool ok = true;
    // Scores of tile j from its accumulator; a failed wait is decided jointly.
    auto epilogue = [&](int j) -> bool {
      const int buf = j & 1;
      const bool fail = !mbar_wait(&acc_full[buf], (j >> 1) & 1, abort, p.flags, p.wait_ns);
      if (bar_red_or(1, 128, fail)) return false;
      tc_fence_after();
      float v[32];
      tmem_ld32(tmem + t_lane + 32 * buf, v);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&acc_free[buf]);
      float sc = 0.f;
#pragma unroll
      for (int h = 0; h < kIHeads; ++h) sc = fmaf(w_s[h], fmaxf(v[h], 0.f), sc);
      const int t = (tb + j) * kITile + 32 * qd + lane;
      if (t < p.T_cap) srow[t] = (t <= pos) ? sc : -INFINITY;
      if (hp) {  // candidates only; one atomic per distinct bin of the warp
        const bool cand = t <= pos;
        const uint32_t bin = ordered_key(sc) >> 21;
        const unsigned am = __ballot_sync(0xffffffffu, cand);
        if (cand) {
          const unsigned peers = __match_any_sync(am, bin);
          if (lane == __ffs(peers) - 1) atomicAdd(&hp[bin], (uint32_t)__popc(peers));
        }
      }
      return true;
    };
    for (int i = 0; ok && i <= na; ++i) {
      if (i < na) {
        const int st = i % kIStages;
        const bool fail = !mbar_wait(&hi_done[st], (i / kIStages) & 1, abort, p.flags, p.wait_ns);
        if (bar_red_or(1, 128, fail)) {
          ok = false;
          break;
        }
        // Does the tile have low bits?  Read-only: a tf32-exact tile skips the
        // rewrite and the third product.
        float4* tv = reinterpret_cast<float4*>(sTile + st * kITileBytes);
        uint32_t bits = 0;
#pragma unroll 8
        for (int u = e; u < (int)(kITileBytes / 16); u += 128) {
          const uint4 x = reinterpret_cast<const uint4*>(tv)[u];
          bits |= (x.x | x.y | x.z | x.w) & 0x1FFFu;
        }
        const bool has_lo = bar_red_or(1, 128, bits != 0);
        if (has_lo) {
          // tile -> tile - tf32(tile), in place (the first products have read it)
#pragma unroll 8
          for (int u = e; u < (int)(kITileBytes / 16); u += 128) {
            float4 x = tv[u];
            x.x = tf32_lo(x.x);
            x.y = tf32_lo(x.y);
            x.z = tf32_lo(x.z);
            x.w = tf32_lo(x.w);
            tv[u] = x;
          }
          fence_proxy_async_smem();
        }
        if (e == 0) {
          lo_needed[st] = has_lo ? 1 : 0;
          // An exact tile is read for the last time: free its stage now rather
          // than after the next tile's first products.
          if (!has_lo) mbar_arrive(&empty_bar[st]);
        }
        mbar_arrive(&lo_ready[st]);
      }
      if (i > 0) ok = epilogue(i - 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

}  // namespace

namespace {
// Tiles per CTA: about two CTAs' worth of tiles per SM pass, at least 4 tiles per CTA to fill the ring.
int tiles_per_cta(int B, int S, int T_cap) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long ntiles = (T_cap + kITile - 1) / kITile;
  const long long rows = (long long)B * S;
  long long tpc = (rows * ntiles + sms - 1) / sms;
  if (tpc < 4) tpc = 4;
  if (tpc > ntiles) tpc = ntiles;
  return (int)tpc;
}
}  // namespace

int index_tc_parts(int B, int S, int n_ih, int hd, int T_cap) {
  if (n_ih != kIHeads || hd != kIHd || B < 1 || S < 1 || T_cap < 1) return 0;
  const int ntiles = (T_cap + kITile - 1) / kITile;
  const int tpc = tiles_per_cta(B, S, T_cap);
  return (ntiles + tpc - 1) / tpc;
}

cudaError_t launch_index_scores_tc(const IndexArgs& a, cudaStream_t st) {
  // 16-byte aligned Ic (TMA) and q_idx (vector loads); anything else takes the CUDA-core kernel
  if (a.n_ih != kIHeads || a.hd != kIHd || (reinterpret_cast<uintptr_t>(a.Ic) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(a.q_idx) & 15u) != 0)
    return cudaErrorNotSupported;
  IdxTcParams p{};
  if (!make_tmap_2d_f32(&p.mI, a.Ic, (uint64_t)a.B * a.T_cap, kIHd, kIHd, kITile, 32)) return cudaErrorNotSupported;
  p.q = a.q_idx;
  p.w = a.w;
  p.T = a.T;
  p.scores = a.scores;
  p.B = a.B;
  p.S = a.S;
  p.T_cap = a.T_cap;
  p.ntiles = (a.T_cap + kITile - 1) / kITile;
  p.flags = a.flags;
  p.wait_ns = a.wait_ns;
  p.tpc = tiles_per_cta(a.B, a.S, a.T_cap);
  p.hpart = a.hpart;
  int dev = 0;
  cudaGetDevice(&dev);
  static int attr_done = -1;
  if (attr_done != dev) {
    cudaError_t e = cudaFuncSetAttribute(index_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kIDynSmem);
    if (e != cudaSuccess) return e;
    attr_done = dev;
  }
  dim3 grid((p.ntiles + p.tpc - 1) / p.tpc, a.S, a.B);
  index_tc_kernel<<<grid, kIThreads, kIDynSmem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
