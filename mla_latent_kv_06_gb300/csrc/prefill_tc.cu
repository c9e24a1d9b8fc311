// prefill_tc.cu -- tensor-core non-absorbed prefill for the GLM-5.2 shape
// (64 heads, qk_nope 192 + qk_rope 64, v_head 256).
//
// The non-absorbed path of the page "MLA 注意力与 KV 缓存", §2.3:
//   1. one kv_b product rebuilds k_nope and the value of every key,
//      KV[t, h, :] = kv_b[h] Lc[t]  -> the batched tcgen05 GEMM (gemm_tc.cu);
//   2. causal attention per head with score = q_pass . k_nope + q_rot . k_rot,
//      k_rot = Rc[t] shared by all heads, softmax, and a value sum.
//
// Step 2 is a flash-attention forward on tcgen05.  CTA = (128 queries, head,
// sequence).  Query rows live in the 128 TMEM lanes; two softmax threads share
// a row (64 keys of each tile and 128 value columns each), so max, sum and
// rescale stay in registers but for one shared-memory exchange.  Per
// 128-key tile j:
//   S(j)  = Q K(j)^T       M=128, N=128, K=256  (Q and K K-major)
//   O    += P(j-1) V(j-1)  M=128, N=256, K=128  (P from TMEM, V MN-major)
// A 128-key tile halves the score product's instructions and its re-reads of
// the query block against 64-key tiles; shared memory then holds one K and
// one V buffer (K released by the score product, V by the value product).
// S is double-buffered in TMEM, and P(j) is written as bf16 over the columns
// of S(j) that the writing thread has read: the value product takes its A
// operand from TMEM, so the softmax of tile j never waits for the value
// product of tile j - 1 (only a rescale of O does), and the S buffer is
// released by the value product's commit.
#include <atomic>
#include <cmath>

#include <cuda_fp16.h>

#include "common.cuh"
#include "gemm_tc.h"
#include "internal.h"
#include "prefill_tc.h"
#include "sm100.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace sm100;

constexpr int kH = 64, kDn = 192, kDr = 64, kDq = 256, kDv = 256, kDkv = kDn + kDv;  // kDkv = 448
constexpr int kQT = 128;                    // queries per CTA
constexpr int kKT = 128;                    // keys per tile
constexpr uint32_t kAtom = 128 * 128;       // 16 KB: 128 rows x 64 bf16 (one 128-byte swizzled atom)
constexpr uint32_t kQBytes = 4 * kAtom;     // 64 KB: 256 query dims
constexpr uint32_t kKBytes = 4 * kAtom;     // 64 KB: 192 k_nope + 64 k_rot dims of 128 keys
constexpr uint32_t kVBytes = 4 * kAtom;     // 64 KB: 256 value dims of 128 keys (MN-major atoms)
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kQBytes;
constexpr uint32_t kOffV = kOffK + kKBytes;
constexpr uint32_t kPrefillSmem = kOffV + kVBytes + 1024;
constexpr int kSoftThreads = 256;  // eight softmax warps
constexpr int kPThreads = 64 + kSoftThreads;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;    // two S buffers of 128 columns; P(j) over S(j): keys 64h.. at column 64h
constexpr uint32_t kTmemO = 256;  // O: 256 columns
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTau = 8.f;
constexpr long long kDrainNs = 1000000000LL;

struct FlashParams {
  CUtensorMap mQ;   // q as 3D {256 dims, 64 heads, B*S tokens}, box {64, 1, 128}
  CUtensorMap mKV;  // KV as 2D [B*Tk rows, 64*448 cols], box {64 cols, 64 rows}
  CUtensorMap mR;   // Rc as 2D [B*Tk rows, 64 cols], box {64, 64 rows}
  const __nv_bfloat16* q;
  float* out;
  int B, S, Tk, pos_base;
  float c;                // softmax scale * log2(e)
  uint64_t turn[kDr / 2];  // rope_turns(rope_base^(-2j/qk_rope))
  unsigned int* flags;
  long long wait_ns;
};

__global__ void __launch_bounds__(kPThreads, 1) flash_kernel(const __grid_constant__ FlashParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  unsigned char* sQ = smem + kOffQ;
  unsigned char* sK = smem + kOffK;
  unsigned char* sV = smem + kOffV;
  // Single K and V buffers (k_full / v_full complete once per tile, phase j
  // for tile j); S/P is double-buffered.  Two commits per tile signal the
  // MMA side: s_full[j & 1] once S(j) = Q K(j)^T retired (the softmax reads
  // S(j); the producer may reload K), pv_done[j & 1] once O += P(j) V(j)
  // retired (the producer may reload V, the MMA warp may reuse the S/P
  // buffer, a rescale or the final read may touch O); both are in phase
  // j >> 1 for tile j.  No waiter can fall two phases behind: the MMA order
  // is S(0), S(1), PV(0), S(2), PV(1), ..., so S(j) retired implies PV(j - 2)
  // retired, and the next phase of each barrier needs the waiter's own next
  // step (a K or V load, a P, or the MMA warp's issue).
  __shared__ uint64_t q_full, q_rope, k_full, v_full, s_full[2], pv_done[2], p_full, mma_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  // [half][row]: the halves' maxima, after the loop their row sums.  A thread
  // rewrites its entry only after the bar.red that ends each tile, which its
  // partner reaches after reading it.
  __shared__ float red_row[2][kQT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int s0 = qt * kQT;
  const int s_end = min(s0 + kQT, p.S);
  const int nkt = (p.pos_base + s_end + kKT - 1) / kKT;  // key tiles holding keys <= the last query

  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&q_rope, kSoftThreads);
    mbar_init(&k_full, 1);
    mbar_init(&v_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(&p_full, kSoftThreads);
    mbar_init(&mma_done, 1);
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&p.mQ);
    prefetch_tensormap(&p.mKV);
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
  grid_dep_wait();  // KV comes from the kv_b GEMM

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      mbar_arrive_expect_tx(&q_full, 3 * kAtom);
      for (int a = 0; a < 3; ++a) tma_load_3d(sQ + a * kAtom, &p.mQ, 64 * a, h, b * p.S + s0, &q_full);
      // K(j) waits for the score product of tile j - 1, V(j) for the value
      // product of tile j - 1: the key half of the stream runs one tile ahead.
      int last_k = -1, last_v = -1;
      auto load_k = [&](int j) -> bool {
        if (j > 0 && !mbar_wait(&s_full[(j - 1) & 1], ((j - 1) >> 1) & 1, abort, p.flags, p.wait_ns)) return false;
        const int y = b * p.Tk + j * kKT;
        mbar_arrive_expect_tx(&k_full, kKBytes);
        for (int a = 0; a < 3; ++a) tma_load_2d(sK + a * kAtom, &p.mKV, h * kDkv + 64 * a, y, &k_full);
        tma_load_2d(sK + 3 * kAtom, &p.mR, 0, y, &k_full);
        last_k = j;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        if (j > 0 && !mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort, p.flags, p.wait_ns)) return false;
        const int y = b * p.Tk + j * kKT;
        mbar_arrive_expect_tx(&v_full, kVBytes);
        for (int a = 0; a < 4; ++a) tma_load_2d(sV + a * kAtom, &p.mKV, h * kDkv + kDn + 64 * a, y, &v_full);
        last_v = j;
        return true;
      };
      if (nkt > 0) ok = load_k(0);
      for (int j = 0; j < nkt && ok; ++j) {
        if (j + 1 < nkt) ok = load_k(j + 1);  // the score product S(j) retires before O(j - 1)
        if (ok) ok = load_v(j);
      }
      volatile int no_abort = 0;
      const long long dn = p.wait_ns > kDrainNs ? p.wait_ns : kDrainNs;
      mbar_wait(&q_full, 0, &no_abort, p.flags, dn);
      if (last_k >= 0) mbar_wait(&k_full, last_k & 1, &no_abort, p.flags, dn);
      if (last_v >= 0) mbar_wait(&v_full, last_v & 1, &no_abort, p.flags, dn);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, kKT, 0, 0);
      const uint32_t idesc_o = idesc_bf16_f32(128, kDv, 0, 1);
      const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK), v0 = smem_u32(sV);
      bool ok = mbar_wait(&q_full, 0, abort, p.flags, p.wait_ns) && mbar_wait(&q_rope, 0, abort, p.flags, p.wait_ns);
      bool issued = false;
      auto pv = [&](int j) -> bool {  // O += P(j) V(j)
        if (!mbar_wait(&p_full, j & 1, abort, p.flags, p.wait_ns)) return false;
        if (!mbar_wait(&v_full, j & 1, abort, p.flags, p.wait_ns)) return false;
        tc_fence_after();
        const uint32_t pj = tmem + kTmemS + kKT * (j & 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // 16 keys per step: 8 columns of P, V rows 16 kk ..
          const uint64_t db = smem_desc_sw128(v0 + kk * 2048, kAtom, 1024);
          mma_bf16_ts(tmem + kTmemO, pj + (kk >> 2) * 64 + (kk & 3) * 8, db, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&pv_done[j & 1]);
        return true;
      };
      for (int j = 0; j < nkt && ok; ++j) {
        const int st = j & 1, n = j >> 1;
        ok = mbar_wait(&pv_done[st], (n & 1) ^ 1, abort, p.flags, p.wait_ns) &&  // PV(j - 2) read P from it
             mbar_wait(&k_full, j & 1, abort, p.flags, p.wait_ns);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t da = smem_desc_sw128(q0 + a * kAtom + kk * 32, 16, 1024);
            const uint64_t db = smem_desc_sw128(k0 + a * kAtom + kk * 32, 16, 1024);
            mma_bf16(tmem + kTmemS + kKT * st, da, db, idesc_s, (a | kk) != 0);
          }
        mma_commit(&s_full[st]);
        issued = true;
        if (j > 0) ok = pv(j - 1);
      }
      if (ok && nkt > 0) ok = pv(nkt - 1);
      if (issued) {
        mma_commit(&mma_done);
        volatile int no_abort = 0;
        mbar_wait(&mma_done, 0, &no_abort, p.flags, p.wait_ns > kDrainNs ? p.wait_ns : kDrainNs);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps 2..9
    // Thread (row m, half) owns keys 64*half .. 64*half+63 of each tile of
    // query row m and value columns 128*half .. 128*half+127; the two halves of
    // a row exchange their maxima through shared memory.
    const int wq = warp & 3;
    const int half = (warp - 2) >> 2;
    const int m = 32 * wq + lane;
    const int s = s0 + m;
    const bool row_ok = s < p.S;
    const int pos = p.pos_base + s;
    const uint32_t t_lane = (uint32_t)(32 * wq) << 16;
    // rotary part of the query row into Q atom 3 (128-byte swizzled like TMA
    // would): this half writes y[16*half ..] and y[32 + 16*half ..]
    {
      uint32_t lo[8], hi[8];
      if (row_ok) {
        const __nv_bfloat16* qr = p.q + (((size_t)b * p.S + s) * kH + h) * kDq + kDn;
#pragma unroll
        for (int u = 0; u < 16; u += 2) {
          float r0[2], r1[2];
#pragma unroll
          for (int v2 = 0; v2 < 2; ++v2) {
            const int jj = 16 * half + u + v2;
            float sn, cs;
            rope_cs_turns(pos, p.turn[jj], &cs, &sn);
            const float x0 = __bfloat162float(qr[2 * jj]), x1 = __bfloat162float(qr[2 * jj + 1]);
            r0[v2] = x0 * cs - x1 * sn;   // -> y[jj]
            r1[v2] = x1 * cs + x0 * sn;   // -> y[32 + jj]
          }
          lo[u / 2] = pack2(r0[0], r0[1]);
          hi[u / 2] = pack2(r1[0], r1[1]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) lo[i] = hi[i] = 0u;
      }
      unsigned char* row = sQ + 3 * kAtom + m * 128;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c_lo = 2 * half + cc, c_hi = 4 + 2 * half + cc;
        *reinterpret_cast<uint4*>(row + ((c_lo ^ (m & 7)) << 4)) = make_uint4(lo[4 * cc], lo[4 * cc + 1], lo[4 * cc + 2], lo[4 * cc + 3]);
        *reinterpret_cast<uint4*>(row + ((c_hi ^ (m & 7)) << 4)) = make_uint4(hi[4 * cc], hi[4 * cc + 1], hi[4 * cc + 2], hi[4 * cc + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&q_rope);
    }
    const float c = p.c;
    float m_run = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkt && ok; ++j) {
      const int st = j & 1;
      // failed waits are decided jointly by the 256 softmax threads (bar.red),
      // so that none is left at a barrier the others quit
      bool fail = !mbar_wait(&s_full[st], (j >> 1) & 1, abort, p.flags, p.wait_ns);
      if (bar_red_or(2, kSoftThreads, fail)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float v[64];
      tmem_ld64(tmem + t_lane + kTmemS + kKT * st + 64 * half, v);
      tmem_wait_ld();
      const int t0 = j * kKT + 64 * half;
      const int nvalid = row_ok ? max(0, min(64, pos - t0 + 1)) : 0;  // keys t0..t0+nvalid-1 are visible
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 64; ++i)
        if (i < nvalid) mx = fmaxf(mx, v[i]);
      red_row[half][m] = mx;
      named_barrier(1, kSoftThreads);
      mx = fmaxf(red_row[0][m], red_row[1][m]);
      float alpha = 1.f;
      const float cand = mx * c;
      if (cand > m_run + kTau) {
        alpha = exp2f(m_run - cand);
        m_run = cand;
      }
      // Probabilities two at a time through the half-precision exp2 (one
      // MUFU operation per pair, the exponent unit being this loop's limit):
      // the arguments are <= 0 and P is rounded to bf16 for the value
      // product anyway; masked keys get -inf, whose exp2 is exactly 0.
      uint32_t pk[32];
      float psum = 0.f;
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        const float x0 = i < nvalid ? fmaf(v[i], c, -m_run) : -INFINITY;
        const float x1 = i + 1 < nvalid ? fmaf(v[i + 1], c, -m_run) : -INFINITY;
        const float2 e = __half22float2(h2exp2(__floats2half2_rn(x0, x1)));
        pk[i / 2] = pack2(e.x, e.y);
        const float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&pk[i / 2]));
        psum += f.x + f.y;
      }
      l = l * alpha + psum;
      // A rescale rewrites O: it waits until O += P(j - 1) V(j - 1) retired
      // (tcgen05.ld/st are warp-wide, so the warp decides together).
      fail = false;
      if (__any_sync(0xffffffffu, alpha != 1.f && j > 0)) {
        fail = !__all_sync(0xffffffffu, mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort, p.flags, p.wait_ns));
        if (!fail) {
          tc_fence_after();
#pragma unroll 1
          for (int cb = 128 * half; cb < 128 * half + 128; cb += 64) {
            float w[64];
            tmem_ld64(tmem + t_lane + kTmemO + cb, w);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 64; ++i) w[i] *= alpha;
            tmem_st64(tmem + t_lane + kTmemO + cb, w);
          }
        }
      }
      if (!fail) {
        // P(j): this thread's 64 keys as 32 bf16 pairs, over the first half of
        // the 64 columns of S(j) it read (the other thread of the row writes
        // its own columns)
        tmem_st32(tmem + t_lane + kTmemS + kKT * st + 64 * half, reinterpret_cast<const float*>(pk));
        tmem_wait_st();
      }
      if (bar_red_or(2, kSoftThreads, fail)) {
        ok = false;
        break;
      }
      tc_fence_before();
      mbar_arrive(&p_full);
    }
    // row sums: the two halves of a row
    red_row[half][m] = l;
    bool fail = !ok;
    if (!fail && nkt > 0) fail = !mbar_wait(&pv_done[(nkt - 1) & 1], ((nkt - 1) >> 1) & 1, abort, p.flags, p.wait_ns);
    if (!bar_red_or(2, kSoftThreads, fail) && nkt > 0) {
      tc_fence_after();
      float* orow = p.out + (((size_t)b * p.S + s) * kH + h) * kDv;
      const float il = 1.f / (red_row[0][m] + red_row[1][m]);
#pragma unroll 1
      for (int cb = 128 * half; cb < 128 * half + 128; cb += 64) {
        float w[64];
        tmem_ld64(tmem + t_lane + kTmemO + cb, w);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 64; i += 4)
            *reinterpret_cast<float4*>(orow + cb + i) = make_float4(w[i] * il, w[i + 1] * il, w[i + 2] * il, w[i + 3] * il);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

std::atomic<unsigned long long> g_flash_attr{0};

}  // namespace

bool tc_prefill_geometry_ok(const Geometry& g) {
  return g.H == kH && g.Dn == kDn && g.Dr == kDr && g.Dv == kDv && g.Dl >= 64 && g.Dl % 64 == 0 && g.Dl <= 4096;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, unsigned int* flags, long long wait_ns, cudaStream_t st) {
  const Geometry& g = a.g;
  const int Tk = a.pos_base + a.S;
  // 1. KV[t, h*448 + j] = sum_l Lc[t, l] kv_b[h*448 + j, l]
  GemmArgs ga{};
  ga.a_base = a.Lc;
  ga.a_ld_z = g.Dl;
  ga.a_ld_m = g.Dl;
  ga.b_base = a.kv_b;
  ga.b_rows = (long long)kH * kDkv;
  ga.b_cols = g.Dl;
  ga.b_ld = g.Dl;
  ga.b_mn_major = 0;
  ga.b_row0 = 0;
  ga.b_rows_per_z = 0;
  ga.b_col0 = 0;
  ga.c_base = a.kv;
  ga.c_ld_m = (long long)kH * kDkv;
  ga.c_ld_z = 0;
  ga.out_kind = kGemmOutBf16;
  ga.M = a.B * Tk;
  ga.N = kH * kDkv;
  ga.K = g.Dl;
  ga.Z = 1;
  ga.flags = flags;
  ga.wait_ns = wait_ns;
  kernel_mark(st, "kv_gemm");
  cudaError_t e = launch_gemm_tc(ga, false, st);
  if (e != cudaSuccess) return e;
  // 2. causal flash attention over the rebuilt keys / values
  FlashParams fp{};
  const uint64_t qdims[3] = {(uint64_t)kDq, (uint64_t)kH, (uint64_t)a.B * a.S};
  const uint64_t qstr[2] = {(uint64_t)kDq * 2, (uint64_t)kH * kDq * 2};
  const uint32_t qbox[3] = {64, 1, (uint32_t)kQT};
  if (!make_tmap_3d_bf16(&fp.mQ, a.q, qdims, qstr, qbox) ||
      !make_tmap_2d_bf16(&fp.mKV, a.kv, (uint64_t)a.B * Tk, (uint64_t)kH * kDkv, (uint64_t)kH * kDkv, kKT, 64) ||
      !make_tmap_2d_bf16(&fp.mR, a.Rc, (uint64_t)a.B * Tk, kDr, kDr, kKT, 64))
    return cudaErrorInvalidValue;
  fp.q = static_cast<const __nv_bfloat16*>(a.q);
  fp.out = a.out;
  fp.B = a.B;
  fp.S = a.S;
  fp.Tk = Tk;
  fp.pos_base = a.pos_base;
  fp.c = g.scale * kLog2e;
  for (int j = 0; j < kDr / 2; ++j) fp.turn[j] = rope_turns(std::pow(g.rope_base, -2.0 * j / kDr));
  fp.flags = flags;
  fp.wait_ns = wait_ns;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(g_flash_attr.load() & bit)) {
    e = cudaFuncSetAttribute(flash_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrefillSmem);
    if (e != cudaSuccess) return e;
    g_flash_attr.fetch_or(bit);
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((a.S + kQT - 1) / kQT, kH, a.B);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPrefillSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  kernel_mark(st, "flash_attention");
  return cudaLaunchKernelEx(&cfg, flash_kernel, fp);
}

}  // namespace mla
