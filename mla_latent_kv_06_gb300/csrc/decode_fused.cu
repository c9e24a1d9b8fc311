// decode_fused.cu -- the absorbed decode of a few query rows (B*S <= 4) in a
// single launch: absorb, attention, split merge and W_UV lift as the phases
// of one persistent grid of one CTA per SM.
//
// The method is the absorbed path of the page "MLA 注意力与 KV 缓存", §2.3:
// qabs = W_UK^T q_nope, scores qabs . Lc + q_rot . Rc, softmax, latent context
// clat = sum p Lc, out = W_UV clat.  At a handful of query rows every step is
// a stream of weights or cache rows with little arithmetic, so the time of a
// chain of kernels is their hand-over latency rather than their bytes.  Here
// the three streams (W_UK, the cache, W_UV) start together and the phases
// hand over through global-memory flags:
//
//   phase A  (warps 2-9)  qabs for 64-column blocks of W_UK, dealt over all
//                         CTAs; the rotated query tail; -> qcat (bf16).
//            meanwhile warp 0 has the CTA's first key tile in flight and
//            warp 10 pulls this CTA's share of W_UV into L2.
//   barrier 1             every CTA has written its part of qcat.
//   phase B  (warps 0-9)  the attention pass of attn_core.cuh over this
//                         CTA's share of the key tiles -> (m, l, O) partials.
//   barrier 2             every partial is written.
//   phase C  (all warps)  per (head, 128-latent quarter): log-sum-exp merge of
//                         the partials, then the quarter's share of W_UV clat
//                         (W_UV registers loaded before the barrier wait); the
//                         last quarter of a head to finish sums the four.
//
// The flags live in the caller's workspace.  A call's token is one more than
// the epoch word it reads at start (CTA 0 advances the epoch once every CTA
// has read it), and a barrier is complete when every CTA's arrival word holds
// the token, so no memory needs clearing between calls: stale words hold an
// older token, and memory other calls wrote matches a 64-bit token only by a
// 2^-64 accident.  Every wait is bounded by the call's wait limit.
#include <atomic>
#include <cmath>

#include "attn_core.cuh"
#include "decode_tc.h"
#include "tmap.h"

namespace mla {
namespace {

constexpr int kFusedRows = 4;                     // query rows (B*S) of this path
constexpr int kSyncWarp = 10;                     // grid barriers, epoch, query-row copies
constexpr int kFusedThreads = kAttnThreads + 32;  // 352
constexpr int kAbsUnitCols = 64;                  // W_UK columns per phase-A unit
constexpr int kAbsUnits = kH * (kDl / kAbsUnitCols);  // 512
constexpr int kMaxAbsPerCta = 4;                  // units per CTA (grids of >= 128 CTAs)
constexpr int kLiftUnits = kH * 2;                // (head, half of the v_head rows): one per CTA
constexpr int kLiftRows = 128;                    // W_UV rows (output columns) per lift unit
constexpr int kMaxGrid = 256;                     // CTAs (one per SM)
constexpr int kMaxDq = 320;                       // qk_nope + qk_rope, qk_nope <= 256
constexpr uint32_t kFusedDynSmem = kQBytes + kKVBytes + 1024;
constexpr uint32_t kLiftWBytes = kLiftRows * kDl * 2;  // 128 W_UV rows of one head, bf16 (contiguous)

// Phase-A scratch inside the query-block space (free until barrier 1).
constexpr uint32_t kRedOff = 0;                                          // [4][R][8][64] fp32
constexpr uint32_t kQRowOff = kMaxAbsPerCta * kFusedRows * 8 * kAbsUnitCols * 4;  // 32 KB
// Phase-C scratch inside the query-block space (free after the attention).
constexpr uint32_t kCRedOff = 0;                                         // [11][512] fp32
constexpr uint32_t kCMlOff = 11 * kDl * 4;                               // [11][2] fp32
constexpr uint32_t kClatOff = kCMlOff + 128;                             // [R][512] fp32
static_assert(kClatOff + kFusedRows * kDl * 4 <= kQBytes, "phase-C scratch");
static_assert(kQRowOff + kMaxAbsPerCta * kFusedRows * kMaxDq * 2 <= kQBytes, "phase-A scratch");
static_assert(kLiftWBytes <= kKVBytes, "W_UV half block");

struct FusedParams {
  AttnParams at;
  const __nv_bfloat16* q;     // [R, 64, Dn + 64]
  const __nv_bfloat16* kv_b;  // [64, Dn + Dv, 512]
  __nv_bfloat16* qcat;        // [R, 64, 576]
  float* out;                 // [R, 64, Dv]
  unsigned long long* epoch;  // 1 word
  unsigned long long* arr1;   // [grid] barrier-1 arrival words
  unsigned long long* arr2;   // [grid] barrier-2 arrival words
  int Dn, Dv, R, attn_ctas;
  uint64_t turn[kDr / 2];     // rope_turns(rope_base^(-2j/qk_rope))
};

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Contiguous global -> shared copy by the bulk-copy engine, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// One warp waits until arr[0..n) all hold tok: every lane reads its words
// with independent relaxed loads per round, and one acquire fence follows.
// Returns false (and raises MLA_DEV_TIMEOUT) when the limit runs out first.
__device__ bool grid_wait(const unsigned long long* arr, int n, unsigned long long tok, long long limit_ns,
                          unsigned int* flags) {
  constexpr int kPer = kMaxGrid / 32;
  const int lane = threadIdx.x & 31;
  uint32_t seen = 0;  // bit k: word lane + 32k holds tok (or does not exist)
#pragma unroll
  for (int k = 0; k < kPer; ++k)
    if (lane + 32 * k >= n) seen |= 1u << k;
  const uint32_t want = (1u << kPer) - 1u;
  const unsigned long long t0 = global_ns();
  for (;;) {
    unsigned long long v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) v[k] = ((seen >> k) & 1u) ? tok : ld_relaxed_u64(arr + lane + 32 * k);
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if (v[k] == tok) seen |= 1u << k;
    if (__all_sync(0xffffffffu, seen == want)) break;
    if ((long long)(global_ns() - t0) > limit_ns) {
      if (lane == 0) raise_flag(flags, MLA_DEV_TIMEOUT);
      return false;
    }
  }
  fence_acq_rel_gpu();
  return true;
}

// ---------------------------------------------------------------- phase A
// Unit u = (head h, 64-column block cb): qcat[r, h, 64cb + c] = sum_i q[r,h,i]
// W_UK[h][i][64cb + c] for every row r.  256 threads: thread t holds 8
// columns (t & 7) of rows (t >> 3) + 32k.  Units of this CTA: u = blockIdx.x +
// k * gridDim.x; their W_UK loads are all in flight before the first product.
__device__ __forceinline__ int absorb_units(int* units) {
  int nu = 0;
  for (int u = blockIdx.x; u < kAbsUnits && nu < kMaxAbsPerCta; u += gridDim.x) units[nu++] = u;
  return nu;
}

template <int NV>  // NV = Dn / 32 rows per thread
__device__ __forceinline__ void absorb_load(const FusedParams& fp, const int* units, int nu,
                                            uint4 (&wv)[kMaxAbsPerCta][NV]) {
  const int t = threadIdx.x - 64;  // 0..255
  const int c8 = t & 7, rg = t >> 3;
#pragma unroll
  for (int k = 0; k < kMaxAbsPerCta; ++k)
    if (k < nu) {
      const int h = units[k] / (kDl / kAbsUnitCols), cb = units[k] % (kDl / kAbsUnitCols);
      const __nv_bfloat16* W = fp.kv_b + (size_t)h * (fp.Dn + fp.Dv) * kDl + cb * kAbsUnitCols + c8 * 8;
#pragma unroll
      for (int v = 0; v < NV; ++v) wv[k][v] = __ldg(reinterpret_cast<const uint4*>(W + (size_t)(rg + 32 * v) * kDl));
    }
}

// The query rows of the CTA's units (q[r, h, 0:Dq] for each unit k and row r)
// land in shared memory by bulk copies that one warp issues at kernel start.
__device__ __forceinline__ void issue_qrow_copies(const FusedParams& fp, const int* units, int nu,
                                                  unsigned char* smem, uint64_t* bar) {
  const int lane = threadIdx.x & 31;
  const int Dq = fp.Dn + kDr, R = fp.R;
  const uint32_t row_bytes = (uint32_t)Dq * 2;
  if (lane == 0) mbar_arrive_expect_tx(bar, row_bytes * nu * R);
  __syncwarp();
  if (lane < nu * R) {
    const int k = lane / R, r = lane % R;
    const int h = units[k] / (kDl / kAbsUnitCols);
    bulk_g2s(smem + kQRowOff + (k * kFusedRows + r) * kMaxDq * 2, fp.q + ((size_t)r * kH + h) * Dq, row_bytes, bar);
  }
}

// Rotary tail of each unit of column block 0: thread t < R * 32 handles pair
// j = t % 32 of row r = t / 32 at pos = T[b] - S + s; Tr is T[b] of that row,
// loaded at kernel start.
__device__ __forceinline__ void absorb_rotary(const FusedParams& fp, const int* units, int nu, int Tr,
                                              const __nv_bfloat16* qrow) {
  const int t = threadIdx.x - 64;
  if (t >= fp.R * (kDr / 2)) return;
  const int r = t / (kDr / 2), j = t % (kDr / 2);
  const int S = fp.at.S, s = r % S;
  const int pos = (Tr < S || Tr > fp.at.T_cap) ? 0 : Tr - S + s;
  float sn, cs;
  rope_cs_turns(pos, fp.turn[j], &cs, &sn);
  for (int k = 0; k < nu; ++k) {
    const int h = units[k] / (kDl / kAbsUnitCols), cb = units[k] % (kDl / kAbsUnitCols);
    if (cb != 0) continue;
    const __nv_bfloat16* qr = qrow + (k * kFusedRows + r) * kMaxDq + fp.Dn;
    const float x0 = __bfloat162float(qr[2 * j]), x1 = __bfloat162float(qr[2 * j + 1]);
    __nv_bfloat16* dst = fp.qcat + ((size_t)r * kH + h) * kDc + kDl;
    dst[j] = __float2bfloat16_rn(x0 * cs - x1 * sn);
    dst[kDr / 2 + j] = __float2bfloat16_rn(x1 * cs + x0 * sn);
  }
}

template <int NV>
__device__ __forceinline__ void phase_absorb(const FusedParams& fp, const int* units, int nu,
                                             const uint4 (&wv)[kMaxAbsPerCta][NV], unsigned char* smem,
                                             uint64_t* qrow_bar, volatile int* abort, int Tr) {
  const int t = threadIdx.x - 64;  // 0..255
  const int c8 = t & 7, rg = t >> 3;
  const int warp = t >> 5, lane = t & 31;
  const int Dn = fp.Dn, R = fp.R;
  float* red = reinterpret_cast<float*>(smem + kRedOff);  // [4][R][8 warps][64]
  const __nv_bfloat16* qrow = reinterpret_cast<const __nv_bfloat16*>(smem + kQRowOff);
  mbar_wait(qrow_bar, 0, abort, fp.at.flags, fp.at.wait_ns > kDrainNs ? fp.at.wait_ns : kDrainNs);
  absorb_rotary(fp, units, nu, Tr, qrow);  // needs only the query rows: done while W_UK lands
#pragma unroll
  for (int k = 0; k < kMaxAbsPerCta; ++k) {
    if (k >= nu) break;
    for (int r = 0; r < R; ++r) {
      const __nv_bfloat16* qr = qrow + (k * kFusedRows + r) * kMaxDq;
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const float qv = __bfloat162float(qr[rg + 32 * v]);
        const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&wv[k][v]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __bfloat1622float2(w2[j]);
          acc[2 * j] = fmaf(qv, f.x, acc[2 * j]);
          acc[2 * j + 1] = fmaf(qv, f.y, acc[2 * j + 1]);
        }
      }
      // sum over the warp's four row groups (lane bits 3, 4)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], 8);
        acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], 16);
      }
      if (lane < 8) {
        float* d = red + ((k * kFusedRows + r) * 8 + warp) * kAbsUnitCols + c8 * 8;
        *reinterpret_cast<float4*>(d) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4*>(d + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
      }
    }
  }
  named_barrier(1, kSoftThreads);
  for (int e = t; e < nu * R * kAbsUnitCols; e += kSoftThreads) {
    const int k = e / (R * kAbsUnitCols), r = (e / kAbsUnitCols) % R, col = e % kAbsUnitCols;
    const float* src = red + ((k * kFusedRows + r) * 8) * kAbsUnitCols + col;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) v += src[w * kAbsUnitCols];
    const int h = units[k] / (kDl / kAbsUnitCols), cb = units[k] % (kDl / kAbsUnitCols);
    fp.qcat[((size_t)r * kH + h) * kDc + cb * kAbsUnitCols + col] = __float2bfloat16_rn(v);
  }
  // qcat is read by other CTAs' TMA copies, and the scratch becomes the TMA
  // destination of the query block: order these generic accesses before both.
  fence_proxy_async_global();
  fence_proxy_async_smem();
}

// ---------------------------------------------------------------- phase C
// Lift unit u = (head h, row half qv), one per CTA u < 128: the log-sum-exp
// merge of head h's partials of every row into clat (all 512 latent columns),
// then out[r, h, 128 qv + v] = W_UV[h][128 qv + v] . clat[r] for v < 128.  The
// unit's 128 W_UV rows are one contiguous 128 KB block that a bulk copy brings
// into the free key-tile space when the CTA's attention work is done.
__device__ __forceinline__ const __nv_bfloat16* lift_w(const FusedParams& fp, int u) {
  return fp.kv_b + ((size_t)(u >> 1) * (fp.Dn + fp.Dv) + fp.Dn + kLiftRows * (u & 1)) * kDl;
}

struct LiftShared {
  int nslot[kFusedRows];
  short slot[kFusedRows][kMaxGrid + kFusedRows];
};

// Partial slots of every row, in chunk order (one warp per row).
__device__ void list_pieces(const FusedParams& fp, const int32_t* ts, long long N, LiftShared& ls, int r) {
  const AttnParams& p = fp.at;
  const int lane = threadIdx.x & 31;
  const int b = r / p.S, s = r % p.S;
  int cnt = 0;
  const long long a = ts[b], e = ts[b + 1];
  if (e > a && N > 0) {
    const int glo = chunk_of(a, N, p.G), ghi = chunk_of(e - 1, N, p.G);
    for (int g0 = glo; g0 <= ghi; g0 += 32) {
      const int gg = g0 + lane;
      int lo = 0, hi = 0;
      if (gg <= ghi) piece_range<false>(ts, p.T, p.S, s, b, gg, p.G, N, &lo, &hi);
      const bool has = lo < hi;
      const unsigned m = __ballot_sync(0xffffffffu, has);
      if (has) ls.slot[r][cnt + __popc(m & ((1u << lane) - 1))] = (short)((gg + b) * p.S + s);
      cnt += __popc(m);
    }
  }
  if (lane == 0) ls.nslot[r] = cnt;
}

__device__ void lift_unit(const FusedParams& fp, int u, const unsigned char* sw, const LiftShared& ls,
                          unsigned char* smem, uint64_t* wbar) {
  const AttnParams& p = fp.at;
  const int h = u >> 1, qv = u & 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int nw = kFusedThreads / 32;
  const int R = fp.R;
  float* red = reinterpret_cast<float*>(smem + kCRedOff);   // [11][512]
  float* mlw = reinterpret_cast<float*>(smem + kCMlOff);    // [11][2]
  float* clat = reinterpret_cast<float*>(smem + kClatOff);  // [R][512]
  for (int r = 0; r < R; ++r) {
    // (a) warp w merges pieces w, w + 11, ... with a running maximum: the
    // (m, l) pair and the O row of a piece load together.
    const int cnt = ls.nslot[r];
    float m = -INFINITY, l = 0.f;
    float4 acc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
    for (int i = warp; i < cnt; i += nw) {
      const size_t row = (size_t)ls.slot[r][i] * kH + h;
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.ml_part + row * 2));
      const float4* o = reinterpret_cast<const float4*>(p.o_part + row * kDl);
      float4 x[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) x[j] = __ldcg(o + 32 * j + lane);
      const float mn = fmaxf(m, ml.x);
      const float so = m == -INFINITY ? 0.f : exp2f(m - mn);
      const float si = ml.x == -INFINITY ? 0.f : exp2f(ml.x - mn);
      m = mn;
      l = fmaf(l, so, ml.y * si);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[j].x = fmaf(acc[j].x, so, x[j].x * si);
        acc[j].y = fmaf(acc[j].y, so, x[j].y * si);
        acc[j].z = fmaf(acc[j].z, so, x[j].z * si);
        acc[j].w = fmaf(acc[j].w, so, x[j].w * si);
      }
    }
    float4* d = reinterpret_cast<float4*>(red + warp * kDl);
#pragma unroll
    for (int j = 0; j < 4; ++j) d[32 * j + lane] = acc[j];
    if (lane == 0) {
      mlw[2 * warp] = m;
      mlw[2 * warp + 1] = l;
    }
    __syncthreads();
    // (b) across the warps: clat = sum_w 2^(m_w - M) acc_w / sum_w 2^(m_w - M) l_w
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < nw; ++w) M = fmaxf(M, mlw[2 * w]);
    float L = 0.f, sc[nw];
#pragma unroll
    for (int w = 0; w < nw; ++w) {
      sc[w] = mlw[2 * w] == -INFINITY ? 0.f : exp2f(mlw[2 * w] - M);
      L = fmaf(sc[w], mlw[2 * w + 1], L);
    }
    // a row without keys (or a bad length) has L = 0: its outputs are NaN
    const float inv = (cnt > 0 && L > 0.f) ? 1.f / L : __int_as_float(0x7fc00000);
    for (int c = threadIdx.x; c < kDl; c += kFusedThreads) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < nw; ++w) v = fmaf(sc[w], red[w * kDl + c], v);
      clat[r * kDl + c] = v * inv;
    }
    __syncthreads();
  }
  // (c) out[r, h, 128 qv + v] = W_UV row v . clat[r]: warps 0-7, warp w rows
  // 16w .. 16w + 15; lane takes the 16-byte column chunks lane and lane + 32.
  if (warp < 8) {
    volatile int no_abort = 0;
    mbar_wait(wbar, 0, &no_abort, p.flags, p.wait_ns > kDrainNs ? p.wait_ns : kDrainNs);
    for (int r = 0; r < R; ++r) {
      float cv[16];
      const float* cr = clat + r * kDl;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        *reinterpret_cast<float4*>(&cv[8 * j]) = *reinterpret_cast<const float4*>(cr + 256 * j + lane * 8);
        *reinterpret_cast<float4*>(&cv[8 * j + 4]) = *reinterpret_cast<const float4*>(cr + 256 * j + lane * 8 + 4);
      }
      float d[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const unsigned char* wrow = sw + (size_t)(16 * warp + k) * (kDl * 2);
        float a = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint4 w = *reinterpret_cast<const uint4*>(wrow + 512 * j + lane * 16);
          const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(w2[e]);
            a = fmaf(f.x, cv[8 * j + 2 * e], a);
            a = fmaf(f.y, cv[8 * j + 2 * e + 1], a);
          }
        }
        d[k] = a;
      }
      // sum over the 32 lanes: the lane halves first, then a transposing
      // reduction over 16 lanes; afterwards lane L < 16 holds row 16w + L.
#pragma unroll
      for (int k = 0; k < 16; ++k) d[k] += __shfl_xor_sync(0xffffffffu, d[k], 16);
#pragma unroll
      for (int step = 0; step < 4; ++step) {
        const int o = 8 >> step;
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
          const float send = upper ? d[i] : d[i + o];
          const float keep = upper ? d[i + o] : d[i];
          d[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      if (lane < 16)
        fp.out[((size_t)r * kH + h) * fp.Dv + kLiftRows * qv + 16 * warp + lane] = d[0];
    }
  }
}

template <int NV>
__global__ void __launch_bounds__(kFusedThreads, 1) fused_decode_kernel(const __grid_constant__ FusedParams fp) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  __shared__ AttnShared sh;
  __shared__ int plan_ts[kFusedRows + 1];
  __shared__ uint64_t qready, wbar, qrow_bar, plan_bar;
  __shared__ int q_failed;
  __shared__ unsigned long long tok_sh;
  __shared__ LiftShared ls;
  const AttnParams& p = fp.at;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.S;
  const bool attn = (int)blockIdx.x < fp.attn_ctas;
  const bool lift = (int)blockIdx.x < kLiftUnits;
  const int part = attn ? (int)blockIdx.x % p.qsplit : 0, brow = attn ? (int)blockIdx.x / p.qsplit : 0;
  const bool absorb_warp = warp >= 2 && warp < kSyncWarp;

  // W_UK of this CTA's phase-A units: the first bytes the grid asks for.
  int units[kMaxAbsPerCta];
  const int nu = absorb_units(units);
  uint4 wv[kMaxAbsPerCta][NV];
  int Tr = 0;  // T[b] of the row whose rotary pairs this thread takes
  if (absorb_warp) {
    const int t = threadIdx.x - 64;
    if (t < fp.R * (kDr / 2)) Tr = __ldg(p.T + (t / (kDr / 2)) / S);
    absorb_load<NV>(fp, units, nu, wv);
  }

  if (warp == kSyncWarp) {
    if (lane == 0) {
      mbar_init(&qrow_bar, 1);
      fence_mbar_init();
    }
    __syncwarp();
    issue_qrow_copies(fp, units, nu, smem, &qrow_bar);
  } else if (threadIdx.x == 0) {
    attn_init_barriers(sh);
    mbar_init(&qready, 1);
    mbar_init(&wbar, 1);
    mbar_init(&plan_bar, 1);
    q_failed = 0;
    fence_mbar_init();
    if (attn) {
      prefetch_tensormap(&p.mQ);
      prefetch_tensormap(&p.mL);
      prefetch_tensormap(&p.mR);
    }
  }
  if (warp == 1 && attn) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // Tile-start prefix over the B <= 4 sequences, built by warp 0 (the
  // producer) and published through plan_bar to the other attention roles.
  if (warp == 0) {
    int x = lane < p.B ? row_tiles<false>(p, lane) : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane < p.B) plan_ts[lane + 1] = x;
    if (lane == 0) plan_ts[0] = 0;
    __syncwarp();
    if (lane == 0) mbar_arrive(&plan_bar);
  }

  AttnCtx cx;
  cx.NR = p.B;
  cx.ts = plan_ts;
  cx.g = brow / S;
  cx.s = brow % S;
  cx.part = part;
  cx.mb0 = part * (4 / p.qsplit);
  cx.mb1 = cx.mb0 + 4 / p.qsplit;
  cx.sQ = smem;
  cx.sKV = smem + kQBytes;
  cx.tmem = sh.tmem_base;
  auto plan_ready = [&]() {
    volatile int no_abort = 0;
    mbar_wait(&plan_bar, 0, &no_abort, p.flags, p.wait_ns > kDrainNs ? p.wait_ns : kDrainNs);
    cx.N = cx.ts[cx.NR];
    cx.row0 = first_row(cx.ts, cx.NR, chunk_begin(cx.N, cx.g, p.G));
  };

  if (warp == 0) {
    plan_ready();
    if (attn && lane == 0)
      attn_producer<false, false>(p, sh, cx, [&]() -> bool {
        volatile int no_abort = 0;
        if (!mbar_wait(&qready, 0, &no_abort, p.flags, p.wait_ns > kDrainNs ? p.wait_ns : kDrainNs)) return false;
        fence_proxy_async_global();  // qcat was written by other CTAs' generic stores
        return q_failed == 0;
      });
    __syncwarp();
  } else if (warp == 1) {
    plan_ready();
    if (attn) attn_mma<false>(p, sh, cx);
  } else if (absorb_warp) {
    phase_absorb<NV>(fp, units, nu, wv, smem, &qrow_bar, &sh.abort_flag, Tr);
    named_barrier(3, kSoftThreads + 32);  // phase A of this CTA done -> the sync warp arrives
    plan_ready();
    if (attn) attn_softmax<false>(p, sh, cx);
  } else {
    // sync warp: the epoch gives this call's token; barrier 1 (all of qcat
    // written); then the W_UV bytes into L2 while the attention runs.
    const unsigned long long tok = *reinterpret_cast<volatile unsigned long long*>(fp.epoch) + 1ull;
    if (lane == 0) tok_sh = tok;
    named_barrier(3, kSoftThreads + 32);
    if (lane == 0) st_release_u64(fp.arr1 + blockIdx.x, tok);
    const bool ok = grid_wait(fp.arr1, gridDim.x, tok, p.wait_ns, p.flags);
    if (lane == 0) {
      if (!ok) q_failed = 1;
      if (attn) mbar_arrive(&qready);
      if (lift) l2_prefetch(lift_w(fp, blockIdx.x), kLiftWBytes);  // the lift unit's W_UV rows
    }
    __syncwarp();
    // the lift unit's partial slots, while the attention runs
    if (lift) {
      volatile int no_abort = 0;
      mbar_wait(&plan_bar, 0, &no_abort, p.flags, p.wait_ns > kDrainNs ? p.wait_ns : kDrainNs);
      for (int r = 0; r < fp.R; ++r) list_pieces(fp, plan_ts, plan_ts[p.B], ls, r);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1 && attn) {
    tc_fence_after();
    tmem_dealloc(cx.tmem, kTmemCols);
  }
  const unsigned long long tok = tok_sh;
  // barrier 2: every partial written.  Right after the arrival the lift
  // unit's W_UV block starts loading into the free key-tile space (issued
  // after the release, which would otherwise wait for the copy too).
  if (warp == kSyncWarp) {
    if (lane == 0) {
      st_release_u64(fp.arr2 + blockIdx.x, tok);
      if (lift) {
        mbar_arrive_expect_tx(&wbar, kLiftWBytes);
        bulk_g2s(smem + kQBytes, lift_w(fp, blockIdx.x), kLiftWBytes, &wbar);
      }
    }
    grid_wait(fp.arr2, gridDim.x, tok, p.wait_ns, p.flags);
    if (blockIdx.x == 0) {
      // Every CTA read the epoch before its barrier-1 arrival: once all have
      // arrived, the next call may see the new epoch.
      const bool all = grid_wait(fp.arr1, gridDim.x, tok, p.wait_ns > kDrainNs ? p.wait_ns : kDrainNs, p.flags);
      if (lane == 0 && all) *reinterpret_cast<volatile unsigned long long*>(fp.epoch) = tok;
    }
  }
  __syncthreads();

  // phase C (the query block and key tile are free now)
  if (lift) {
    lift_unit(fp, blockIdx.x, smem + kQBytes, ls, smem, &wbar);
    if (threadIdx.x == 0) {  // never exit with the W_UV copy in flight
      volatile int no_abort = 0;
      mbar_wait(&wbar, 0, &no_abort, p.flags, p.wait_ns > kDrainNs ? p.wait_ns : kDrainNs);
    }
  }
  // rows whose lengths are out of range: flag them (their outputs are NaN)
  if (blockIdx.x == 0 && threadIdx.x < p.B) {
    const int Tb = p.T[threadIdx.x];
    if (Tb < S || Tb > p.T_cap) raise_flag(p.flags, MLA_DEV_BAD_LENGTH);
  }
}

std::atomic<unsigned long long> g_fused_attr[4] = {};

size_t align256f(size_t x) { return (x + 255) & ~(size_t)255; }

struct FusedPlan {
  int grid, G, qsplit, attn_ctas, P;
  size_t off_q, off_o, off_ml, off_sync, total;
};

int fused_grid() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

bool make_fused_plan(int B, int S, int T_cap, int Dv, FusedPlan* pl) {
  const int R = B * S;
  if (R < 1 || R > kFusedRows) return false;
  const int grid = fused_grid();
  if (grid < kLiftUnits || grid > kMaxGrid || grid * kMaxAbsPerCta < kAbsUnits) return false;
  pl->grid = grid;
  const long long tiles = (long long)B * ((T_cap + kTile - 1) / kTile);
  long long G = grid / S;
  if (G > tiles) G = tiles;
  if (G < 1) G = 1;
  pl->G = (int)G;
  const int pieces = pl->G * S;
  pl->qsplit = pieces * 4 <= grid ? 4 : pieces * 2 <= grid ? 2 : 1;
  pl->attn_ctas = pieces * pl->qsplit;
  pl->P = (pl->G + B - 1) * S;
  size_t off = 0;
  pl->off_q = off;
  off = align256f(off + (size_t)R * kH * kDc * 2);
  pl->off_o = off;
  off = align256f(off + (size_t)pl->P * kH * kDl * 4);
  pl->off_ml = off;
  off = align256f(off + (size_t)pl->P * kH * 2 * 4);
  pl->off_sync = off;
  off = align256f(off + 8 + (size_t)2 * grid * 8);
  pl->total = off;
  return true;
}

}  // namespace

bool fused_decode_ok(const DecodeArgs& a, bool sparse) {
  FusedPlan pl;
  return !sparse && !a.lat_fp8 && a.pages.table == nullptr && a.g.Dv == 256 &&
         make_fused_plan(a.B, a.S, a.T_cap, a.g.Dv, &pl);
}

size_t fused_decode_workspace_bytes(const Geometry& g, int B, int S, int T_cap) {
  FusedPlan pl;
  if (g.Dv != 256 || !make_fused_plan(B, S, T_cap, g.Dv, &pl)) return 0;
  return pl.total;
}

cudaError_t launch_decode_fused(const DecodeArgs& a, void* ws, cudaStream_t st) {
  const Geometry& g = a.g;
  FusedPlan pl;
  if (!make_fused_plan(a.B, a.S, a.T_cap, g.Dv, &pl)) return cudaErrorInvalidValue;
  if ((long long)a.B * a.T_cap >= (1ll << 31)) return cudaErrorInvalidValue;
  unsigned char* w = static_cast<unsigned char*>(ws);
  FusedParams fp{};
  AttnParams& tp = fp.at;
  __nv_bfloat16* qcat = reinterpret_cast<__nv_bfloat16*>(w + pl.off_q);
  bool maps_ok = make_tmap_2d_bf16(&tp.mQ, qcat, (uint64_t)a.B * a.S * kH, kDc, kDc, kH, 64) &&
                 make_tmap_2d_bf16(&tp.mL, a.Lc, (uint64_t)a.B * a.T_cap, kDl, kDl, kTile, 64) &&
                 make_tmap_2d_bf16(&tp.mR, a.Rc, (uint64_t)a.B * a.T_cap, kDr, kDr, kTile, 64);
  if (!maps_ok) return cudaErrorInvalidValue;
  tp.T = a.T;
  tp.B = a.B;
  tp.S = a.S;
  tp.T_cap = a.T_cap;
  tp.G = pl.G;
  tp.topk = 0;
  tp.kv_rows = a.T_cap;
  tp.qsplit = pl.qsplit;
  tp.read_once = (a.S == 1 && pl.qsplit == 1) ? 1 : 0;
  tp.c = g.scale * kLog2e;
  tp.lat_scale = 1.f;
  tp.o_part = reinterpret_cast<float*>(w + pl.off_o);
  tp.ml_part = reinterpret_cast<float*>(w + pl.off_ml);
  tp.flags = a.flags;
  tp.wait_ns = a.wait_limit_ns;
  fp.q = static_cast<const __nv_bfloat16*>(a.q);
  fp.kv_b = static_cast<const __nv_bfloat16*>(a.kv_b);
  fp.qcat = qcat;
  fp.out = a.out;
  unsigned long long* sync = reinterpret_cast<unsigned long long*>(w + pl.off_sync);
  fp.epoch = sync;
  fp.arr1 = sync + 1;
  fp.arr2 = sync + 1 + pl.grid;
  fp.Dn = g.Dn;
  fp.Dv = g.Dv;
  fp.R = a.B * a.S;
  fp.attn_ctas = pl.attn_ctas;
  for (int j = 0; j < kDr / 2; ++j) fp.turn[j] = rope_turns(std::pow(g.rope_base, -2.0 * j / kDr));

  using Kern = void (*)(const FusedParams);
  static const Kern kerns[4] = {fused_decode_kernel<2>, fused_decode_kernel<4>, fused_decode_kernel<6>,
                                fused_decode_kernel<8>};
  const int ki = g.Dn / 64 - 1;
  const Kern kern = kerns[ki];
  {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(g_fused_attr[ki].load() & bit)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFusedDynSmem);
      if (e != cudaSuccess) return e;
      g_fused_attr[ki].fetch_or(bit);
    }
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = kFusedDynSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident at once, or no launch
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  kernel_mark(st, "fused_decode");
  return cudaLaunchKernelEx(&cfg, kern, fp);
}

}  // namespace mla
