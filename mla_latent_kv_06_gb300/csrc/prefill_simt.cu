// prefill_simt.cu -- CUDA-core non-absorbed prefill (general shapes).
//
// The non-absorbed path of the page "MLA 注意力与 KV 缓存", §2.3: one kv_b
// product rebuilds k_nope and the value of every key, then each new query
// attends causally with score = q_pass . k_nope + q_rot . k_rot (k_rot = Rc,
// shared by all heads), softmax, and a value sum.
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

// KV[r, c] = sum_l Lc[r, l] * kvb[c, l] for r < B*Tk, c < H*(Dn+Dv): a plain
// 64x64-tiled product with 4x4 outputs per thread.
constexpr int kBM = 64, kBN = 64, kBK = 16;

template <typename Tin>
__global__ void __launch_bounds__(256) kv_rebuild_kernel(const Tin* __restrict__ Lc,
                                                          const Tin* __restrict__ kvb,
                                                          Tin* __restrict__ kv, int M, int N, int K) {
  __shared__ float As[kBK][kBM + 4];
  __shared__ float Bs[kBK][kBN + 4];
  const int tid = threadIdx.x;
  const int tr = tid / 16, tc = tid % 16;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kBK) {
    for (int e = tid; e < kBM * kBK; e += 256) {
      int r = e / kBK, c = e % kBK;
      int gm = m0 + r, gk = k0 + c;
      As[c][r] = (gm < M && gk < K) ? to_f32(Lc[(size_t)gm * K + gk]) : 0.f;
      int gn = n0 + r;
      Bs[c][r] = (gn < N && gk < K) ? to_f32(kvb[(size_t)gn * K + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][tr * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tc * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 4; ++j) {
      int gm = m0 + tr * 4 + i, gn = n0 + tc * 4 + j;
      if (gm < M && gn < N) {
        if constexpr (sizeof(Tin) == 4)
          kv[(size_t)gm * N + gn] = acc[i][j];
        else
          kv[(size_t)gm * N + gn] = __float2bfloat16_rn(acc[i][j]);
      }
    }
}

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 64;

// One CTA per (h, s, b): online softmax over the keys t <= pos_base + s.
template <typename Tin>
__global__ void __launch_bounds__(kThreads) prefill_attn_kernel(PrefillArgs a) {
  const Geometry g = a.g;
  const int h = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Dq = g.Dn + g.Dr, Dkv = g.Dn + g.Dv;
  const int Tk = a.pos_base + a.S;
  const int pos = a.pos_base + s;
  extern __shared__ float smem[];
  float* qs = smem;            // [Dq]: q_pass then rotated q_rot
  float* acc = qs + Dq;        // [Dv]
  float* sc = acc + g.Dv;      // [kChunk]

  const Tin* q = static_cast<const Tin*>(a.q) + (((size_t)b * a.S + s) * g.H + h) * Dq;
  const Tin* kv = static_cast<const Tin*>(a.kv) + (size_t)b * Tk * g.H * Dkv + (size_t)h * Dkv;
  const Tin* Rc = static_cast<const Tin*>(a.Rc) + (size_t)b * Tk * g.Dr;
  const size_t kv_ld = (size_t)g.H * Dkv;

  for (int i = tid; i < g.Dn; i += kThreads) qs[i] = to_f32(q[i]);
  const int half = g.Dr / 2;
  for (int j = tid; j < half; j += kThreads) {
    float c, sn;
    rope_cos_sin(pos, j, g.Dr, g.rope_base, &c, &sn);
    float x0 = to_f32(q[g.Dn + 2 * j]), x1 = to_f32(q[g.Dn + 2 * j + 1]);
    qs[g.Dn + j] = x0 * c - x1 * sn;
    qs[g.Dn + half + j] = x1 * c + x0 * sn;
  }
  for (int j = tid; j < g.Dv; j += kThreads) acc[j] = 0.f;
  __syncthreads();
  const int n = pos + 1;
  float m = -INFINITY, lsum = 0.f;
  for (int c0 = 0; c0 < n; c0 += kChunk) {
    const int cn = min(kChunk, n - c0);
    for (int j = warp; j < cn; j += kWarps) {
      const int t = c0 + j;
      const Tin* kr = kv + (size_t)t * kv_ld;
      const Tin* rr = Rc + (size_t)t * g.Dr;
      float dot = 0.f;
      for (int i = lane; i < g.Dn; i += 32) dot = fmaf(qs[i], to_f32(kr[i]), dot);
      for (int r = lane; r < g.Dr; r += 32) dot = fmaf(qs[g.Dn + r], to_f32(rr[r]), dot);
      dot = warp_sum(dot);
      if (lane == 0) sc[j] = dot * g.scale;
    }
    __syncthreads();
    float cm = -INFINITY;
    for (int j = 0; j < cn; ++j) cm = fmaxf(cm, sc[j]);
    const float m_new = fmaxf(m, cm);
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
    __syncthreads();
    for (int j = tid; j < cn; j += kThreads) sc[j] = expf(sc[j] - m_new);
    __syncthreads();
    float psum = 0.f;
    for (int j = 0; j < cn; ++j) psum += sc[j];
    lsum = lsum * alpha + psum;
    for (int v = tid; v < g.Dv; v += kThreads) {
      float x = acc[v] * alpha;
      for (int j = 0; j < cn; ++j) x = fmaf(sc[j], to_f32(kv[(size_t)(c0 + j) * kv_ld + g.Dn + v]), x);
      acc[v] = x;
    }
    m = m_new;
    __syncthreads();
  }
  float* out = a.out + (((size_t)b * a.S + s) * g.H + h) * g.Dv;
  const float inv = 1.f / lsum;
  for (int v = tid; v < g.Dv; v += kThreads) out[v] = acc[v] * inv;
}

template <typename Tin>
cudaError_t launch(const PrefillArgs& a, cudaStream_t st) {
  const Geometry& g = a.g;
  const int Tk = a.pos_base + a.S;
  const int M = a.B * Tk, N = g.H * (g.Dn + g.Dv), K = g.Dl;
  dim3 grid1((N + kBN - 1) / kBN, (M + kBM - 1) / kBM);
  kv_rebuild_kernel<Tin><<<grid1, 256, 0, st>>>(static_cast<const Tin*>(a.Lc),
                                                static_cast<const Tin*>(a.kv_b),
                                                static_cast<Tin*>(a.kv), M, N, K);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  size_t smem = sizeof(float) * (g.Dn + g.Dr + g.Dv + kChunk);
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(prefill_attn_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid2(g.H, a.S, a.B);
  prefill_attn_kernel<Tin><<<grid2, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs& a, int dtype, cudaStream_t st) {
  return dtype == MLA_F32 ? launch<float>(a, st) : launch<__nv_bfloat16>(a, st);
}

}  // namespace mla
