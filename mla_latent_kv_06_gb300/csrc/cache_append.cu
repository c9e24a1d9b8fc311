// cache_append.cu -- writing the new tokens' rows of the caches.
//
// The page "MLA 注意力与 KV 缓存", §2.1 (KV path): the kv_a output of each
// new token splits into kv_lora values, which go through RMSNorm(kv_a_ln)
// into the latent cache Lc, and qk_rope values, which go through the RoPE
// shared by all heads into Rc.  §2.2: the indexer key goes through layernorm
// (eps 1e-6) and RoPE into Ic (fp32, page "第 7 章 · 03 token 精确前向验证与
// faithful DSA", §二).  The S new tokens of sequence b sit at rows
// pos = T[b] - S + s.  The FP8 cache stores the latent row as E4M3 codes of
// the normalised values divided by the cache's scale (round to nearest even,
// saturating at 448).  One CTA per new token.  A row is a few KB, so the
// kernels are bound by latency, not bandwidth: every thread issues all of
// its loads (the row's values, the norm weights, T[b]) before the first use,
// so that each row costs one DRAM round trip, then one block reduction
// (two for the LayerNorm) and the stores.  Both launch as programmatic
// dependents: the launch overlaps the preceding kernel, the loads wait for it.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kAppThreads = 128;

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < kAppThreads / 32; ++i) t += red[i];
  __syncthreads();
  return t;
}

__device__ __forceinline__ void store(float* p, float v) { *p = v; }
__device__ __forceinline__ void store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Pair j of a rope segment at position pos: (x0, x1) -> (y_j, y_{d/2+j}).
__device__ __forceinline__ void rope_pair(int pos, uint64_t turn, float x0, float x1, float* y0, float* y1) {
  float cs, sn;
  rope_cs_turns(pos, turn, &cs, &sn);
  *y0 = x0 * cs - x1 * sn;
  *y1 = x1 * cs + x0 * sn;
}

// Cache row of new token s of a sequence of length Tb, or -1 when Tb is out of range.
__device__ __forceinline__ int new_row(int Tb, int s, int S, int T_cap, unsigned int* flags) {
  if (Tb < S || Tb > T_cap) {
    if (s == 0 && threadIdx.x == 0) raise_flag(flags, MLA_DEV_BAD_LENGTH);
    return -1;
  }
  return Tb - S + s;
}

// kPer values of the latent part per thread (element tid + k * kAppThreads).
// kFp8: the latent row goes out as E4M3 codes.
template <typename Tv, int kPer, bool kFp8 = false>
__global__ void __launch_bounds__(kAppThreads) cache_append_kernel(AppendArgs a) {
  __shared__ float red[kAppThreads / 32];
  const int tid = threadIdx.x;
  const int b = blockIdx.x / a.S, s = blockIdx.x % a.S;
  const Tv* x = static_cast<const Tv*>(a.comp) + (size_t)blockIdx.x * (a.kv_lora + a.qk_rope);
  const Tv* w = static_cast<const Tv*>(a.kv_a_ln);
  const int half = a.qk_rope / 2;
  grid_dep_launch();
  grid_dep_wait();  // comp and the cache rows may belong to the preceding kernels
  // all loads first
  const int Tb = __ldg(a.T + b);
  float xv[kPer], wv[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int i = tid + k * kAppThreads;
    xv[k] = i < a.kv_lora ? to_f32(x[i]) : 0.f;
    wv[k] = i < a.kv_lora ? to_f32(w[i]) : 0.f;
  }
  float r0 = 0.f, r1 = 0.f;
  if (tid < half) {
    r0 = to_f32(x[a.kv_lora + 2 * tid]);
    r1 = to_f32(x[a.kv_lora + 2 * tid + 1]);
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kPer; ++k) ss = fmaf(xv[k], xv[k], ss);
  const float inv = rsqrtf(block_sum(ss, red) / (float)a.kv_lora + a.eps);
  const int pos = new_row(Tb, s, a.S, a.T_cap, a.flags);
  if (pos < 0) return;
  bool bad_page = false;
  const long long row = cache_row(a.pages, b, a.T_cap, pos, &bad_page);
  if (bad_page) {
    if (tid == 0) raise_flag(a.flags, MLA_DEV_BAD_INDEX);
    return;
  }
  if constexpr (kFp8) {
    unsigned char* lc = static_cast<unsigned char*>(a.Lc) + (size_t)row * a.kv_lora;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = tid + k * kAppThreads;
      if (i < a.kv_lora)
        lc[i] = (unsigned char)__nv_cvt_float_to_fp8(xv[k] * inv * wv[k] * a.lat_inv_scale, __NV_SATFINITE, __NV_E4M3);
    }
  } else {
    Tv* lc = static_cast<Tv*>(a.Lc) + (size_t)row * a.kv_lora;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = tid + k * kAppThreads;
      if (i < a.kv_lora) store(lc + i, xv[k] * inv * wv[k]);
    }
  }
  if (tid < half) {
    Tv* rc = static_cast<Tv*>(a.Rc) + (size_t)row * a.qk_rope;
    float y0, y1;
    rope_pair(pos, a.turn[tid], r0, r1, &y0, &y1);
    store(rc + tid, y0);
    store(rc + half + tid, y1);
  }
}

// kPer key values per thread (element tid + k * kAppThreads); the normalised
// row goes through shared memory because a rope pair spans two threads.
template <int kPer>
__global__ void __launch_bounds__(kAppThreads) key_append_kernel(KeyAppendArgs a) {
  __shared__ float red[kAppThreads / 32];
  extern __shared__ float row[];  // [hd] normalised key
  const int tid = threadIdx.x;
  const int b = blockIdx.x / a.S, s = blockIdx.x % a.S;
  const float* k = a.k + (size_t)blockIdx.x * a.hd;
  grid_dep_launch();
  grid_dep_wait();
  const int Tb = __ldg(a.T + b);
  float kv[kPer], wv[kPer], bv[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = tid + u * kAppThreads;
    kv[u] = i < a.hd ? k[i] : 0.f;
    wv[u] = i < a.hd ? a.ln_w[i] : 0.f;
    bv[u] = (i < a.hd && a.ln_b) ? a.ln_b[i] : 0.f;
  }
  float sum = 0.f;
#pragma unroll
  for (int u = 0; u < kPer; ++u) sum += kv[u];
  const float mean = block_sum(sum, red) / (float)a.hd;
  float sq = 0.f;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = tid + u * kAppThreads;
    const float d = i < a.hd ? kv[u] - mean : 0.f;
    sq = fmaf(d, d, sq);
  }
  const float inv = rsqrtf(block_sum(sq, red) / (float)a.hd + a.eps);
  const int pos = new_row(Tb, s, a.S, a.T_cap, a.flags);
  if (pos < 0) return;
  float* ic = a.Ic + ((size_t)b * a.T_cap + pos) * a.hd;
  const int r0 = a.hd - a.rope_dim, half = a.rope_dim / 2;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = tid + u * kAppThreads;
    if (i < a.hd) {
      const float y = (kv[u] - mean) * inv * wv[u] + bv[u];
      if (i < r0) ic[i] = y;
      else row[i - r0] = y;
    }
  }
  if (half == 0) return;
  __syncthreads();
  for (int j = tid; j < half; j += kAppThreads) {
    float y0, y1;
    rope_pair(pos, a.turn[j], row[2 * j], row[2 * j + 1], &y0, &y1);
    ic[r0 + j] = y0;
    ic[r0 + half + j] = y1;
  }
}

template <typename Tv>
cudaError_t launch_append_t(const AppendArgs& a, cudaStream_t st) {
  const dim3 grid(a.B * a.S), block(kAppThreads);
  if (a.lat_fp8) {
    if (a.kv_lora <= 4 * kAppThreads) return launch_pdl(cache_append_kernel<Tv, 4, true>, grid, block, 0, st, a);
    return launch_pdl(cache_append_kernel<Tv, kMaxAppendPer, true>, grid, block, 0, st, a);
  }
  if (a.kv_lora <= 4 * kAppThreads) return launch_pdl(cache_append_kernel<Tv, 4>, grid, block, 0, st, a);
  return launch_pdl(cache_append_kernel<Tv, kMaxAppendPer>, grid, block, 0, st, a);
}

}  // namespace

cudaError_t launch_cache_append(const AppendArgs& a, int dtype, cudaStream_t st) {
  if (a.lat_fp8 && dtype != MLA_BF16) return cudaErrorInvalidValue;  // the FP8 cache keeps Rc in bf16
  return dtype == MLA_BF16 ? launch_append_t<__nv_bfloat16>(a, st) : launch_append_t<float>(a, st);
}

cudaError_t launch_index_key_append(const KeyAppendArgs& a, cudaStream_t st) {
  const size_t smem = (size_t)a.rope_dim * sizeof(float);
  const dim3 grid(a.B * a.S), block(kAppThreads);
  if (a.hd <= 2 * kAppThreads) return launch_pdl(key_append_kernel<2>, grid, block, smem, st, a);
  return launch_pdl(key_append_kernel<kMaxAppendPer>, grid, block, smem, st, a);
}

}  // namespace mla
