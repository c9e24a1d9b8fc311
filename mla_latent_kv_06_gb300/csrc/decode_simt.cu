// decode_simt.cu -- CUDA-core weight-absorbed decode (dense and DSA-sparse).
//
// Follows the absorbed path of the page "MLA 注意力与 KV 缓存", §2.3: the
// key part of kv_b is folded into the query (qabs), scores are taken straight
// on the latent cache plus the shared rotated key, the softmax-weighted latent
// context clat is formed, and the value part of kv_b lifts clat per head.
//
// One CTA computes one (b, s, h) row in fp32 with an online softmax over
// chunks of 64 keys.  This is the general-shape path: any head geometry, fp32
// or bf16 inputs.  The GLM-shaped bf16 case runs on the tensor-core kernels.
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 64;

template <typename Tin, bool kSparse>
__global__ void __launch_bounds__(kThreads) decode_simt_kernel(DecodeArgs a) {
  const Geometry g = a.g;
  const int h = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Dq = g.Dn + g.Dr;
  const int Dkv = g.Dn + g.Dv;
  float* out = a.out + (((size_t)b * a.S + s) * g.H + h) * g.Dv;

  extern __shared__ float smem[];
  float* qn = smem;               // [Dn]
  float* qr = qn + g.Dn;          // [Dr] rotated rope part
  float* qabs = qr + g.Dr;        // [Dl]
  float* clat = qabs + g.Dl;      // [Dl]
  float* sc = clat + g.Dl;        // [kChunk] scores, then probabilities
  int* tok = reinterpret_cast<int*>(sc + kChunk);  // [kChunk] cache row of each slot, -1 if masked

  const int Tb = a.T[b];
  const bool bad_len = (Tb < a.S || Tb > a.T_cap);
  const int pos = Tb - a.S + s;
  int n = pos + 1;
  bool bad_sel = false;
  if (!bad_len && kSparse) {
    n = a.nsel[(size_t)b * a.S + s];
    bad_sel = (n < 1 || n > a.topk);
  }
  if (bad_len || bad_sel) {
    if (tid == 0) raise_flag(a.flags, bad_len ? MLA_DEV_BAD_LENGTH : MLA_DEV_BAD_INDEX);
    for (int j = tid; j < g.Dv; j += kThreads) out[j] = qnan();
    return;
  }
  const int32_t* sel = kSparse ? a.sel + ((size_t)b * a.S + s) * a.topk : nullptr;

  const Tin* q = static_cast<const Tin*>(a.q) + (((size_t)b * a.S + s) * g.H + h) * Dq;
  const Tin* Lc = static_cast<const Tin*>(a.Lc);  // rows: cache_row() of (b, t)
  const Tin* Rc = static_cast<const Tin*>(a.Rc);
  const Tin* Wuk = static_cast<const Tin*>(a.kv_b) + (size_t)h * Dkv * g.Dl;
  const Tin* Wuv = Wuk + (size_t)g.Dn * g.Dl;

  for (int i = tid; i < g.Dn; i += kThreads) qn[i] = to_f32(q[i]);
  const int half = g.Dr / 2;
  for (int j = tid; j < half; j += kThreads) {
    float c, sn;
    rope_cos_sin(pos, j, g.Dr, g.rope_base, &c, &sn);
    float x0 = to_f32(q[g.Dn + 2 * j]), x1 = to_f32(q[g.Dn + 2 * j + 1]);
    qr[j] = x0 * c - x1 * sn;
    qr[half + j] = x1 * c + x0 * sn;
  }
  __syncthreads();
  // qabs[l] = sum_i qn[i] * W_UK[i][l]
  for (int l = tid; l < g.Dl; l += kThreads) {
    float acc = 0.f;
    for (int i = 0; i < g.Dn; ++i) acc = fmaf(qn[i], to_f32(Wuk[(size_t)i * g.Dl + l]), acc);
    qabs[l] = acc;
    clat[l] = 0.f;
  }
  __syncthreads();

  float m = -INFINITY, lsum = 0.f;
  int bad_index = 0;
  for (int c0 = 0; c0 < n; c0 += kChunk) {
    const int cn = min(kChunk, n - c0);
    for (int j = warp; j < cn; j += kWarps) {
      int t = kSparse ? sel[c0 + j] : c0 + j;
      bool ok = (t >= 0 && t <= pos);
      long long row = 0;
      if (ok) {
        bool bad_page = false;
        row = cache_row(a.pages, b, a.T_cap, t, &bad_page);
        ok = !bad_page;
      }
      float dot = 0.f;
      if (ok) {
        const Tin* lrow = Lc + (size_t)row * g.Dl;
        const Tin* rrow = Rc + (size_t)row * g.Dr;
        for (int l = lane; l < g.Dl; l += 32) dot = fmaf(qabs[l], to_f32(lrow[l]), dot);
        for (int r = lane; r < g.Dr; r += 32) dot = fmaf(qr[r], to_f32(rrow[r]), dot);
        dot = warp_sum(dot);
      }
      if (lane == 0) {
        sc[j] = ok ? dot * g.scale : -INFINITY;
        tok[j] = ok ? (int)row : -1;  // pool row (< 2^31, checked on the host)
      }
    }
    __syncthreads();
    float cm = -INFINITY;
    for (int j = 0; j < cn; ++j) cm = fmaxf(cm, sc[j]);
    const float m_new = fmaxf(m, cm);
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
    __syncthreads();
    for (int j = tid; j < cn; j += kThreads) sc[j] = (tok[j] >= 0) ? expf(sc[j] - m_new) : 0.f;
    __syncthreads();
    float psum = 0.f;
    for (int j = 0; j < cn; ++j) {
      psum += sc[j];
      bad_index |= (tok[j] < 0);
    }
    lsum = lsum * alpha + psum;
    for (int l = tid; l < g.Dl; l += kThreads) {
      float acc = clat[l] * alpha;
      for (int j = 0; j < cn; ++j)
        if (tok[j] >= 0) acc = fmaf(sc[j], to_f32(Lc[(size_t)tok[j] * g.Dl + l]), acc);
      clat[l] = acc;
    }
    m = m_new;
    __syncthreads();
  }
  if (bad_index) {
    if (tid == 0) raise_flag(a.flags, MLA_DEV_BAD_INDEX);
    for (int j = tid; j < g.Dv; j += kThreads) out[j] = qnan();
    return;
  }
  const float inv = 1.f / lsum;
  for (int l = tid; l < g.Dl; l += kThreads) clat[l] *= inv;
  __syncthreads();
  // out[j] = W_UV[j] . clat
  for (int j = warp; j < g.Dv; j += kWarps) {
    const Tin* wrow = Wuv + (size_t)j * g.Dl;
    float acc = 0.f;
    for (int l = lane; l < g.Dl; l += 32) acc = fmaf(to_f32(wrow[l]), clat[l], acc);
    acc = warp_sum(acc);
    if (lane == 0) out[j] = acc;
  }
}

template <typename Tin, bool kSparse>
cudaError_t launch(const DecodeArgs& a, cudaStream_t st) {
  const Geometry& g = a.g;
  size_t smem = sizeof(float) * (g.Dn + g.Dr + 2 * g.Dl + kChunk) + sizeof(int) * kChunk;
  auto kern = decode_simt_kernel<Tin, kSparse>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(g.H, a.S, a.B);
  kern<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs& a, int dtype, bool sparse, cudaStream_t st) {
  if (dtype == MLA_F32) return sparse ? launch<float, true>(a, st) : launch<float, false>(a, st);
  return sparse ? launch<__nv_bfloat16, true>(a, st) : launch<__nv_bfloat16, false>(a, st);
}

}  // namespace mla
