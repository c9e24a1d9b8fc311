// oproj.cu -- the output projection that ends both attention paths.
//
// The page "MLA 注意力与 KV 缓存", §2.3: the absorbed and the non-absorbed
// path both finish with the o output projection of the per-head outputs,
// y[r, :] = W_O vec(out[r, :, :]).  Its weight is the largest tensor of the
// layer's attention (hidden x 64*256 values), so the projection is a stream
// of W_O from HBM:
//   * up to kOprojGemvRows rows: a GEMV, one warp per output row n, 16-byte
//     loads of W_O[n, :] (read once, marked evict-first in L2) against the
//     rows of x held in L1; fp32 accumulation, a warp butterfly at the end;
//   * more rows with bf16 weights: x rounded to bf16, then the batched
//     tcgen05 GEMM (W_O read once per 128 rows of x).
// Launched as a programmatic dependent, the GEMV issues its first W_O loads
// before it waits for the kernel that writes x.
#include "common.cuh"
#include "gemm_tc.h"
#include "internal.h"

namespace mla {
namespace {

constexpr int kOpThreads = 256;
constexpr int kOpWarps = kOpThreads / 32;

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 8 consecutive weights of a 16-byte chunk as fp32 (bf16: 8 values; fp32: 4 values, kVals = 4).
template <typename Tw>
struct WChunk;
template <>
struct WChunk<__nv_bfloat16> {
  static constexpr int kVals = 8;
  __device__ static void unpack(const uint4& v, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
};
template <>
struct WChunk<float> {
  static constexpr int kVals = 4;
  __device__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};

// CTA = kOpRows output rows; warp w takes a 1/kOpWarps slice of the in_dim
// axis for all of them, so that each x value loaded serves kOpRows rows of
// W_O; the warps' partial sums meet in shared memory.  R (<= 8) rows of x.
constexpr int kOpRows = 8;

template <typename Tw, int R>
__global__ void __launch_bounds__(kOpThreads) oproj_gemv_kernel(OprojArgs a) {
  constexpr int V = WChunk<Tw>::kVals;  // weights per 16-byte chunk
  constexpr int kStep = 32 * V;         // weights per warp step and row
  __shared__ float part[kOpWarps][kOpRows][R];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n0 = blockIdx.x * kOpRows;
  const int nrows = min(kOpRows, a.hidden - n0);
  // this warp's slice of the in_dim axis, in whole steps
  const int steps = (a.in_dim + kStep - 1) / kStep;
  const int s0 = (int)((long long)steps * warp / kOpWarps), s1 = (int)((long long)steps * (warp + 1) / kOpWarps);
  const Tw* W = static_cast<const Tw*>(a.w_o) + (size_t)n0 * a.in_dim;
  float acc[kOpRows][R];
#pragma unroll
  for (int i = 0; i < kOpRows; ++i)
#pragma unroll
    for (int r = 0; r < R; ++r) acc[i][r] = 0.f;
  uint4 cur[kOpRows], nxt[kOpRows];
  auto load = [&](uint4 (&dst)[kOpRows], int st) {
    const int k = st * kStep + lane * V;
#pragma unroll
    for (int i = 0; i < kOpRows; ++i)
      dst[i] = (i < nrows && k < a.in_dim) ? ld_stream(W + (size_t)i * a.in_dim + k) : make_uint4(0, 0, 0, 0);
  };
  if (s0 < s1) load(cur, s0);
  grid_dep_wait();  // x comes from the preceding kernel; the first weights are already on their way
  for (int st = s0; st < s1; ++st) {
    if (st + 1 < s1) load(nxt, st + 1);
    const int k = st * kStep + lane * V;
    if (k < a.in_dim) {
      float xv[R][V];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float4* xr = reinterpret_cast<const float4*>(a.x + (size_t)r * a.in_dim + k);
#pragma unroll
        for (int c = 0; c < V / 4; ++c) {
          const float4 t = __ldg(xr + c);
          xv[r][4 * c] = t.x;
          xv[r][4 * c + 1] = t.y;
          xv[r][4 * c + 2] = t.z;
          xv[r][4 * c + 3] = t.w;
        }
      }
#pragma unroll
      for (int i = 0; i < kOpRows; ++i) {
        float w[V];
        WChunk<Tw>::unpack(cur[i], w);
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int v = 0; v < V; ++v) acc[i][r] = fmaf(w[v], xv[r][v], acc[i][r]);
      }
    }
#pragma unroll
    for (int i = 0; i < kOpRows; ++i) cur[i] = nxt[i];
  }
#pragma unroll
  for (int i = 0; i < kOpRows; ++i)
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float v = warp_sum(acc[i][r]);
      if (lane == 0) part[warp][i][r] = v;
    }
  __syncthreads();
  for (int e = threadIdx.x; e < nrows * R; e += kOpThreads) {
    const int i = e / R, r = e % R;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kOpWarps; ++w) v += part[w][i][r];
    a.y[(size_t)r * a.hidden + n0 + i] = v;
  }
}

template <typename Tw>
cudaError_t launch_gemv(const OprojArgs& b, bool pdl, cudaStream_t st) {
  const dim3 grid((b.hidden + kOpRows - 1) / kOpRows), block(kOpThreads);
  switch (b.R) {
    case 1: return launch_pdl(oproj_gemv_kernel<Tw, 1>, grid, block, 0, st, b, pdl);
    case 2: return launch_pdl(oproj_gemv_kernel<Tw, 2>, grid, block, 0, st, b, pdl);
    case 3: return launch_pdl(oproj_gemv_kernel<Tw, 3>, grid, block, 0, st, b, pdl);
    case 4: return launch_pdl(oproj_gemv_kernel<Tw, 4>, grid, block, 0, st, b, pdl);
    case 5: return launch_pdl(oproj_gemv_kernel<Tw, 5>, grid, block, 0, st, b, pdl);
    case 6: return launch_pdl(oproj_gemv_kernel<Tw, 6>, grid, block, 0, st, b, pdl);
    case 7: return launch_pdl(oproj_gemv_kernel<Tw, 7>, grid, block, 0, st, b, pdl);
    default: return launch_pdl(oproj_gemv_kernel<Tw, 8>, grid, block, 0, st, b, pdl);
  }
}

// x (fp32) -> bf16 rows for the GEMM path (n even: in_dim is a multiple of 64 there).
struct XCast {
  const float* x;
  __nv_bfloat16* xb;
  long long n;
};
__global__ void __launch_bounds__(256) oproj_x_bf16_kernel(XCast c) {
  grid_dep_wait();
  for (long long i = (long long)blockIdx.x * 256 + threadIdx.x; i < c.n / 2; i += (long long)gridDim.x * 256) {
    const float2 v = reinterpret_cast<const float2*>(c.x)[i];
    reinterpret_cast<__nv_bfloat162*>(c.xb)[i] = __floats2bfloat162_rn(v.x, v.y);
  }
}

// The GEMM takes K and N in multiples of 64.
bool use_gemm(int R, int in_dim, int hidden, int dtype) {
  return R > kOprojGemvRows && dtype == MLA_BF16 && in_dim % 64 == 0 && hidden % 64 == 0;
}

}  // namespace

size_t oproj_workspace_bytes(int R, int in_dim, int hidden, int dtype) {
  return use_gemm(R, in_dim, hidden, dtype) ? (size_t)R * in_dim * 2 : 0;
}

cudaError_t launch_oproj(const OprojArgs& a, bool pdl, unsigned int* flags, long long wait_ns, cudaStream_t st) {
  if (use_gemm(a.R, a.in_dim, a.hidden, a.dtype)) {
    kernel_mark(st, "oproj_x_bf16");
    const long long n = (long long)a.R * a.in_dim;
    const long long blocks = (n / 2 + 255) / 256 < 1024 ? (n / 2 + 255) / 256 : 1024;
    const XCast c{a.x, static_cast<__nv_bfloat16*>(a.x_bf16), n};
    cudaError_t e = launch_pdl(oproj_x_bf16_kernel, dim3((unsigned)blocks), dim3(256), 0, st, c, pdl);
    if (e != cudaSuccess) return e;
    GemmArgs g{};
    g.a_base = a.x_bf16;
    g.a_ld_m = a.in_dim;
    g.a_ld_z = 0;
    g.b_base = a.w_o;
    g.b_rows = a.hidden;
    g.b_cols = a.in_dim;
    g.b_ld = a.in_dim;
    g.b_mn_major = 0;
    g.b_row0 = 0;
    g.b_rows_per_z = 0;
    g.b_col0 = 0;
    g.c_base = a.y;
    g.c_ld_m = a.hidden;
    g.c_ld_z = 0;
    g.out_kind = kGemmOutF32;
    g.M = a.R;
    g.N = a.hidden;
    g.K = a.in_dim;
    g.Z = 1;
    g.flags = flags;
    g.wait_ns = wait_ns;
    kernel_mark(st, "oproj_gemm");
    return launch_gemm_tc(g, true, st);
  }
  kernel_mark(st, "oproj_gemv");
  cudaError_t e = cudaSuccess;
  for (int r0 = 0; r0 < a.R && e == cudaSuccess; r0 += kOprojGemvRows) {
    OprojArgs b = a;
    b.R = a.R - r0 < kOprojGemvRows ? a.R - r0 : kOprojGemvRows;
    b.x = a.x + (size_t)r0 * a.in_dim;
    b.y = a.y + (size_t)r0 * a.hidden;
    e = a.dtype == MLA_BF16 ? launch_gemv<__nv_bfloat16>(b, pdl, st) : launch_gemv<float>(b, pdl, st);
    pdl = false;
  }
  return e;
}

}  // namespace mla
