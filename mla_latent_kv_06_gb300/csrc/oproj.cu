// oproj.cu -- the output projection that ends both attention paths.
//
// The page "MLA 注意力与 KV 缓存", §2.3: the absorbed and the non-absorbed
// path both finish with the o output projection of the per-head outputs,
// y[r, :] = W_O vec(out[r, :, :]).  Its weight is the largest tensor of the
// layer's attention (hidden x 64*256 values), so the projection is a stream
// of W_O from HBM:
//   * one or two rows of bf16 weights, in_dim a multiple of 2048 up to 16384:
//     a ring of whole W_O rows per SM (bulk copies into six 32 KB stages, one
//     producer thread), eight consumer warps against x held in registers;
//   * otherwise up to kOprojGemvRows rows: a GEMV, one warp per output row n, 16-byte
//     loads of W_O[n, :] (read once, marked evict-first in L2) against the
//     rows of x held in L1; fp32 accumulation, a warp butterfly at the end;
//   * more rows with bf16 weights: x rounded to bf16, then the batched
//     tcgen05 GEMM (W_O read once per 128 rows of x).
// Launched as a programmatic dependent, the GEMV issues its first W_O loads
// before it waits for the kernel that writes x.
#include <atomic>

#include "common.cuh"
#include "gemm_tc.h"
#include "internal.h"
#include "sm100.cuh"

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
  grid_dep_launch();  // a dependent may start; whatever it reads of ours, it waits for this grid first
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

// ---------------------------------------------------------------- ring GEMV
// CTA c owns the output rows [c*hidden/G, (c+1)*hidden/G): one contiguous
// range of W_O.  Warp 8's lane 0 streams the rows through kRingStages
// shared-memory stages with bulk copies (contiguous 32 KB reads, the form
// that keeps HBM busiest); consumer thread t holds x[r, 8(t + 256j) + e] in
// registers and, per row, dots its 8*per weights with them, reduces over its
// warp and frees the stage.  The warps' sums meet in shared memory at the
// end.  W_O is an input no kernel of this library writes, so the ring fills
// before the dependency wait that x needs.
constexpr int kRingWarps = 8;
constexpr int kRingThreads = 32 * (kRingWarps + 1);
constexpr int kRingStages = 6;
constexpr int kRingRowMax = 16384;              // weights of one W_O row a stage holds
constexpr uint32_t kRingStageBytes = kRingRowMax * 2;
constexpr int kRingRowsMax = 256;               // output rows of one CTA
constexpr int kRingPer = kRingRowMax / 8 / (32 * kRingWarps);  // 16-byte chunks per thread and row, at most

struct RingArgs {
  OprojArgs a;
  unsigned int* flags;
  long long wait_ns;
};

template <int R>
constexpr size_t ring_smem_bytes() {
  return (size_t)kRingStages * kRingStageBytes + (size_t)kRingWarps * kRingRowsMax * R * sizeof(float);
}

template <int R>
__global__ void __launch_bounds__(kRingThreads, 1) oproj_ring_kernel(const RingArgs ra) {
  using namespace sm100;
  const OprojArgs& a = ra.a;
  extern __shared__ __align__(1024) unsigned char smem[];
  float* part = reinterpret_cast<float*>(smem + (size_t)kRingStages * kRingStageBytes);  // [warp][row][R]
  __shared__ uint64_t full[kRingStages], empty[kRingStages];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int r0 = (int)((long long)a.hidden * c / G), n = (int)((long long)a.hidden * (c + 1) / G) - r0;
  const uint32_t row_bytes = (uint32_t)a.in_dim * 2;
  volatile int* abort = &abort_flag;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRingStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kRingWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  grid_dep_launch();
  if (warp == kRingWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const unsigned char* W = static_cast<const unsigned char*>(a.w_o) + (size_t)r0 * row_bytes;
      int last[kRingStages];
      for (int st = 0; st < kRingStages; ++st) last[st] = -1;
      for (int i = 0; i < n; ++i) {
        const int st = i % kRingStages;
        if (!mbar_wait(&empty[st], ((i / kRingStages) & 1) ^ 1, abort, ra.flags, ra.wait_ns)) break;
        mbar_arrive_expect_tx(&full[st], row_bytes);
        bulk_copy_g2s(smem + (size_t)st * kRingStageBytes, W + (size_t)i * row_bytes, row_bytes, &full[st]);
        last[st] = i;
      }
      // never leave with copies in flight
      volatile int no_abort = 0;
      const long long drain_ns = ra.wait_ns > 1000000000LL ? ra.wait_ns : 1000000000LL;
      for (int st = 0; st < kRingStages; ++st)
        if (last[st] >= 0) mbar_wait(&full[st], (last[st] / kRingStages) & 1, &no_abort, ra.flags, drain_ns);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- consumers
    const int t = threadIdx.x, per = a.in_dim / (8 * 32 * kRingWarps);
    grid_dep_wait();  // x comes from the preceding kernel
    float xr[R][kRingPer * 8];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int j = 0; j < kRingPer; ++j) {
        if (j >= per) break;
        const float4* xp = reinterpret_cast<const float4*>(a.x + (size_t)r * a.in_dim + (size_t)(t + 256 * j) * 8);
        const float4 lo = __ldg(xp), hi = __ldg(xp + 1);
        xr[r][8 * j + 0] = lo.x;
        xr[r][8 * j + 1] = lo.y;
        xr[r][8 * j + 2] = lo.z;
        xr[r][8 * j + 3] = lo.w;
        xr[r][8 * j + 4] = hi.x;
        xr[r][8 * j + 5] = hi.y;
        xr[r][8 * j + 6] = hi.z;
        xr[r][8 * j + 7] = hi.w;
      }
    for (int i = 0; i < n; ++i) {
      const int st = i % kRingStages;
      int okl = 1;
      if (lane == 0) okl = mbar_wait(&full[st], (i / kRingStages) & 1, abort, ra.flags, ra.wait_ns) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, okl, 0)) break;
      const uint4* row = reinterpret_cast<const uint4*>(smem + (size_t)st * kRingStageBytes);
      float acc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) acc[r] = 0.f;
#pragma unroll
      for (int j = 0; j < kRingPer; ++j) {
        if (j >= per) break;
        float w[8];
        WChunk<__nv_bfloat16>::unpack(row[t + 256 * j], w);
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[r] = fmaf(w[e], xr[r][8 * j + e], acc[r]);
      }
      __syncwarp();  // every lane has read the stage
      if (lane == 0) mbar_arrive(&empty[st]);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float v = warp_sum(acc[r]);
        if (lane == 0) part[((size_t)warp * kRingRowsMax + i) * R + r] = v;
      }
    }
  }
  __syncthreads();
  if (*abort) return;  // a wait gave up (MLA_DEV_TIMEOUT is raised): leave y unwritten
  for (int e = threadIdx.x; e < n * R; e += kRingThreads) {
    const int i = e / R, r = e % R;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kRingWarps; ++w) v += part[((size_t)w * kRingRowsMax + i) * R + r];
    a.y[(size_t)r * a.hidden + r0 + i] = v;
  }
}

bool use_ring(const OprojArgs& a) {
  return a.dtype == MLA_BF16 && a.R >= 1 && a.R <= 2 && a.in_dim % (8 * 32 * kRingWarps) == 0 &&
         a.in_dim <= kRingRowMax;
}

template <int R>
cudaError_t launch_ring_r(const RingArgs& ra, bool pdl, cudaStream_t st) {
  static std::atomic<int> attr_set{0};
  const size_t smem = ring_smem_bytes<R>();
  if (!attr_set.load()) {
    cudaError_t e = cudaFuncSetAttribute(oproj_ring_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set.store(1);
  }
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  long long G = sms;
  const long long need = ((long long)ra.a.hidden + kRingRowsMax - 1) / kRingRowsMax;  // rows per CTA <= kRingRowsMax
  if (G < need) G = need;
  if (G > ra.a.hidden) G = ra.a.hidden;
  return launch_pdl(oproj_ring_kernel<R>, dim3((unsigned)G), dim3(kRingThreads), smem, st, ra, pdl);
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
  if (use_ring(a)) {
    const RingArgs ra{a, flags, wait_ns};
    return a.R == 1 ? launch_ring_r<1>(ra, pdl, st) : launch_ring_r<2>(ra, pdl, st);
  }
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
