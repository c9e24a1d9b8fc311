// gemm_tc.cu -- batched bf16 GEMM on tcgen05 tensor cores (see gemm_tc.h).
//
// Persistent: one CTA per SM walks the 128 x BN tiles of C (n fastest).  Warp
// 0 streams 64-wide K slabs of A (3D TMA, 128-byte swizzle) and B through a
// ring of stages that runs on across tiles, warp 1 issues tcgen05.mma
// (M=128, N=BN, K=16) into one of two TMEM accumulators, and warps 2-5 (one
// output row per thread) read the other accumulator back and store C, so the
// epilogue of a tile overlaps the products of the next.
#include <atomic>

#include "common.cuh"
#include "gemm_tc.h"
#include "sm100.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace sm100;

constexpr int kGThreads = 192;
constexpr int kGBM = 128;
constexpr long long kGDrainNs = 1000000000LL;

template <int BN>
struct GemmCfg {
  static constexpr uint32_t kA = kGBM * 128;  // 128 rows x 64 bf16
  static constexpr uint32_t kB = BN * 128;    // BN x 64 bf16 (either major)
  static constexpr uint32_t kStage = kA + kB;
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr uint32_t kSmem = kStages * kStage + 1024;
};

struct GemmParams {
  CUtensorMap mA;  // 3D {k, z, m}, box {64, 1, 128}
  CUtensorMap mB;  // 2D; K-major box {64, BN}; MN-major box {64, 64}
  long long b_row0, b_rows_per_z, b_col0;
  void* c_base;
  long long c_ld_m, c_ld_z;
  int out_kind;
  const float* scale;
  int M, N, K, Z;
  unsigned int* flags;
  long long wait_ns;
};

template <int BN, bool kBMN>
__global__ void __launch_bounds__(kGThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  using Cfg = GemmCfg<BN>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  // The ring of K slabs runs on across the CTA's tiles; the accumulator is
  // double-buffered in TMEM, so that the epilogue of one tile overlaps the
  // products of the next.  acc_full/acc_empty[b] complete once per tile that
  // uses buffer b.
  __shared__ uint64_t full_bar[Cfg::kStages], empty_bar[Cfg::kStages], acc_full[2], acc_empty[2], mma_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = p.K / 64;
  const int tn = (p.N + BN - 1) / BN, tm = (p.M + kGBM - 1) / kGBM;
  const int ntiles = tn * tm * p.Z;
  // tile t -> (z, m tile, n tile), n fastest
  auto tile_of = [&](int t, int* n0, int* m0, int* z) {
    *n0 = (t % tn) * BN;
    *m0 = ((t / tn) % tm) * kGBM;
    *z = t / (tn * tm);
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 128);
    }
    mbar_init(&mma_done, 1);
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&p.mA);
    prefetch_tensormap(&p.mB);
  }
  // B is a weight no kernel of this library writes: the B halves of the first
  // ring stages load before the dependency wait that A needs (thread 0 is the
  // producer lane; each stage expects its A and B bytes together).
  int npre = 0;
  if (threadIdx.x == 0) {
    for (int t = blockIdx.x; t < ntiles && npre < Cfg::kStages; t += gridDim.x) {
      int n0, m0, z;
      tile_of(t, &n0, &m0, &z);
      const int brow = (int)(p.b_row0 + (long long)z * p.b_rows_per_z);
      for (int kb = 0; kb < nk && npre < Cfg::kStages; ++kb, ++npre) {
        unsigned char* sB = smem + npre * Cfg::kStage + Cfg::kA;
        mbar_arrive_expect_tx(&full_bar[npre], Cfg::kStage);
        if (!kBMN) {
          tma_load_2d(sB, &p.mB, (int)p.b_col0 + kb * 64, brow + n0, &full_bar[npre]);
        } else {
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)
            tma_load_2d(sB + j * 8192, &p.mB, (int)p.b_col0 + n0 + 64 * j, brow + kb * 64, &full_bar[npre]);
        }
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  volatile int* abort = &abort_flag;
  grid_dep_wait();  // A (and the epilogue's scale) may come from the previous kernel
  grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) {
      int g = 0, last = -1;  // slab counter over all tiles of this CTA
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        int n0, m0, z;
        tile_of(t, &n0, &m0, &z);
        const int brow = (int)(p.b_row0 + (long long)z * p.b_rows_per_z);
        for (int kb = 0; kb < nk && ok; ++kb, ++g) {
          const int st = g % Cfg::kStages, u = g / Cfg::kStages;
          unsigned char* sA = smem + st * Cfg::kStage;
          unsigned char* sB = sA + Cfg::kA;
          if (g < npre) {  // B already on its way: the stage's A half
            tma_load_3d(sA, &p.mA, kb * 64, z, m0, &full_bar[st]);
            last = g;
            continue;
          }
          ok = mbar_wait(&empty_bar[st], (u & 1) ^ 1, abort, p.flags, p.wait_ns);
          if (!ok) break;
          mbar_arrive_expect_tx(&full_bar[st], Cfg::kStage);
          tma_load_3d(sA, &p.mA, kb * 64, z, m0, &full_bar[st]);
          if (!kBMN) {
            tma_load_2d(sB, &p.mB, (int)p.b_col0 + kb * 64, brow + n0, &full_bar[st]);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(sB + j * 8192, &p.mB, (int)p.b_col0 + n0 + 64 * j, brow + kb * 64, &full_bar[st]);
          }
          last = g;
        }
      }
      if (last >= 0) {  // never leave with copies in flight
        volatile int no_abort = 0;
        const long long dn = p.wait_ns > kGDrainNs ? p.wait_ns : kGDrainNs;
        for (int q = last - Cfg::kStages + 1; q <= last; ++q)
          if (q >= 0) mbar_wait(&full_bar[q % Cfg::kStages], (q / Cfg::kStages) & 1, &no_abort, p.flags, dn);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kGBM, BN, 0, kBMN ? 1 : 0);
      bool ok = true, issued = false;
      int g = 0, i = 0;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++i) {
        const int buf = i & 1;
        ok = mbar_wait(&acc_empty[buf], ((i >> 1) & 1) ^ 1, abort, p.flags, p.wait_ns);
        if (!ok) break;
        tc_fence_after();
        const uint32_t acc = tmem + BN * buf;
        for (int kb = 0; kb < nk && ok; ++kb, ++g) {
          const int st = g % Cfg::kStages, u = g / Cfg::kStages;
          ok = mbar_wait(&full_bar[st], u & 1, abort, p.flags, p.wait_ns);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + st * Cfg::kStage), b0 = a0 + Cfg::kA;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t da = smem_desc_sw128(a0 + kk * 32, 16, 1024);
            const uint64_t db = kBMN ? smem_desc_sw128(b0 + kk * 2048, 8192, 1024) : smem_desc_sw128(b0 + kk * 32, 16, 1024);
            mma_bf16(acc, da, db, idesc, (kb | kk) != 0);
          }
          mma_commit(&empty_bar[st]);
          issued = true;
        }
        if (ok) mma_commit(&acc_full[buf]);
      }
      if (issued) {  // every product retired before TMEM is released
        mma_commit(&mma_done);
        volatile int no_abort = 0;
        mbar_wait(&mma_done, 0, &no_abort, p.flags, p.wait_ns > kGDrainNs ? p.wait_ns : kGDrainNs);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;
    const uint32_t t_lane = (uint32_t)(32 * wq) << 16;
    int i = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
      const int buf = i & 1;
      int n0, m0, z;
      tile_of(t, &n0, &m0, &z);
      const int m = m0 + 32 * wq + lane;
      // a failed wait is decided jointly by the 128 epilogue threads
      const bool fail = !mbar_wait(&acc_full[buf], (i >> 1) & 1, abort, p.flags, p.wait_ns);
      if (bar_red_or(1, 128, fail)) break;
      tc_fence_after();
      float scale = 1.f;
      if (p.out_kind == kGemmOutF32Scaled && m < p.M) scale = p.scale[(size_t)m * p.Z + z];
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 64) {
        float v[64];
        tmem_ld64(tmem + t_lane + BN * buf + c0, v);
        tmem_wait_ld();
        const int n = n0 + c0;
        if (m < p.M && n < p.N) {
          if (p.out_kind == kGemmOutBf16) {
            __nv_bfloat16* c = static_cast<__nv_bfloat16*>(p.c_base) + (size_t)m * p.c_ld_m + (size_t)z * p.c_ld_z + n;
#pragma unroll
            for (int j = 0; j < 64; j += 8) {
              uint4 q;
              q.x = pack2(v[j], v[j + 1]);
              q.y = pack2(v[j + 2], v[j + 3]);
              q.z = pack2(v[j + 4], v[j + 5]);
              q.w = pack2(v[j + 6], v[j + 7]);
              *reinterpret_cast<uint4*>(c + j) = q;
            }
          } else {
            float* c = static_cast<float*>(p.c_base) + (size_t)m * p.c_ld_m + (size_t)z * p.c_ld_z + n;
#pragma unroll
            for (int j = 0; j < 64; j += 4)
              *reinterpret_cast<float4*>(c + j) = make_float4(v[j] * scale, v[j + 1] * scale, v[j + 2] * scale, v[j + 3] * scale);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * BN);
  }
}

template <int BN, bool kBMN>
cudaError_t launch_one(const GemmParams& gp, bool pdl, cudaStream_t st) {
  using Cfg = GemmCfg<BN>;
  static std::atomic<unsigned long long> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(done.load() & bit)) {
    e = cudaFuncSetAttribute(gemm_kernel<BN, kBMN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit);
  }
  cudaLaunchConfig_t cfg{};
  const long long tiles = (long long)((gp.N + BN - 1) / BN) * ((gp.M + kGBM - 1) / kGBM) * gp.Z;
  int sms = 148;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cfg.gridDim = dim3((unsigned)(tiles < sms ? tiles : sms));  // persistent: one CTA per SM walks the tiles
  cfg.blockDim = dim3(kGThreads);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<BN, kBMN>, gp);
}

}  // namespace

cudaError_t launch_gemm_tc(const GemmArgs& a, bool pdl, cudaStream_t st) {
  if (a.K % 64 != 0 || a.N % 64 != 0 || a.M < 1 || a.Z < 1) return cudaErrorInvalidValue;
  // BN = 256 when the N extent allows and the grid stays wide, else 128.
  const int BN = (a.N % 256 == 0 && (long long)(a.N / 256) * ((a.M + 127) / 128) * a.Z >= 148) ? 256 : 128;
  GemmParams gp{};
  const uint64_t adims[3] = {(uint64_t)a.K, (uint64_t)a.Z, (uint64_t)a.M};
  const uint64_t astr[2] = {(uint64_t)a.a_ld_z * 2, (uint64_t)a.a_ld_m * 2};
  const uint32_t abox[3] = {64, 1, (uint32_t)kGBM};
  if (!make_tmap_3d_bf16(&gp.mA, a.a_base, adims, astr, abox)) return cudaErrorInvalidValue;
  const uint32_t brows = a.b_mn_major ? 64u : (uint32_t)BN;
  if (!make_tmap_2d_bf16(&gp.mB, a.b_base, (uint64_t)a.b_rows, (uint64_t)a.b_cols, (uint64_t)a.b_ld, brows, 64))
    return cudaErrorInvalidValue;
  gp.b_row0 = a.b_row0;
  gp.b_rows_per_z = a.b_rows_per_z;
  gp.b_col0 = a.b_col0;
  gp.c_base = a.c_base;
  gp.c_ld_m = a.c_ld_m;
  gp.c_ld_z = a.c_ld_z;
  gp.out_kind = a.out_kind;
  gp.scale = a.scale;
  gp.M = a.M;
  gp.N = a.N;
  gp.K = a.K;
  gp.Z = a.Z;
  gp.flags = a.flags;
  gp.wait_ns = a.wait_ns;
  if (BN == 256) return a.b_mn_major ? launch_one<256, true>(gp, pdl, st) : launch_one<256, false>(gp, pdl, st);
  return a.b_mn_major ? launch_one<128, true>(gp, pdl, st) : launch_one<128, false>(gp, pdl, st);
}

}  // namespace mla
