// gemm_tc.h -- batched tcgen05 GEMM used by the weight products of the path:
//   C_z[m, n] = sum_k A_z[m, k] * B_z[n, k]     (bf16 inputs, fp32 accumulate)
// for z in [0, Z).  A rows are addressed through a 3D TMA map (k, z, m), so
// A_z may be a strided slice of a larger tensor (for example one head of a
// [rows, heads, width] query).  B_z is either K-major (B_z[n, k] contiguous
// in k) or MN-major (stored as [k][n], n contiguous), and starts at row
// `b_row0 + z * b_rows_per_z` of its 2D map.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

enum GemmOut {
  kGemmOutBf16 = 0,        // C (bf16)  = acc
  kGemmOutF32Scaled = 1,   // C (fp32)  = acc * scale[m * Z + z]
  kGemmOutF32 = 2          // C (fp32)  = acc
};

struct GemmArgs {
  // A: bf16 tensor with element (m, z, k) at a_base + m*a_ld_m + z*a_ld_z + k (elements)
  const void* a_base;
  long long a_ld_m, a_ld_z;
  // B: bf16 2D tensor of `b_rows` rows x `b_cols` columns (row pitch b_ld elements)
  const void* b_base;
  long long b_rows, b_cols, b_ld;
  int b_mn_major;      // 0: row n holds B_z[n, :] ; 1: row k holds B_z[:, n]
  long long b_row0, b_rows_per_z;
  long long b_col0;    // first column used (MN-major: column of n = 0)
  // C: element (m, z, n) at c_base + m*c_ld_m + z*c_ld_z + n
  void* c_base;
  long long c_ld_m, c_ld_z;
  int out_kind;        // GemmOut
  const float* scale;  // kGemmOutF32Scaled: [M * Z]
  int M, N, K, Z;      // K % 64 == 0, N % 64 == 0
  unsigned int* flags;
  long long wait_ns;
};

// Enqueues the GEMM (one CTA per 128 x BN output tile and batch entry).
// `pdl` launches it with programmatic stream serialization (the kernel waits
// for the previous grid before reading A).
cudaError_t launch_gemm_tc(const GemmArgs& a, bool pdl, cudaStream_t st);

}  // namespace mla
