// internal.h -- launchers shared between the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

struct Geometry {
  int H, Dn, Dr, Dl, Dv;  // heads, qk_nope, qk_rope, kv_lora, v_head
  float scale;            // resolved softmax scale
  double rope_base;       // resolved RoPE base
};

// Paged cache layout.  Token t of sequence b sits at row
// table[b * max_pages + t / page_size] * page_size + t % page_size of the page
// pool; table == nullptr means the contiguous layout (row b * T_cap + t).
struct PageTable {
  const int32_t* table;
  int max_pages, page_size, num_pages;
};

// Pool row of token t of sequence b.  A page index outside [0, num_pages)
// sets *bad and yields row 0, so that no access leaves the pool.
__host__ __device__ __forceinline__ long long cache_row(const PageTable& pt, int b, int T_cap, int t, bool* bad) {
  if (!pt.table) return (long long)b * T_cap + t;
  const int pg = pt.table[(size_t)b * pt.max_pages + t / pt.page_size];
  if (pg < 0 || pg >= pt.num_pages) {
    *bad = true;
    return 0;
  }
  return (long long)pg * pt.page_size + t % pt.page_size;
}

// Arguments common to the decode kernels (dense and sparse).
struct DecodeArgs {
  Geometry g;
  int B, S, T_cap;
  const void* q;
  const void* Lc;
  const void* Rc;
  const int32_t* T;
  const void* kv_b;
  float* out;
  const int32_t* sel;   // sparse only: [B,S,topk]
  const int32_t* nsel;  // sparse only: [B,S]
  int topk;
  unsigned int* flags;
  long long wait_limit_ns;
  PageTable pages;  // table == nullptr: contiguous [B, T_cap] caches
  int lat_fp8;      // Lc holds E4M3 codes (the FP8 cache); latent = lat_scale * code
  float lat_scale;
  // Sparse decode inside a multi-layer call: staging buffer 0 or 1, and
  // whether the gather may launch as a programmatic dependent of the
  // previous kernel (true only when that buffer was last read two layers back)
  int stage_parity;
  int gather_pdl;
};

cudaError_t launch_decode_simt(const DecodeArgs& a, int dtype, bool sparse, cudaStream_t st);

struct PrefillArgs {
  Geometry g;
  int B, S, pos_base;
  const void* q;
  const void* Lc;
  const void* Rc;
  const void* kv_b;
  void* kv;  // rebuilt [B, Tk, H, Dn+Dv], input dtype
  float* out;
};

cudaError_t launch_prefill_simt(const PrefillArgs& a, int dtype, cudaStream_t st);

struct IndexArgs {
  int B, S, n_ih, hd, T_cap;
  const float* q_idx;
  const float* w;
  const float* Ic;
  const int32_t* T;
  float* scores;
  unsigned int* flags;
  long long wait_ns;  // bound of every wait inside a kernel
  // Optional [B*S, parts, 2048] histograms of the top 11 bits of the ordered
  // score keys of the candidates t <= pos, one per indexer CTA of a row (the
  // first radix pass of the top-k); only the tensor-core indexer writes them.
  uint32_t* hpart;
};

cudaError_t launch_index_scores(const IndexArgs& a, cudaStream_t st);
// Tensor-core indexer (32 index heads x 128, fp32 through three tf32 products);
// returns cudaErrorNotSupported when the request does not fit it.
cudaError_t launch_index_scores_tc(const IndexArgs& a, cudaStream_t st);
// CTAs per (b, s) row of the tensor-core indexer, 0 when it does not take the shape.
int index_tc_parts(int B, int S, int n_ih, int hd, int T_cap);

struct TopkArgs {
  int B, S, T_cap, topk;
  const float* scores;
  const int32_t* T;
  int32_t* sel;
  int32_t* nsel;
  unsigned int* flags;
  const uint32_t* hpart;  // optional first-pass histograms from the indexer (IndexArgs::hpart)
  int hparts;
};

cudaError_t launch_topk_select(const TopkArgs& a, cudaStream_t st);

// Output projection y[r, n] = sum_k W_O[n, k] x[r, k] (W_O [hidden, in_dim] in dtype, x and y fp32).
struct OprojArgs {
  int R, in_dim, hidden, dtype;
  const void* w_o;
  const float* x;
  float* y;
  void* x_bf16;  // [R, in_dim] scratch for the tensor-core path (R > 8, bf16 weights), else unused
};
// Rows per GEMV launch; more rows take the tensor-core GEMM (bf16 weights).
constexpr int kOprojGemvRows = 8;
size_t oproj_workspace_bytes(int R, int in_dim, int hidden, int dtype);
cudaError_t launch_oproj(const OprojArgs& a, bool pdl, unsigned int* flags, long long wait_ns, cudaStream_t st);

// RoPE frequencies base^(-2j/d) travel in the launch parameters: rope widths up to 2 * kMaxRopePairs.
constexpr int kMaxRopePairs = 128;
// The append kernels hold a row in registers: at most kMaxAppendPer values per thread of 128.
constexpr int kMaxAppendPer = 32;
constexpr int kMaxAppendWidth = 128 * kMaxAppendPer;

struct AppendArgs {
  int B, S, T_cap, kv_lora, qk_rope;
  const void* comp;     // [B, S, kv_lora + qk_rope]
  const void* kv_a_ln;  // [kv_lora]
  float eps;
  const int32_t* T;
  void* Lc;  // [B, T_cap, kv_lora] or the page pool
  void* Rc;  // [B, T_cap, qk_rope] or the page pool
  unsigned int* flags;
  PageTable pages;
  uint64_t turn[kMaxRopePairs];  // rope_turns(rope_base^(-2j/qk_rope))
  int lat_fp8;          // Lc receives E4M3 codes of the normalised row * lat_inv_scale
  float lat_inv_scale;
};
cudaError_t launch_cache_append(const AppendArgs& a, int dtype, cudaStream_t st);

struct KeyAppendArgs {
  int B, S, T_cap, hd, rope_dim;
  const float* k;     // [B, S, hd]
  const float* ln_w;  // [hd]
  const float* ln_b;  // [hd] or null
  float eps;
  const int32_t* T;
  float* Ic;  // [B, T_cap, hd]
  unsigned int* flags;
  uint64_t turn[kMaxRopePairs];  // rope_turns(rope_base^(-2j/rope_dim))
};
cudaError_t launch_index_key_append(const KeyAppendArgs& a, cudaStream_t st);

// Sets the thread-local message returned by mla_last_error().
void set_last_error(const char* msg);

// Device address of the library's status word on the current device (null
// when it cannot be resolved), and the bound of every wait inside a kernel
// (mla_set_wait_limit_ns).
unsigned int* device_flags();
long long wait_limit_ns();

// Per-call launch bookkeeping behind mla_set_kernel_events / mla_last_launch_names:
// call_begin() at the start of each API call, kernel_mark() right before each
// kernel launch, call_end() after the last one.
void call_begin();
void kernel_mark(cudaStream_t st, const char* name);
void call_end(cudaStream_t st);

}  // namespace mla
