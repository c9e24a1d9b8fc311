// prefill_tc.h -- tensor-core non-absorbed prefill (kv_b GEMM + causal flash attention).
#pragma once

#include <cuda_runtime.h>

#include "internal.h"

namespace mla {

// True for the GLM-5.2 head geometry the tensor-core prefill is built for
// (64 heads, qk_nope 192, qk_rope 64, v_head 256, kv_lora a multiple of 64).
bool tc_prefill_geometry_ok(const Geometry& g);

// Enqueues the kv_b GEMM (rebuilt KV into a.kv, bf16) and the attention.
cudaError_t launch_prefill_tc(const PrefillArgs& a, unsigned int* flags, long long wait_ns, cudaStream_t st);

}  // namespace mla
