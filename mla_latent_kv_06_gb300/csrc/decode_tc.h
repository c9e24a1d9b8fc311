// decode_tc.h -- tensor-core (tcgen05/TMEM/TMA) absorbed and sparse decode.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "internal.h"

namespace mla {

// True when the head geometry matches the tensor-core kernels (GLM-5.2 shape:
// 64 heads, 512-wide latent, 64-wide rope key, qk_nope and v_head multiples of 16).
bool tc_decode_geometry_ok(const Geometry& g);

// Workspace of the tensor-core path.  sparse_topk = 0 for dense decode (then
// T_cap bounds the keys per sequence), else the selection width.
size_t tc_decode_workspace_bytes(const Geometry& g, int B, int S, int T_cap, int sparse_topk);

// Kernels launched by one tensor-core decode call.
int tc_decode_launch_count(bool sparse, int B, int S);

cudaError_t launch_decode_tc(const DecodeArgs& a, void* ws, size_t ws_bytes, cudaStream_t st);

cudaError_t launch_sparse_decode_tc(const DecodeArgs& a, void* ws, size_t ws_bytes, cudaStream_t st);

}  // namespace mla
