// decode_tc.cu -- placeholder until the tensor-core decode lands.
#include "decode_tc.h"

namespace mla {

bool tc_decode_geometry_ok(const Geometry&) { return false; }
int tc_decode_launch_count(bool) { return 0; }
size_t tc_decode_workspace_bytes(const Geometry&, int, int, int, int) { return 0; }
cudaError_t launch_decode_tc(const DecodeArgs&, void*, size_t, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t launch_sparse_decode_tc(const DecodeArgs&, void*, size_t, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace mla
