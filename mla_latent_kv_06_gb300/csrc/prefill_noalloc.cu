// prefill_noalloc.cu -- mla_prefill_naive_noalloc: the non-absorbed prefill
// with its rebuilt-KV scratch held in a fixed device array of this library,
// for callers that cannot allocate device memory themselves.
//
// Who needs it: a caller whose device memory belongs to another component
// (for example a host framework whose pool owns the whole GPU and forbids
// third-party cudaMalloc), or a caller on a latency-critical path that cannot
// afford the device-wide synchronisation cudaMalloc/cudaFree may cause, or a
// plain C program that has no allocator of its own at hand.  Such a caller
// passes only inputs and outputs; the scratch lives in kScratchBytes of
// static device memory that every GPU loading this library holds until exit.
#include <mutex>
#include <string>

#include "common.cuh"
#include "internal.h"

#define MLA_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

// Largest rebuilt KV ([B, pos_base+S, H, qk_nope+v_head] in the input dtype)
// this entry point accepts.
constexpr size_t kScratchBytes = 32ull << 20;

// Shared by every call on a device.  In host code this name is only a
// host-side stand-in: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_prefill_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_scratch_ptr[kMaxDevices] = {};

int fail(int code, const std::string& msg) {
  mla::set_last_error(msg.c_str());  // read back through mla_last_error()
  return code;
}

// Device address of g_prefill_scratch on the current device, looked up once
// per device (first call on that device) with that device current.
cudaError_t scratch_ptr(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_prefill_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

MLA_EXPORT int mla_prefill_naive_noalloc(const mla_dims* d, int dtype, int B, int S, int pos_base,
                                         const void* q, const void* Lc, const void* Rc,
                                         const void* kv_b, float* out, void* stream) {
  if (!d || d->H < 1 || d->qk_nope < 0 || d->qk_rope < 0 || d->qk_rope % 2 != 0 || d->kv_lora < 1 ||
      d->v_head < 1 || d->qk_nope + d->qk_rope < 1)
    return fail(MLA_ERR_INVALID, "invalid mla_dims (null, non-positive size or odd qk_rope)");
  if (dtype != MLA_F32 && dtype != MLA_BF16) return fail(MLA_ERR_INVALID, "unknown dtype");
  if (B < 1 || S < 1 || pos_base < 0) return fail(MLA_ERR_INVALID, "B, S must be >= 1 and pos_base >= 0");
  if (!q || !Lc || !Rc || !kv_b || !out) return fail(MLA_ERR_INVALID, "null tensor pointer");
  const size_t el = dtype == MLA_F32 ? 4 : 2;
  const size_t need = (size_t)B * ((size_t)pos_base + S) * d->H * (d->qk_nope + d->v_head) * el;
  if (need > kScratchBytes)
    return fail(MLA_ERR_INVALID, "rebuilt KV needs " + std::to_string(need) + " bytes, more than the " +
                                     std::to_string(kScratchBytes) + "-byte static scratch of this entry point");
  unsigned char* scratch = nullptr;
  cudaError_t e = scratch_ptr(&scratch);
  if (e != cudaSuccess)
    return fail(MLA_ERR_CUDA, std::string("scratch address lookup: ") + cudaGetErrorString(e));
  mla::PrefillArgs a{};
  a.g.H = d->H;
  a.g.Dn = d->qk_nope;
  a.g.Dr = d->qk_rope;
  a.g.Dl = d->kv_lora;
  a.g.Dv = d->v_head;
  a.g.scale = d->scale > 0.f ? d->scale : (float)(1.0 / sqrt((double)(d->qk_nope + d->qk_rope)));
  a.g.rope_base = d->rope_base > 0.f ? (double)d->rope_base : 10000.0;
  a.B = B;
  a.S = S;
  a.pos_base = pos_base;
  a.q = q;
  a.Lc = Lc;
  a.Rc = Rc;
  a.kv_b = kv_b;
  a.kv = scratch;  // every entry is written by the rebuild kernel before it is read
  a.out = out;
  e = mla::launch_prefill_simt(a, dtype, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(e));
  return MLA_OK;
}
