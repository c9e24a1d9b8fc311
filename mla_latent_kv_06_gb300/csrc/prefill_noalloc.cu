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
#include "prefill_tc.h"

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

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

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
  // Rebuilt KV bytes, B * (pos_base + S) * H * (qk_nope + v_head) * element size, each
  // product checked: a request whose size does not fit in 64 bits is refused too.
  const size_t el = dtype == MLA_F32 ? 4 : 2;
  const long long Tk = (long long)pos_base + S;
  size_t need = 0;
  const bool fits = Tk <= 0x7fffffffLL && (long long)B * Tk <= 0x7fffffffLL &&
                    !__builtin_mul_overflow((size_t)B * (size_t)Tk, (size_t)d->H, &need) &&
                    !__builtin_mul_overflow(need, (size_t)d->qk_nope + (size_t)d->v_head, &need) &&
                    !__builtin_mul_overflow(need, el, &need);
  if (!fits || need > kScratchBytes)
    return fail(MLA_ERR_INVALID, "rebuilt KV needs " + (fits ? std::to_string(need) : std::string("over 2^64")) +
                                     " bytes, more than the " + std::to_string(kScratchBytes) +
                                     "-byte static scratch of this entry point");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int cur = 0, sdev = 0;
  cudaError_t e = cudaGetDevice(&cur);
  if (e == cudaSuccess) e = cudaStreamGetDevice(st, &sdev);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, std::string("device lookup: ") + cudaGetErrorString(e));
  if (sdev != cur)
    return fail(MLA_ERR_INVALID, "the stream belongs to device " + std::to_string(sdev) +
                                     ", not the current device " + std::to_string(cur));
  unsigned char* scratch = nullptr;
  e = scratch_ptr(&scratch);
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
  a.kv = scratch;  // every entry is written by the rebuild before it is read
  a.out = out;
  // the same dispatch as mla_prefill_naive: the tensor-core kernels for bf16
  // GLM-shaped heads with 16-byte aligned tensors, the CUDA-core ones otherwise
  mla::call_begin();
  if (dtype == MLA_BF16 && mla::tc_prefill_geometry_ok(a.g) && aligned16(q) && aligned16(Lc) && aligned16(Rc) &&
      aligned16(kv_b)) {
    unsigned int* flags = mla::device_flags();
    if (!flags) return fail(MLA_ERR_CUDA, "cannot resolve the device status word");
    e = mla::launch_prefill_tc(a, flags, mla::wait_limit_ns(), st);
  } else {
    mla::kernel_mark(st, "prefill_simt");
    e = mla::launch_prefill_simt(a, dtype, st);
  }
  mla::call_end(st);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(e));
  return MLA_OK;
}
