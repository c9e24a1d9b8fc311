// api.cu -- the C ABI declared in include/mla.h: argument checks, workspace
// sizing, choice of kernel path, and the device status word.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "common.cuh"
#include "decode_tc.h"
#include "internal.h"
#include "prefill_tc.h"

#define MLA_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

thread_local std::string g_err;
thread_local void* const* g_events = nullptr;
thread_local int g_event_count = 0;
thread_local int g_event_next = 0;
thread_local std::string g_launch_names;
std::atomic<long long> g_wait_limit_ns{2000000000LL};

// Flags raised by kernels on this device (see mla_device_flag).
__device__ unsigned int g_dev_flags;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_flag_ptr[kMaxDevices] = {};

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(MLA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

// Device address of g_dev_flags for the current device (looked up once).
unsigned int* flags_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_flag_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_flags) != cudaSuccess) return nullptr;
    g_flag_ptr[dev] = static_cast<unsigned int*>(p);
  }
  return g_flag_ptr[dev];
}

bool resolve(const mla_dims* d, mla::Geometry* g) {
  if (!d) return false;
  if (d->H < 1 || d->qk_nope < 0 || d->qk_rope < 0 || d->kv_lora < 1 || d->v_head < 1) return false;
  if (d->qk_rope % 2 != 0 || d->qk_nope + d->qk_rope < 1) return false;
  g->H = d->H;
  g->Dn = d->qk_nope;
  g->Dr = d->qk_rope;
  g->Dl = d->kv_lora;
  g->Dv = d->v_head;
  g->scale = d->scale > 0.f ? d->scale : (float)(1.0 / std::sqrt((double)(d->qk_nope + d->qk_rope)));
  g->rope_base = d->rope_base > 0.f ? (double)d->rope_base : 10000.0;
  return true;
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(const mla_dims* d, int dtype, int B, int S, mla::Geometry* g) {
  if (!resolve(d, g)) return fail(MLA_ERR_INVALID, "invalid mla_dims (null, non-positive size or odd qk_rope)");
  if (dtype != MLA_F32 && dtype != MLA_BF16) return fail(MLA_ERR_INVALID, "unknown dtype %d", dtype);
  if (B < 1 || S < 1) return fail(MLA_ERR_INVALID, "B=%d and S=%d must be >= 1", B, S);
  return MLA_OK;
}

// The tensor-core decode covers the GLM-5.2 head geometry with bf16 inputs.
bool tc_decode_ok(const mla::Geometry& g, int dtype, const void* q, const void* Lc, const void* Rc,
                  const void* kv_b) {
  return dtype == MLA_BF16 && mla::tc_decode_geometry_ok(g) && aligned16(q) && aligned16(Lc) &&
         aligned16(Rc) && aligned16(kv_b);
}

}  // namespace

void mla::set_last_error(const char* msg) { g_err = msg ? msg : ""; }
unsigned int* mla::device_flags() { return flags_ptr(); }
long long mla::wait_limit_ns() { return g_wait_limit_ns.load(); }

namespace {
// Inside a stream capture a plain record only orders the graph; the external
// flag makes the graph record a timestamp on every replay.
void record_event(void* ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(st, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), st, cudaEventRecordExternal);
  else
    cudaEventRecord(static_cast<cudaEvent_t>(ev), st);
}
}  // namespace

void mla::call_begin() {
  g_event_next = 0;
  g_launch_names.clear();
}

void mla::kernel_mark(cudaStream_t st, const char* name) {
  if (g_events && g_event_next < g_event_count) record_event(g_events[g_event_next++], st);
  if (!g_launch_names.empty()) g_launch_names += ",";
  g_launch_names += name;
}

void mla::call_end(cudaStream_t st) {
  if (g_events && g_event_next < g_event_count) record_event(g_events[g_event_next++], st);
}

MLA_EXPORT int mla_set_kernel_events(void* const* events, int count) {
  g_events = count > 0 ? events : nullptr;
  g_event_count = count > 0 ? count : 0;
  return MLA_OK;
}

MLA_EXPORT const char* mla_last_launch_names(void) { return g_launch_names.c_str(); }

MLA_EXPORT const char* mla_last_error(void) { return g_err.c_str(); }

MLA_EXPORT int mla_abi_version(void) { return 1; }

MLA_EXPORT void mla_set_wait_limit_ns(long long ns) { g_wait_limit_ns.store(ns > 0 ? ns : 1); }

MLA_EXPORT int mla_device_status(void* stream, int* flags) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_device_status: stream synchronize");
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_dev_flags, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "mla_device_status: read flags");
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_dev_flags, &zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(e, "mla_device_status: clear flags");
  if (flags) *flags = (int)v;
  if (v) return fail(MLA_ERR_DEVICE, "device flags 0x%x raised", v);
  return MLA_OK;
}

// ---------------------------------------------------------------- decode
MLA_EXPORT size_t mla_decode_absorbed_workspace_size(const mla_dims* d, int dtype, int B, int S,
                                                      int T_cap) {
  mla::Geometry g;
  if (!resolve(d, &g) || B < 1 || S < 1 || T_cap < S) return 0;
  if (dtype == MLA_BF16 && mla::tc_decode_geometry_ok(g))
    return round256(mla::tc_decode_workspace_bytes(g, B, S, T_cap, /*sparse_topk=*/0));
  return 0;
}

namespace {
// Enqueues one absorbed decode (dense or over selected keys) on either path.
int run_decode(mla::DecodeArgs& a, int dtype, bool sparse, void* workspace, size_t workspace_bytes,
               void* stream, const char* what, bool own_call = true) {
  if (!a.pages.table && (long long)a.B * a.T_cap >= (1ll << 31))
    return fail(MLA_ERR_UNSUPPORTED, "B*T_cap of 2^31 rows or more");
  a.flags = flags_ptr();
  a.wait_limit_ns = g_wait_limit_ns.load();
  if (!a.flags) return fail(MLA_ERR_CUDA, "cannot resolve the device status word");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool pages_ok = !a.pages.table || a.pages.page_size % 128 == 0;
  cudaError_t e;
  if (own_call) mla::call_begin();
  if (pages_ok && tc_decode_ok(a.g, dtype, a.q, a.Lc, a.Rc, a.kv_b)) {
    size_t need = mla::tc_decode_workspace_bytes(a.g, a.B, a.S, sparse ? a.topk : a.T_cap, sparse ? a.topk : 0);
    if (need && (!workspace || workspace_bytes < need))
      return fail(MLA_ERR_INVALID, "workspace of %zu bytes < %zu required", workspace_bytes, need);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
      return fail(MLA_ERR_INVALID, "workspace must be 256-byte aligned");
    e = sparse ? mla::launch_sparse_decode_tc(a, workspace, workspace_bytes, st)
               : mla::launch_decode_tc(a, workspace, workspace_bytes, st);
  } else {
    mla::kernel_mark(st, sparse ? "sparse_decode_simt" : "decode_simt");
    e = mla::launch_decode_simt(a, dtype, sparse, st);
  }
  if (own_call) mla::call_end(st);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return MLA_OK;
}

// Page-pool arguments of the paged entry points.
int check_pages(int S, int num_pages, int page_size, const int32_t* block_table, int max_pages,
                mla::PageTable* pt) {
  if (!block_table) return fail(MLA_ERR_INVALID, "null block table");
  if (num_pages < 1 || page_size < 1 || max_pages < 1)
    return fail(MLA_ERR_INVALID, "num_pages=%d, page_size=%d and max_pages=%d must be >= 1", num_pages, page_size,
                max_pages);
  const long long cap = (long long)max_pages * page_size, pool = (long long)num_pages * page_size;
  if (cap >= (1ll << 31) || pool >= (1ll << 31))
    return fail(MLA_ERR_UNSUPPORTED, "page pool or per-sequence capacity of 2^31 rows or more");
  if (cap < S) return fail(MLA_ERR_INVALID, "max_pages*page_size=%lld < S=%d", cap, S);
  *pt = mla::PageTable{block_table, max_pages, page_size, num_pages};
  return MLA_OK;
}
}  // namespace

MLA_EXPORT int mla_decode_absorbed(const mla_dims* d, int dtype, int B, int S, const void* q,
                                   const void* Lc, const void* Rc, int T_cap, const int32_t* T,
                                   const void* kv_b, float* out, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  mla::Geometry g;
  int rc = check_common(d, dtype, B, S, &g);
  if (rc) return rc;
  if (T_cap < S) return fail(MLA_ERR_INVALID, "T_cap=%d < S=%d", T_cap, S);
  if (!q || !Lc || !Rc || !T || !kv_b || !out) return fail(MLA_ERR_INVALID, "null tensor pointer");
  mla::DecodeArgs a{};
  a.g = g;
  a.B = B;
  a.S = S;
  a.T_cap = T_cap;
  a.q = q;
  a.Lc = Lc;
  a.Rc = Rc;
  a.T = T;
  a.kv_b = kv_b;
  a.out = out;
  return run_decode(a, dtype, false, workspace, workspace_bytes, stream, "mla_decode_absorbed launch");
}

MLA_EXPORT size_t mla_decode_paged_workspace_size(const mla_dims* d, int dtype, int B, int S, int max_pages,
                                                  int page_size) {
  mla::Geometry g;
  if (!resolve(d, &g) || B < 1 || S < 1 || max_pages < 1 || page_size < 1) return 0;
  const long long cap = (long long)max_pages * page_size;
  if (cap < S || cap >= (1ll << 31)) return 0;
  if (dtype == MLA_BF16 && mla::tc_decode_geometry_ok(g) && page_size % 128 == 0)
    return round256(mla::tc_decode_workspace_bytes(g, B, S, (int)cap, /*sparse_topk=*/0));
  return 0;
}

MLA_EXPORT int mla_decode_paged(const mla_dims* d, int dtype, int B, int S, const void* q, const void* Lc_pages,
                                const void* Rc_pages, int num_pages, int page_size, const int32_t* block_table,
                                int max_pages, const int32_t* T, const void* kv_b, float* out, void* workspace,
                                size_t workspace_bytes, void* stream) {
  mla::Geometry g;
  int rc = check_common(d, dtype, B, S, &g);
  if (rc) return rc;
  mla::DecodeArgs a{};
  rc = check_pages(S, num_pages, page_size, block_table, max_pages, &a.pages);
  if (rc) return rc;
  if (!q || !Lc_pages || !Rc_pages || !T || !kv_b || !out) return fail(MLA_ERR_INVALID, "null tensor pointer");
  a.g = g;
  a.B = B;
  a.S = S;
  a.T_cap = max_pages * page_size;
  a.q = q;
  a.Lc = Lc_pages;
  a.Rc = Rc_pages;
  a.T = T;
  a.kv_b = kv_b;
  a.out = out;
  return run_decode(a, dtype, false, workspace, workspace_bytes, stream, "mla_decode_paged launch");
}

namespace {
int run_decode_fp8(mla::DecodeArgs& a, float lat_scale, void* workspace, size_t workspace_bytes, void* stream,
                   const char* what) {
  if (!(lat_scale > 0.f) || !std::isfinite(lat_scale))
    return fail(MLA_ERR_INVALID, "lat_scale must be positive and finite");
  if (!tc_decode_ok(a.g, MLA_BF16, a.q, a.Lc, a.Rc, a.kv_b))
    return fail(MLA_ERR_UNSUPPORTED, "the FP8 cache needs the 64-head, 512+64 latent geometry and 16-byte aligned "
                                     "tensors");
  if (a.pages.table && a.pages.page_size % 128 != 0)
    return fail(MLA_ERR_UNSUPPORTED, "page_size=%d is not a multiple of 128", a.pages.page_size);
  a.lat_fp8 = 1;
  a.lat_scale = lat_scale;
  return run_decode(a, MLA_BF16, false, workspace, workspace_bytes, stream, what);
}
}  // namespace

MLA_EXPORT size_t mla_decode_fp8_workspace_size(const mla_dims* d, int B, int S, int T_cap) {
  mla::Geometry g;
  if (!resolve(d, &g) || B < 1 || S < 1 || T_cap < S || !mla::tc_decode_geometry_ok(g)) return 0;
  return round256(mla::tc_decode_workspace_bytes(g, B, S, T_cap, /*sparse_topk=*/0));
}

MLA_EXPORT int mla_decode_fp8(const mla_dims* d, int B, int S, const void* q, const uint8_t* Lc8, const void* Rc,
                              float lat_scale, int T_cap, const int32_t* T, const void* kv_b, float* out,
                              void* workspace, size_t workspace_bytes, void* stream) {
  mla::Geometry g;
  int rc = check_common(d, MLA_BF16, B, S, &g);
  if (rc) return rc;
  if (T_cap < S) return fail(MLA_ERR_INVALID, "T_cap=%d < S=%d", T_cap, S);
  if (!q || !Lc8 || !Rc || !T || !kv_b || !out) return fail(MLA_ERR_INVALID, "null tensor pointer");
  mla::DecodeArgs a{};
  a.g = g;
  a.B = B;
  a.S = S;
  a.T_cap = T_cap;
  a.q = q;
  a.Lc = Lc8;
  a.Rc = Rc;
  a.T = T;
  a.kv_b = kv_b;
  a.out = out;
  return run_decode_fp8(a, lat_scale, workspace, workspace_bytes, stream, "mla_decode_fp8 launch");
}

MLA_EXPORT int mla_decode_fp8_paged(const mla_dims* d, int B, int S, const void* q, const uint8_t* Lc8_pages,
                                    const void* Rc_pages, float lat_scale, int num_pages, int page_size,
                                    const int32_t* block_table, int max_pages, const int32_t* T, const void* kv_b,
                                    float* out, void* workspace, size_t workspace_bytes, void* stream) {
  mla::Geometry g;
  int rc = check_common(d, MLA_BF16, B, S, &g);
  if (rc) return rc;
  mla::DecodeArgs a{};
  rc = check_pages(S, num_pages, page_size, block_table, max_pages, &a.pages);
  if (rc) return rc;
  if (!q || !Lc8_pages || !Rc_pages || !T || !kv_b || !out) return fail(MLA_ERR_INVALID, "null tensor pointer");
  a.g = g;
  a.B = B;
  a.S = S;
  a.T_cap = max_pages * page_size;
  a.q = q;
  a.Lc = Lc8_pages;
  a.Rc = Rc_pages;
  a.T = T;
  a.kv_b = kv_b;
  a.out = out;
  return run_decode_fp8(a, lat_scale, workspace, workspace_bytes, stream, "mla_decode_fp8_paged launch");
}

MLA_EXPORT int mla_decode_launch_count(const mla_dims* d, int dtype, int B, int S, int sparse) {
  mla::Geometry g;
  if (!resolve(d, &g) || B < 1 || S < 1) return 0;
  if (dtype == MLA_BF16 && mla::tc_decode_geometry_ok(g)) return mla::tc_decode_launch_count(sparse != 0, B, S);
  return 1;
}

// ---------------------------------------------------------------- sparse decode
MLA_EXPORT size_t mla_sparse_decode_workspace_size(const mla_dims* d, int dtype, int B, int S,
                                                    int topk) {
  mla::Geometry g;
  if (!resolve(d, &g) || B < 1 || S < 1 || topk < 1) return 0;
  if (dtype == MLA_BF16 && mla::tc_decode_geometry_ok(g))
    return round256(mla::tc_decode_workspace_bytes(g, B, S, topk, topk));
  return 0;
}

MLA_EXPORT int mla_sparse_decode(const mla_dims* d, int dtype, int B, int S, const void* q,
                                 const void* Lc, const void* Rc, int T_cap, const int32_t* T,
                                 const void* kv_b, const int32_t* sel, const int32_t* nsel, int topk,
                                 float* out, void* workspace, size_t workspace_bytes, void* stream) {
  mla::Geometry g;
  int rc = check_common(d, dtype, B, S, &g);
  if (rc) return rc;
  if (T_cap < S) return fail(MLA_ERR_INVALID, "T_cap=%d < S=%d", T_cap, S);
  if (topk < 1) return fail(MLA_ERR_INVALID, "topk=%d must be >= 1", topk);
  if (!q || !Lc || !Rc || !T || !kv_b || !out || !sel || !nsel)
    return fail(MLA_ERR_INVALID, "null tensor pointer");
  mla::DecodeArgs a{};
  a.g = g;
  a.B = B;
  a.S = S;
  a.T_cap = T_cap;
  a.q = q;
  a.Lc = Lc;
  a.Rc = Rc;
  a.T = T;
  a.kv_b = kv_b;
  a.out = out;
  a.sel = sel;
  a.nsel = nsel;
  a.topk = topk;
  return run_decode(a, dtype, true, workspace, workspace_bytes, stream, "mla_sparse_decode launch");
}

MLA_EXPORT int mla_sparse_decode_paged(const mla_dims* d, int dtype, int B, int S, const void* q,
                                       const void* Lc_pages, const void* Rc_pages, int num_pages, int page_size,
                                       const int32_t* block_table, int max_pages, const int32_t* T,
                                       const void* kv_b, const int32_t* sel, const int32_t* nsel, int topk,
                                       float* out, void* workspace, size_t workspace_bytes, void* stream) {
  mla::Geometry g;
  int rc = check_common(d, dtype, B, S, &g);
  if (rc) return rc;
  mla::DecodeArgs a{};
  rc = check_pages(S, num_pages, page_size, block_table, max_pages, &a.pages);
  if (rc) return rc;
  if (topk < 1) return fail(MLA_ERR_INVALID, "topk=%d must be >= 1", topk);
  if (!q || !Lc_pages || !Rc_pages || !T || !kv_b || !out || !sel || !nsel)
    return fail(MLA_ERR_INVALID, "null tensor pointer");
  a.g = g;
  a.B = B;
  a.S = S;
  a.T_cap = max_pages * page_size;
  a.q = q;
  a.Lc = Lc_pages;
  a.Rc = Rc_pages;
  a.T = T;
  a.kv_b = kv_b;
  a.out = out;
  a.sel = sel;
  a.nsel = nsel;
  a.topk = topk;
  return run_decode(a, dtype, true, workspace, workspace_bytes, stream, "mla_sparse_decode_paged launch");
}

// ---------------------------------------------------------------- prefill
MLA_EXPORT size_t mla_prefill_naive_workspace_size(const mla_dims* d, int dtype, int B, int S,
                                                    int pos_base) {
  mla::Geometry g;
  if (!resolve(d, &g) || B < 1 || S < 1 || pos_base < 0) return 0;
  size_t el = dtype == MLA_F32 ? 4 : 2;
  size_t Tk = (size_t)pos_base + S;
  return round256((size_t)B * Tk * g.H * (g.Dn + g.Dv) * el);
}

MLA_EXPORT int mla_prefill_naive(const mla_dims* d, int dtype, int B, int S, int pos_base,
                                 const void* q, const void* Lc, const void* Rc, const void* kv_b,
                                 float* out, void* workspace, size_t workspace_bytes, void* stream) {
  mla::Geometry g;
  int rc = check_common(d, dtype, B, S, &g);
  if (rc) return rc;
  if (pos_base < 0) return fail(MLA_ERR_INVALID, "pos_base=%d must be >= 0", pos_base);
  if (!q || !Lc || !Rc || !kv_b || !out) return fail(MLA_ERR_INVALID, "null tensor pointer");
  size_t need = mla_prefill_naive_workspace_size(d, dtype, B, S, pos_base);
  if (!workspace || workspace_bytes < need)
    return fail(MLA_ERR_INVALID, "workspace of %zu bytes < %zu required", workspace_bytes, need);
  mla::PrefillArgs a{};
  a.g = g;
  a.B = B;
  a.S = S;
  a.pos_base = pos_base;
  a.q = q;
  a.Lc = Lc;
  a.Rc = Rc;
  a.kv_b = kv_b;
  a.kv = workspace;
  a.out = out;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  mla::call_begin();
  if (dtype == MLA_BF16 && mla::tc_prefill_geometry_ok(g) && aligned16(q) && aligned16(Lc) && aligned16(Rc) &&
      aligned16(kv_b) && aligned16(workspace)) {
    unsigned int* flags = flags_ptr();
    if (!flags) return fail(MLA_ERR_CUDA, "cannot resolve the device status word");
    e = mla::launch_prefill_tc(a, flags, g_wait_limit_ns.load(), st);
  } else {
    mla::kernel_mark(st, "prefill_simt");
    e = mla::launch_prefill_simt(a, dtype, st);
  }
  mla::call_end(st);
  if (e != cudaSuccess) return cuda_fail(e, "mla_prefill_naive launch");
  return MLA_OK;
}

// ---------------------------------------------------------------- DSA
MLA_EXPORT int dsa_index_scores(int B, int S, int n_ih, int index_hd, const float* q_idx,
                                const float* w, const float* Ic, int T_cap, const int32_t* T,
                                float* scores, void* stream) {
  if (B < 1 || S < 1 || n_ih < 1 || index_hd < 1 || T_cap < S)
    return fail(MLA_ERR_INVALID, "bad sizes B=%d S=%d n_ih=%d index_hd=%d T_cap=%d", B, S, n_ih,
                index_hd, T_cap);
  if (!q_idx || !w || !Ic || !T || !scores) return fail(MLA_ERR_INVALID, "null tensor pointer");
  size_t smem = sizeof(float) * ((size_t)n_ih * index_hd + n_ih + 128 * (size_t)(index_hd + 1) + 256);
  if (smem > 220 * 1024)
    return fail(MLA_ERR_UNSUPPORTED, "n_ih*index_hd too large for one CTA (%zu bytes)", smem);
  mla::IndexArgs a{B, S, n_ih, index_hd, T_cap, q_idx, w, Ic, T, scores, flags_ptr(), g_wait_limit_ns.load(), nullptr};
  if (!a.flags) return fail(MLA_ERR_CUDA, "cannot resolve the device status word");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  mla::call_begin();
  mla::kernel_mark(st, "index_scores");
  cudaError_t e = mla::launch_index_scores(a, st);
  mla::call_end(st);
  if (e != cudaSuccess) return cuda_fail(e, "dsa_index_scores launch");
  return MLA_OK;
}

MLA_EXPORT size_t dsa_topk_select_workspace_size(int B, int S, int T_cap, int topk) {
  (void)B;
  (void)S;
  (void)T_cap;
  (void)topk;
  return 0;
}

MLA_EXPORT int dsa_topk_select(int B, int S, const float* scores, int T_cap, const int32_t* T,
                               int topk, int32_t* sel, int32_t* nsel, void* workspace,
                               size_t workspace_bytes, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (B < 1 || S < 1 || T_cap < S || topk < 1)
    return fail(MLA_ERR_INVALID, "bad sizes B=%d S=%d T_cap=%d topk=%d", B, S, T_cap, topk);
  if (!scores || !T || !sel || !nsel) return fail(MLA_ERR_INVALID, "null tensor pointer");
  mla::TopkArgs a{B, S, T_cap, topk, scores, T, sel, nsel, flags_ptr(), nullptr, 0};
  if (!a.flags) return fail(MLA_ERR_CUDA, "cannot resolve the device status word");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  mla::call_begin();
  mla::kernel_mark(st, "topk_select");
  cudaError_t e = mla::launch_topk_select(a, st);
  mla::call_end(st);
  if (e != cudaSuccess) return cuda_fail(e, "dsa_topk_select launch");
  return MLA_OK;
}

// ---------------------------------------------------------------- fused DSA selection
namespace {
size_t dsa_select_ws(int B, int S, int n_ih, int index_hd, int T_cap) {
  const int parts = mla::index_tc_parts(B, S, n_ih, index_hd, T_cap);
  return parts > 0 ? round256((size_t)B * S * parts * 2048 * sizeof(uint32_t)) : 0;
}
}  // namespace

MLA_EXPORT size_t dsa_select_workspace_size(int B, int S, int n_ih, int index_hd, int T_cap, int topk) {
  if (B < 1 || S < 1 || n_ih < 1 || index_hd < 1 || T_cap < S || topk < 1) return 0;
  return dsa_select_ws(B, S, n_ih, index_hd, T_cap);
}

MLA_EXPORT int dsa_select(int B, int S, int n_ih, int index_hd, const float* q_idx, const float* w,
                          const float* Ic, int T_cap, const int32_t* T, int topk, float* scores, int32_t* sel,
                          int32_t* nsel, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 1 || S < 1 || n_ih < 1 || index_hd < 1 || T_cap < S || topk < 1)
    return fail(MLA_ERR_INVALID, "bad sizes B=%d S=%d n_ih=%d index_hd=%d T_cap=%d topk=%d", B, S, n_ih, index_hd,
                T_cap, topk);
  if (!q_idx || !w || !Ic || !T || !scores || !sel || !nsel) return fail(MLA_ERR_INVALID, "null tensor pointer");
  size_t smem = sizeof(float) * ((size_t)n_ih * index_hd + n_ih + 128 * (size_t)(index_hd + 1) + 256);
  if (smem > 220 * 1024)
    return fail(MLA_ERR_UNSUPPORTED, "n_ih*index_hd too large for one CTA (%zu bytes)", smem);
  const size_t need = dsa_select_ws(B, S, n_ih, index_hd, T_cap);
  if (need && (!workspace || workspace_bytes < need))
    return fail(MLA_ERR_INVALID, "workspace of %zu bytes < %zu required", workspace_bytes, need);
  unsigned int* flags = flags_ptr();
  if (!flags) return fail(MLA_ERR_CUDA, "cannot resolve the device status word");
  uint32_t* hpart = need ? static_cast<uint32_t*>(workspace) : nullptr;
  mla::IndexArgs ia{B, S, n_ih, index_hd, T_cap, q_idx, w, Ic, T, scores, flags, g_wait_limit_ns.load(), hpart};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  mla::call_begin();
  mla::kernel_mark(st, "index_scores");
  cudaError_t e = mla::launch_index_scores_tc(ia, st);
  if (e == cudaErrorNotSupported) {  // other shapes: CUDA-core indexer, the top-k builds its own first pass
    hpart = nullptr;
    ia.hpart = nullptr;
    e = mla::launch_index_scores(ia, st);
  }
  if (e != cudaSuccess) {
    mla::call_end(st);
    return cuda_fail(e, "dsa_select indexer launch");
  }
  const int parts = hpart ? mla::index_tc_parts(B, S, n_ih, index_hd, T_cap) : 0;
  mla::TopkArgs ta{B, S, T_cap, topk, scores, T, sel, nsel, flags, hpart, parts};
  mla::kernel_mark(st, "topk_select");
  e = mla::launch_topk_select(ta, st);
  mla::call_end(st);
  if (e != cudaSuccess) return cuda_fail(e, "dsa_select top-k launch");
  return MLA_OK;
}

// ---------------------------------------------------------------- output projection
namespace {
int check_oproj(int R, int in_dim, int hidden, int dtype, const void* w_o, const float* x, const float* y) {
  if (R < 1 || in_dim < 8 || hidden < 1 || in_dim % 8 != 0)
    return fail(MLA_ERR_INVALID, "bad sizes R=%d in_dim=%d hidden=%d (in_dim a multiple of 8)", R, in_dim, hidden);
  if (dtype != MLA_F32 && dtype != MLA_BF16) return fail(MLA_ERR_INVALID, "unknown dtype %d", dtype);
  if (!w_o || !x || !y) return fail(MLA_ERR_INVALID, "null tensor pointer");
  if (!aligned16(w_o) || !aligned16(x)) return fail(MLA_ERR_INVALID, "w_o and x must be 16-byte aligned");
  return MLA_OK;
}
}  // namespace

MLA_EXPORT size_t mla_o_proj_workspace_size(int R, int in_dim, int hidden, int dtype) {
  if (R < 1 || in_dim < 8 || hidden < 1) return 0;
  return round256(mla::oproj_workspace_bytes(R, in_dim, hidden, dtype));
}

MLA_EXPORT int mla_o_proj(int R, int in_dim, int hidden, int dtype, const void* w_o, const float* x, float* y,
                          void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_oproj(R, in_dim, hidden, dtype, w_o, x, y);
  if (rc) return rc;
  const size_t need = mla::oproj_workspace_bytes(R, in_dim, hidden, dtype);
  if (need && (!workspace || workspace_bytes < need))
    return fail(MLA_ERR_INVALID, "workspace of %zu bytes < %zu required", workspace_bytes, need);
  if (need && !aligned16(workspace)) return fail(MLA_ERR_INVALID, "workspace must be 256-byte aligned");
  unsigned int* flags = flags_ptr();
  if (!flags) return fail(MLA_ERR_CUDA, "cannot resolve the device status word");
  mla::OprojArgs a{R, in_dim, hidden, dtype, w_o, x, y, workspace};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  mla::call_begin();
  cudaError_t e = mla::launch_oproj(a, false, flags, g_wait_limit_ns.load(), st);
  mla::call_end(st);
  if (e != cudaSuccess) return cuda_fail(e, "mla_o_proj launch");
  return MLA_OK;
}

namespace {
// Decode workspace, then out [R, H, v_head] fp32, then the projection's scratch.
struct OprojPlan {
  size_t dec, out_off, op_off, total;
};
OprojPlan oproj_plan(const mla::Geometry& g, int dtype, int B, int S, int T_cap, int hidden) {
  OprojPlan p{};
  p.dec = (dtype == MLA_BF16 && mla::tc_decode_geometry_ok(g)) ? round256(mla::tc_decode_workspace_bytes(g, B, S, T_cap, 0))
                                                               : 0;
  p.out_off = p.dec;
  p.op_off = p.out_off + round256((size_t)B * S * g.H * g.Dv * sizeof(float));
  p.total = p.op_off + round256(mla::oproj_workspace_bytes(B * S, g.H * g.Dv, hidden, dtype));
  return p;
}
}  // namespace

MLA_EXPORT size_t mla_decode_oproj_workspace_size(const mla_dims* d, int dtype, int B, int S, int T_cap, int hidden) {
  mla::Geometry g;
  if (!resolve(d, &g) || B < 1 || S < 1 || T_cap < S || hidden < 1) return 0;
  return oproj_plan(g, dtype, B, S, T_cap, hidden).total;
}

MLA_EXPORT int mla_decode_oproj(const mla_dims* d, int dtype, int B, int S, const void* q, const void* Lc,
                                const void* Rc, int T_cap, const int32_t* T, const void* kv_b, const void* w_o,
                                int hidden, float* y, void* workspace, size_t workspace_bytes, void* stream) {
  mla::Geometry g;
  int rc = check_common(d, dtype, B, S, &g);
  if (rc) return rc;
  if (T_cap < S) return fail(MLA_ERR_INVALID, "T_cap=%d < S=%d", T_cap, S);
  if (!q || !Lc || !Rc || !T || !kv_b) return fail(MLA_ERR_INVALID, "null tensor pointer");
  const int in_dim = g.H * g.Dv;
  if (!workspace) return fail(MLA_ERR_INVALID, "null workspace (the attention output lives there)");
  rc = check_oproj(B * S, in_dim, hidden, dtype, w_o, static_cast<const float*>(workspace), y);
  if (rc) return rc;
  const OprojPlan pl = oproj_plan(g, dtype, B, S, T_cap, hidden);
  if (workspace_bytes < pl.total)
    return fail(MLA_ERR_INVALID, "workspace of %zu bytes < %zu required", workspace_bytes, pl.total);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(MLA_ERR_INVALID, "workspace must be 256-byte aligned");
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  float* out = reinterpret_cast<float*>(ws + pl.out_off);
  mla::DecodeArgs a{};
  a.g = g;
  a.B = B;
  a.S = S;
  a.T_cap = T_cap;
  a.q = q;
  a.Lc = Lc;
  a.Rc = Rc;
  a.T = T;
  a.kv_b = kv_b;
  a.out = out;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  mla::call_begin();
  rc = run_decode(a, dtype, false, pl.dec ? ws : nullptr, pl.dec, stream, "mla_decode_oproj attention launch", false);
  if (rc) {
    mla::call_end(st);
    return rc;
  }
  mla::OprojArgs o{B * S, in_dim, hidden, dtype, w_o, out, y, ws + pl.op_off};
  cudaError_t e = mla::launch_oproj(o, true, a.flags, a.wait_limit_ns, st);
  mla::call_end(st);
  if (e != cudaSuccess) return cuda_fail(e, "mla_decode_oproj projection launch");
  return MLA_OK;
}

// Layers sharing one DSA selection: workspace = the sparse decode's, then the
// projection's (bf16 rows of x for its GEMM path).
namespace {
struct LayersPlan {
  size_t dec, op_off, total;
};
LayersPlan layers_plan(const mla::Geometry& g, int dtype, int B, int S, int topk, int hidden) {
  LayersPlan p{};
  p.dec = (dtype == MLA_BF16 && mla::tc_decode_geometry_ok(g))
              ? round256(mla::tc_decode_workspace_bytes(g, B, S, topk, topk))
              : 0;
  p.op_off = p.dec;
  p.total = p.op_off + (hidden > 0 ? round256(mla::oproj_workspace_bytes(B * S, g.H * g.Dv, hidden, dtype)) : 0);
  return p;
}
}  // namespace

MLA_EXPORT size_t mla_sparse_decode_layers_workspace_size(const mla_dims* d, int dtype, int B, int S, int topk,
                                                          int hidden) {
  mla::Geometry g;
  if (!resolve(d, &g) || B < 1 || S < 1 || topk < 1 || hidden < 0) return 0;
  return layers_plan(g, dtype, B, S, topk, hidden).total;
}

MLA_EXPORT int mla_sparse_decode_layers(const mla_dims* d, int dtype, int L, int B, int S, const void* const* q,
                                        const void* const* Lc, const void* const* Rc, int T_cap, const int32_t* T,
                                        const void* const* kv_b, const int32_t* sel, const int32_t* nsel, int topk,
                                        float* const* out, const void* const* w_o, int hidden, float* const* y,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  mla::Geometry g;
  int rc = check_common(d, dtype, B, S, &g);
  if (rc) return rc;
  if (L < 1) return fail(MLA_ERR_INVALID, "L=%d must be >= 1", L);
  if (T_cap < S) return fail(MLA_ERR_INVALID, "T_cap=%d < S=%d", T_cap, S);
  if (topk < 1) return fail(MLA_ERR_INVALID, "topk=%d must be >= 1", topk);
  if (!q || !Lc || !Rc || !kv_b || !out) return fail(MLA_ERR_INVALID, "null per-layer pointer array");
  if (!T || !sel || !nsel) return fail(MLA_ERR_INVALID, "null tensor pointer");
  if (w_o && !y) return fail(MLA_ERR_INVALID, "null per-layer pointer array");
  for (int l = 0; l < L; ++l)
    if (!q[l] || !Lc[l] || !Rc[l] || !kv_b[l] || !out[l])
      return fail(MLA_ERR_INVALID, "null tensor pointer for layer %d", l);
  const int in_dim = g.H * g.Dv;
  if (w_o)
    for (int l = 0; l < L; ++l) {
      rc = check_oproj(B * S, in_dim, hidden, dtype, w_o[l], out[l], y[l]);
      if (rc) return rc;
    }
  const LayersPlan pl = layers_plan(g, dtype, B, S, topk, w_o ? hidden : 0);
  if (pl.total && (!workspace || workspace_bytes < pl.total))
    return fail(MLA_ERR_INVALID, "workspace of %zu bytes < %zu required", workspace_bytes, pl.total);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(MLA_ERR_INVALID, "workspace must be 256-byte aligned");
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  mla::call_begin();
  for (int l = 0; l < L && rc == MLA_OK; ++l) {
    mla::DecodeArgs a{};
    a.g = g;
    a.B = B;
    a.S = S;
    a.T_cap = T_cap;
    a.q = q[l];
    a.Lc = Lc[l];
    a.Rc = Rc[l];
    a.T = T;
    a.kv_b = kv_b[l];
    a.out = out[l];
    a.sel = sel;
    a.nsel = nsel;
    a.topk = topk;
    a.stage_parity = l & 1;
    a.gather_pdl = l > 0 ? 1 : 0;
    rc = run_decode(a, dtype, true, pl.dec ? ws : nullptr, pl.dec, stream, "mla_sparse_decode_layers launch", false);
    if (rc == MLA_OK && w_o) {  // the layer's projection, a programmatic dependent of its attention
      mla::OprojArgs o{B * S, in_dim, hidden, dtype, w_o[l], out[l], y[l], ws + pl.op_off};
      cudaError_t e = mla::launch_oproj(o, true, a.flags, a.wait_limit_ns, st);
      if (e != cudaSuccess) rc = cuda_fail(e, "mla_sparse_decode_layers projection launch");
    }
  }
  mla::call_end(st);
  return rc;
}

// ---------------------------------------------------------------- cache append
namespace {
int run_cache_append(const mla_dims* d, int dtype, int B, int S, const void* comp, const void* kv_a_ln,
                     float rms_eps, int T_cap, const int32_t* T, void* Lc, void* Rc, const mla::PageTable& pages,
                     void* stream, const char* what, float lat_scale = 0.f) {
  mla::Geometry g;
  int rc = check_common(d, dtype, B, S, &g);
  if (rc != MLA_OK) return rc;
  if (T_cap < S) return fail(MLA_ERR_INVALID, "T_cap=%d < S=%d", T_cap, S);
  if (!(rms_eps >= 0.f)) return fail(MLA_ERR_INVALID, "rms_eps must be >= 0");
  if (!comp || !kv_a_ln || !T || !Lc || (g.Dr > 0 && !Rc)) return fail(MLA_ERR_INVALID, "null tensor pointer");
  if (g.Dr > 2 * mla::kMaxRopePairs) return fail(MLA_ERR_UNSUPPORTED, "qk_rope=%d above %d", g.Dr, 2 * mla::kMaxRopePairs);
  if (g.Dl > mla::kMaxAppendWidth)
    return fail(MLA_ERR_UNSUPPORTED, "kv_lora=%d above %d", g.Dl, mla::kMaxAppendWidth);
  if (!pages.table && (long long)B * T_cap >= (1ll << 31))
    return fail(MLA_ERR_UNSUPPORTED, "B*T_cap of 2^31 rows or more");
  mla::AppendArgs a{B, S, T_cap, g.Dl, g.Dr, comp, kv_a_ln, rms_eps, T, Lc, Rc, flags_ptr(), pages, {}};
  if (lat_scale != 0.f) {  // the FP8 cache
    a.lat_fp8 = 1;
    a.lat_inv_scale = 1.f / lat_scale;
  }
  for (int j = 0; j < g.Dr / 2; ++j) a.turn[j] = mla::rope_turns(std::pow(g.rope_base, -2.0 * j / g.Dr));
  if (!a.flags) return fail(MLA_ERR_CUDA, "cannot resolve the device status word");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  mla::call_begin();
  mla::kernel_mark(st, "cache_append");
  cudaError_t e = mla::launch_cache_append(a, dtype, st);
  mla::call_end(st);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return MLA_OK;
}
}  // namespace

MLA_EXPORT int mla_cache_append(const mla_dims* d, int dtype, int B, int S, const void* comp,
                                const void* kv_a_ln, float rms_eps, int T_cap, const int32_t* T, void* Lc,
                                void* Rc, void* stream) {
  return run_cache_append(d, dtype, B, S, comp, kv_a_ln, rms_eps, T_cap, T, Lc, Rc, mla::PageTable{}, stream,
                          "mla_cache_append launch");
}

MLA_EXPORT int mla_cache_append_paged(const mla_dims* d, int dtype, int B, int S, const void* comp,
                                      const void* kv_a_ln, float rms_eps, void* Lc_pages, void* Rc_pages,
                                      int num_pages, int page_size, const int32_t* block_table, int max_pages,
                                      const int32_t* T, void* stream) {
  mla::PageTable pt{};
  int rc = check_pages(S, num_pages, page_size, block_table, max_pages, &pt);
  if (rc) return rc;
  return run_cache_append(d, dtype, B, S, comp, kv_a_ln, rms_eps, max_pages * page_size, T, Lc_pages, Rc_pages, pt,
                          stream, "mla_cache_append_paged launch");
}

MLA_EXPORT int mla_cache_append_fp8(const mla_dims* d, int B, int S, const void* comp, const void* kv_a_ln,
                                    float rms_eps, float lat_scale, int T_cap, const int32_t* T, uint8_t* Lc8,
                                    void* Rc, void* stream) {
  if (!(lat_scale > 0.f) || !std::isfinite(lat_scale) || !std::isfinite(1.f / lat_scale))
    return fail(MLA_ERR_INVALID, "lat_scale must be positive and finite with a finite inverse");
  return run_cache_append(d, MLA_BF16, B, S, comp, kv_a_ln, rms_eps, T_cap, T, Lc8, Rc, mla::PageTable{}, stream,
                          "mla_cache_append_fp8 launch", lat_scale);
}

MLA_EXPORT int mla_cache_append_fp8_paged(const mla_dims* d, int B, int S, const void* comp, const void* kv_a_ln,
                                          float rms_eps, float lat_scale, uint8_t* Lc8_pages, void* Rc_pages,
                                          int num_pages, int page_size, const int32_t* block_table, int max_pages,
                                          const int32_t* T, void* stream) {
  if (!(lat_scale > 0.f) || !std::isfinite(lat_scale) || !std::isfinite(1.f / lat_scale))
    return fail(MLA_ERR_INVALID, "lat_scale must be positive and finite with a finite inverse");
  mla::PageTable pt{};
  int rc = check_pages(S, num_pages, page_size, block_table, max_pages, &pt);
  if (rc) return rc;
  return run_cache_append(d, MLA_BF16, B, S, comp, kv_a_ln, rms_eps, max_pages * page_size, T, Lc8_pages, Rc_pages,
                          pt, stream, "mla_cache_append_fp8_paged launch", lat_scale);
}

MLA_EXPORT int dsa_index_key_append(int B, int S, int index_hd, int rope_dim, const float* k_idx,
                                    const float* ln_w, const float* ln_b, float ln_eps, float rope_base,
                                    int T_cap, const int32_t* T, float* Ic, void* stream) {
  if (B < 1 || S < 1 || index_hd < 1 || T_cap < S)
    return fail(MLA_ERR_INVALID, "bad sizes B=%d S=%d index_hd=%d T_cap=%d", B, S, index_hd, T_cap);
  if (rope_dim < 0 || rope_dim > index_hd || rope_dim % 2 != 0)
    return fail(MLA_ERR_INVALID, "rope_dim=%d must be even and within [0, index_hd=%d]", rope_dim, index_hd);
  if (index_hd > mla::kMaxAppendWidth)
    return fail(MLA_ERR_UNSUPPORTED, "index_hd=%d above %d", index_hd, mla::kMaxAppendWidth);
  if (!(ln_eps >= 0.f)) return fail(MLA_ERR_INVALID, "ln_eps must be >= 0");
  if (!k_idx || !ln_w || !T || !Ic) return fail(MLA_ERR_INVALID, "null tensor pointer");
  if (rope_dim > 2 * mla::kMaxRopePairs)
    return fail(MLA_ERR_UNSUPPORTED, "rope_dim=%d above %d", rope_dim, 2 * mla::kMaxRopePairs);
  mla::KeyAppendArgs a{B, S, T_cap, index_hd, rope_dim, k_idx, ln_w, ln_b, ln_eps, T, Ic, flags_ptr(), {}};
  const double base = rope_base > 0.f ? (double)rope_base : 10000.0;
  for (int j = 0; j < rope_dim / 2; ++j) a.turn[j] = mla::rope_turns(std::pow(base, -2.0 * j / rope_dim));
  if (!a.flags) return fail(MLA_ERR_CUDA, "cannot resolve the device status word");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  mla::call_begin();
  mla::kernel_mark(st, "index_key_append");
  cudaError_t e = mla::launch_index_key_append(a, st);
  mla::call_end(st);
  if (e != cudaSuccess) return cuda_fail(e, "dsa_index_key_append launch");
  return MLA_OK;
}
