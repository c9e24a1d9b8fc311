/*
 * mla.h -- C ABI of the GB300 MLA latent-KV hot path.
 *
 * Operations follow two web pages, cited by title and section:
 *   [MLA-KV] "MLA 注意力与 KV 缓存" (colibri-analysis 06)
 *   [FDSA]   "第 7 章 · 03 token 精确前向验证与 faithful DSA"
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *   never frees or keeps it.  Tensors are dense, row-major, innermost dimension
 *   contiguous, with the shapes written beside each argument.
 * - Calls only enqueue work on `stream` (a cudaStream_t; NULL = legacy default
 *   stream) and return at once.  They never synchronise and never allocate
 *   device memory: scratch space is the caller's `workspace` of at least
 *   `*_workspace_size()` bytes (256-byte aligned).  Calls that share a
 *   workspace must be ordered on one stream.
 * - Return value: MLA_OK, or a negative mla_status.  Argument errors are found
 *   on the host before anything is enqueued; the reason is in mla_last_error()
 *   (thread-local).  Bad values that live in device memory (sequence lengths,
 *   selected indices) are found by the kernels, which write NaN for the
 *   offending rows and raise a flag read by mla_device_status().
 * - Query positions: a call holds S new tokens per sequence whose cache rows
 *   are already written, so query s of sequence b sits at
 *   pos = T[b] - S + s and attends to keys t <= pos ([MLA-KV] §2: Tk = pos_base + S).
 * - dtype MLA_F32: q, Lc, Rc, kv_b are float; every kernel computes in fp32.
 *   dtype MLA_BF16: q, Lc, Rc, kv_b are bf16; products run on the tensor cores
 *   with fp32 accumulation.  Outputs are always float.
 */
#ifndef MLA_H
#define MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Head geometry of one attention layer ([MLA-KV] §2: qh = qk_nope + qk_rope,
 * kvb_dim = H * (qk_nope + v_head)). */
typedef struct mla_dims {
  int H;           /* attention heads                                        */
  int qk_nope;     /* non-rotary query/key width per head                    */
  int qk_rope;     /* rotary width (even); the rotated key is shared by heads */
  int kv_lora;     /* latent width of the cache                              */
  int v_head;      /* value width per head                                   */
  float scale;     /* softmax scale; <= 0 selects 1/sqrt(qk_nope + qk_rope)  */
  float rope_base; /* RoPE base; <= 0 selects 10000                          */
} mla_dims;

enum mla_dtype { MLA_F32 = 0, MLA_BF16 = 1 };

enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID = -1,     /* null pointer, bad size, misaligned pointer, short workspace */
  MLA_ERR_UNSUPPORTED = -2, /* valid request this build does not implement (shape/dtype)   */
  MLA_ERR_CUDA = -3,        /* a CUDA runtime call or a launch failed                       */
  MLA_ERR_DEVICE = -4       /* a kernel flagged bad device data or a wait that ran out      */
};

/* Device status flags (bits of the word returned by mla_device_status). */
enum mla_device_flag {
  MLA_DEV_BAD_LENGTH = 1,   /* some T[b] outside [S, T_cap]: that sequence was skipped      */
  MLA_DEV_BAD_INDEX = 2,    /* a selected index < 0 or > pos, or nsel outside [1, topk]     */
  MLA_DEV_TIMEOUT = 4       /* a bounded wait inside a kernel ran out; the kernel returned  */
};

/* Message of the last failing call on this thread ("" if none). */
const char* mla_last_error(void);

/* ABI version (incremented on any signature change). */
int mla_abi_version(void);

/* Waits on `stream`, then returns in *flags (may be NULL) the OR of the
 * mla_device_flag bits raised on the current device since the last call, and
 * clears them.  Returns MLA_OK, MLA_ERR_DEVICE if any flag was set, or
 * MLA_ERR_CUDA. */
int mla_device_status(void* stream, int* flags);

/* Optional per-kernel timing.  While set on the calling thread, every later
 * mla_* / dsa_* call records events[i] on its stream just before launching
 * its i-th kernel and, after its last kernel, one more event (so a call with n
 * kernels uses events[0..n]; it records no more than `count`).  `events` are
 * caller-owned cudaEvent_t handles; the array must stay valid while set.
 * Pass NULL, 0 to switch it off.  Returns MLA_OK. */
int mla_set_kernel_events(void* const* events, int count);

/* Comma-separated names of the kernels launched by the last call on this
 * thread, in launch order (for example "absorb,attention,combine"). */
const char* mla_last_launch_names(void);

/* Limit of every bounded wait inside the kernels, in nanoseconds of
 * %globaltimer (default 2e9).  Host-side setting, read at each launch. */
void mla_set_wait_limit_ns(long long ns);

/* ---------------------------------------------------------------------------
 * Weight-absorbed decode ([MLA-KV] §2.3, absorbed path)
 *
 *   qabs[h]   = sum_i q_nope[h,i] * W_UK[h,i,:]              (qt_addrow)
 *   q_rot[h]  = RoPE(q_rope[h], pos)                          ([MLA-KV] §2.1)
 *   score[t]  = scale * (qabs[h] . Lc[t] + q_rot[h] . Rc[t]), t <= pos
 *   clat[h]   = sum_t softmax(score)[t] * Lc[t]
 *   out[h]    = W_UV[h] * clat[h]                              (qt_matvec_rows)
 * with W_UK[h] = kv_b[h, 0:qk_nope, :], W_UV[h] = kv_b[h, qk_nope:, :].
 * RoPE pairs (x[2j], x[2j+1]) rotate by pos * rope_base^(-2j/qk_rope) into
 * (y[j], y[qk_rope/2 + j]).
 *
 *   q    [B, S, H, qk_nope+qk_rope]  query before RoPE
 *   Lc   [B, T_cap, kv_lora]         latent cache (after the cache writer's RMSNorm)
 *   Rc   [B, T_cap, qk_rope]         rotated key cache (already rotated)
 *   T    [B] int32                   cached rows per sequence, S <= T[b] <= T_cap
 *   kv_b [H, qk_nope+v_head, kv_lora]
 *   out  [B, S, H, v_head] float
 * The tensor-core path takes BF16 with H == 64, kv_lora == 512, qk_rope == 64,
 * qk_nope % 64 == 0 (<= 256), v_head % 128 == 0 and 16-byte aligned pointers;
 * every other valid request runs on the CUDA-core path.
 * ------------------------------------------------------------------------- */
size_t mla_decode_absorbed_workspace_size(const mla_dims* d, int dtype, int B, int S, int T_cap);
int mla_decode_absorbed(const mla_dims* d, int dtype, int B, int S,
                        const void* q, const void* Lc, const void* Rc, int T_cap,
                        const int32_t* T, const void* kv_b, float* out,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Number of kernels one mla_decode_absorbed (sparse = 0) or mla_sparse_decode
 * (sparse = 1) call launches for this geometry, dtype and batch (host-only query). */
int mla_decode_launch_count(const mla_dims* d, int dtype, int B, int S, int sparse);

/* ---------------------------------------------------------------------------
 * Sparse decode over DSA-selected keys ([MLA-KV] §2.2: the top-k keys chosen
 * by the indexer are reused by the attention of the shared layers)
 *
 * Same as mla_decode_absorbed, but query (b,s) attends only to the keys
 * sel[b,s,0:nsel[b,s]] (one selection shared by all heads).
 *   sel  [B, S, topk] int32, entries in [0, pos] (any order)
 *   nsel [B, S] int32 in [1, topk]
 * ------------------------------------------------------------------------- */
size_t mla_sparse_decode_workspace_size(const mla_dims* d, int dtype, int B, int S, int topk);
int mla_sparse_decode(const mla_dims* d, int dtype, int B, int S,
                      const void* q, const void* Lc, const void* Rc, int T_cap,
                      const int32_t* T, const void* kv_b,
                      const int32_t* sel, const int32_t* nsel, int topk, float* out,
                      void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Sparse decode of L layers that share one DSA selection ([MLA-KV] §2.2: the
 * shared layers reuse the indexer's top-k instead of running their own;
 * §2.3: each attention ends with its o projection)
 *
 * For layers l = 0..L-1 in order on `stream`, all with the same T, sel, nsel
 * and topk:
 *   out[l] = mla_sparse_decode(q[l], Lc[l], Rc[l], kv_b[l], sel, nsel)
 *   y[l]   = mla_o_proj(w_o[l], out[l])            (only when w_o != NULL)
 * q, Lc, Rc, kv_b, out, w_o and y are HOST arrays of L device pointers (one
 * layer each; the caller keeps them alive for the call only).  Every layer
 * has the shapes and dtype mla_sparse_decode documents, with one T_cap;
 *   w_o[l] [hidden, H*v_head] dtype, y[l] [B*S, hidden] float, out[l] 16-byte
 *   aligned when projected.
 * w_o == NULL skips the projections (hidden and y are then ignored).  Layer l
 * starts once layer l-1 has finished, as in a model whose query for layer l
 * comes from layer l-1's output; a layer's projection is a programmatic
 * dependent of its attention.  The arguments of all layers are checked
 * before the first launch.
 *   workspace: mla_sparse_decode_layers_workspace_size(d, dtype, B, S, topk,
 *              hidden) bytes (hidden = 0 without projection), 256-byte
 *              aligned, shared by the layers in stream order
 * Errors: as mla_sparse_decode and mla_o_proj; L < 1, a null array or a null
 * entry returns MLA_ERR_INVALID before anything is enqueued.  A launch error
 * in layer l returns at once, with layers 0..l-1 enqueued.
 * ------------------------------------------------------------------------- */
size_t mla_sparse_decode_layers_workspace_size(const mla_dims* d, int dtype, int B, int S, int topk, int hidden);
int mla_sparse_decode_layers(const mla_dims* d, int dtype, int L, int B, int S, const void* const* q,
                             const void* const* Lc, const void* const* Rc, int T_cap, const int32_t* T,
                             const void* const* kv_b, const int32_t* sel, const int32_t* nsel, int topk,
                             float* const* out, const void* const* w_o, int hidden, float* const* y,
                             void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Output projection ([MLA-KV] §2.3: both attention paths end with the o
 * output projection)
 *
 *   y[r, n] = sum_k w_o[n, k] * x[r, k]
 *   w_o [hidden, in_dim]  dtype (bf16 or float), 16-byte aligned
 *   x   [R, in_dim]       float, 16-byte aligned (a decode output [B, S, H, v_head] is R = B*S rows of
 *                         in_dim = H*v_head)
 *   y   [R, hidden]       float
 * in_dim a multiple of 8.  Up to 8 rows: one streaming pass over w_o on the
 * CUDA cores (fp32 arithmetic).  More rows with bf16 weights (in_dim and
 * hidden multiples of 64): x is rounded to bf16 in the workspace and the
 * product runs on the tensor cores; otherwise passes of 8 rows.
 *   workspace: mla_o_proj_workspace_size() bytes (0 for the streaming path)
 * mla_decode_oproj is mla_decode_absorbed followed by the projection of its
 * output, which stays in the workspace; the projection launches as a
 * programmatic dependent and starts reading w_o before the attention ends.
 * ------------------------------------------------------------------------- */
size_t mla_o_proj_workspace_size(int R, int in_dim, int hidden, int dtype);
int mla_o_proj(int R, int in_dim, int hidden, int dtype, const void* w_o, const float* x, float* y,
               void* workspace, size_t workspace_bytes, void* stream);
size_t mla_decode_oproj_workspace_size(const mla_dims* d, int dtype, int B, int S, int T_cap, int hidden);
int mla_decode_oproj(const mla_dims* d, int dtype, int B, int S, const void* q, const void* Lc, const void* Rc,
                     int T_cap, const int32_t* T, const void* kv_b, const void* w_o, int hidden, float* y,
                     void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Fused DSA selection ([MLA-KV] §2.2: indexer scores, then the causal top-k)
 *
 * dsa_index_scores followed by dsa_topk_select in one call, with the same
 * arguments and results (scores as written by dsa_index_scores; sel and nsel
 * bit-identical to dsa_topk_select).  With 32 index heads of 128 values the
 * indexer also writes, per CTA, the histogram of the top 11 bits of each
 * candidate's ordered score key into the workspace, and the top-k takes its
 * first radix pass from those histograms instead of recounting the scores.
 *   workspace: dsa_select_workspace_size() bytes (0 for other shapes), 256-byte aligned
 * ------------------------------------------------------------------------- */
size_t dsa_select_workspace_size(int B, int S, int n_ih, int index_hd, int T_cap, int topk);
int dsa_select(int B, int S, int n_ih, int index_hd, const float* q_idx, const float* w, const float* Ic,
               int T_cap, const int32_t* T, int topk, float* scores, int32_t* sel, int32_t* nsel,
               void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Paged cache layout (the same operations on a shared page pool)
 *
 * The pages fix no storage layout beyond one 576-value row per token
 * ([MLA-KV] §1); this layout lets sequences grow without a per-sequence
 * T_cap reservation.  Token t of sequence b lives at row
 *   block_table[b, t / page_size] * page_size + t % page_size
 * of the pools
 *   Lc_pages [num_pages, page_size, kv_lora]   dtype
 *   Rc_pages [num_pages, page_size, qk_rope]   dtype
 *   block_table [B, max_pages] int32: page indices in [0, num_pages); only the
 *               entries below ceil(T[b] / page_size) are read
 * The capacity of a sequence is max_pages * page_size (it plays the role of
 * T_cap: S <= T[b] <= max_pages * page_size).  A page index outside
 * [0, num_pages) is never dereferenced: the kernels raise MLA_DEV_BAD_INDEX
 * and that sequence's outputs are undefined.  Pools and per-sequence
 * capacities of 2^31 rows or more return MLA_ERR_UNSUPPORTED.  With bf16 and
 * the GLM-5.2 geometry the tensor-core kernels run when page_size is a
 * multiple of 128 (one key tile never spans two pages); other page sizes run
 * the CUDA-core kernels.  Workspace: mla_decode_paged_workspace_size and
 * mla_sparse_decode_workspace_size.
 * ------------------------------------------------------------------------- */
size_t mla_decode_paged_workspace_size(const mla_dims* d, int dtype, int B, int S, int max_pages, int page_size);
int mla_decode_paged(const mla_dims* d, int dtype, int B, int S, const void* q,
                     const void* Lc_pages, const void* Rc_pages, int num_pages, int page_size,
                     const int32_t* block_table, int max_pages, const int32_t* T, const void* kv_b,
                     float* out, void* workspace, size_t workspace_bytes, void* stream);
int mla_sparse_decode_paged(const mla_dims* d, int dtype, int B, int S, const void* q,
                            const void* Lc_pages, const void* Rc_pages, int num_pages, int page_size,
                            const int32_t* block_table, int max_pages, const int32_t* T, const void* kv_b,
                            const int32_t* sel, const int32_t* nsel, int topk, float* out,
                            void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * FP8 latent cache (a cache format of this library: the pages name FP8 only
 * as a weight format)
 *
 * The latent part of each cached row is kv_lora E4M3 codes (1 sign, 4
 * exponent bits with bias 7, 3 mantissa bits, no infinities, 0x7F/0xFF NaN,
 * largest finite value 448) with one scale for the whole cache:
 *   Lc[b,t,:] = lat_scale * e4m3(Lc8[b,t,:])
 *   Lc8 [B, T_cap, kv_lora] uint8 (or the pool [num_pages, page_size, kv_lora])
 *   Rc  [B, T_cap, qk_rope] bf16, unchanged
 * Half the bytes of a bf16 row's latent part.  RMSNorm bounds every written
 * value by sqrt(kv_lora) * max|kv_a_ln|, so lat_scale = that bound / 448
 * never saturates.
 *
 * mla_decode_fp8 / mla_decode_fp8_paged compute the absorbed decode of
 * mla_decode_absorbed (q, kv_b bf16; out float; T, pages as there) over the
 * dequantised latent.  The tensor-core kernels read the codes directly
 * (kind::f8f6f4 MMAs): each query row's absorbed latent query is rounded to
 * E4M3 with its own scale (its largest magnitude / 448), and the softmax
 * probabilities are rounded to E4M3 for the value product (row sums in
 * fp32).  Both roundings carry the E4M3 unit roundoff 2^-4, so results match
 * the exact attention over the dequantised cache to a few percent, not to
 * bf16 accuracy.  Only the GLM-5.2 head geometry (64 heads, kv_lora 512,
 * qk_rope 64) with 16-byte aligned tensors is served; page_size must be a
 * multiple of 128; anything else returns MLA_ERR_UNSUPPORTED.  lat_scale must
 * be positive and finite.  Workspace: mla_decode_fp8_workspace_size (the
 * paged call takes T_cap = max_pages * page_size).
 *
 * mla_cache_append_fp8 / _paged write the new rows as mla_cache_append does
 * (comp, kv_a_ln bf16), the latent values as E4M3 codes of
 * RMSNorm(...) / lat_scale (fp32 arithmetic, round to nearest even,
 * saturating at 448).  lat_scale must be positive, finite, with a finite
 * inverse.
 * ------------------------------------------------------------------------- */
size_t mla_decode_fp8_workspace_size(const mla_dims* d, int B, int S, int T_cap);
int mla_decode_fp8(const mla_dims* d, int B, int S, const void* q, const uint8_t* Lc8, const void* Rc,
                   float lat_scale, int T_cap, const int32_t* T, const void* kv_b, float* out,
                   void* workspace, size_t workspace_bytes, void* stream);
int mla_decode_fp8_paged(const mla_dims* d, int B, int S, const void* q, const uint8_t* Lc8_pages,
                         const void* Rc_pages, float lat_scale, int num_pages, int page_size,
                         const int32_t* block_table, int max_pages, const int32_t* T, const void* kv_b,
                         float* out, void* workspace, size_t workspace_bytes, void* stream);
int mla_cache_append_fp8(const mla_dims* d, int B, int S, const void* comp, const void* kv_a_ln, float rms_eps,
                         float lat_scale, int T_cap, const int32_t* T, uint8_t* Lc8, void* Rc, void* stream);
int mla_cache_append_fp8_paged(const mla_dims* d, int B, int S, const void* comp, const void* kv_a_ln,
                               float rms_eps, float lat_scale, uint8_t* Lc8_pages, void* Rc_pages, int num_pages,
                               int page_size, const int32_t* block_table, int max_pages, const int32_t* T,
                               void* stream);

/* ---------------------------------------------------------------------------
 * Non-absorbed prefill ([MLA-KV] §2.3, non-absorbed path)
 *
 * Step 1: one kv_b product rebuilds, for every key t < Tk = pos_base + S,
 *         KV[b,t,h,:] = kv_b[h] * Lc[b,t]  (k_nope = first qk_nope, value = rest).
 * Step 2: causal attention of query s (pos = pos_base + s):
 *         score = scale * (q_pass . k_nope[t] + q_rot . Rc[t]), t <= pos,
 *         softmax, out = sum_t p_t * value[t].
 *   q    [B, S, H, qk_nope+qk_rope]
 *   Lc   [B, Tk, kv_lora], Rc [B, Tk, qk_rope]
 *   kv_b [H, qk_nope+v_head, kv_lora]
 *   out  [B, S, H, v_head] float
 * The rebuilt KV lives in the workspace (dtype of the inputs).  BF16 with the
 * GLM-5.2 geometry (H 64, qk_nope 192, qk_rope 64, v_head 256) runs on the
 * tensor cores (kv_b GEMM + causal flash attention); other requests run on
 * the CUDA cores.
 * ------------------------------------------------------------------------- */
size_t mla_prefill_naive_workspace_size(const mla_dims* d, int dtype, int B, int S, int pos_base);
int mla_prefill_naive(const mla_dims* d, int dtype, int B, int S, int pos_base,
                      const void* q, const void* Lc, const void* Rc, const void* kv_b,
                      float* out, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Non-absorbed prefill without caller workspace.  The pages have no
 * counterpart of this entry point; it exists for callers that cannot allocate
 * device memory: code whose GPU memory belongs to a host framework's pool
 * that forbids third-party cudaMalloc, code on a latency-critical path that
 * cannot afford the device-wide synchronisation cudaMalloc/cudaFree may
 * cause, and plain C callers with no allocator at hand.
 *
 * Same arguments, results and kernels as mla_prefill_naive (the tensor-core
 * kernels for bf16 GLM-shaped heads with 16-byte aligned tensors, the
 * CUDA-core ones otherwise) minus the workspace: the rebuilt KV lives in a
 * 32 MiB static device array of the library, held by every GPU that loads it
 * until the process exits.  Calls needing more (B * (pos_base+S) * H *
 * (qk_nope+v_head) * sizeof(input dtype) > 32 MiB, for GLM-shaped bf16 heads
 * 585 keys) return MLA_ERR_INVALID with the sizes in mla_last_error().  The
 * stream must belong to the current device (MLA_ERR_INVALID otherwise): the
 * array's address is looked up per device.  The first call on a device looks
 * up that address (cudaGetSymbolAddress, with that device current); make that
 * first call before any stream capture.  The call allocates nothing.  All
 * calls share the one array, which keeps the last call's contents (every
 * entry is rewritten before it is read, so nothing needs clearing); calls
 * whose executions overlap on the GPU race on it, so order them on one stream.
 * ------------------------------------------------------------------------- */
int mla_prefill_naive_noalloc(const mla_dims* d, int dtype, int B, int S, int pos_base,
                              const void* q, const void* Lc, const void* Rc, const void* kv_b,
                              float* out, void* stream);

/* ---------------------------------------------------------------------------
 * DSA lightning-indexer scores ([MLA-KV] §2.2 "ReLU-gated" scores; the key
 * cache Ic holds index_hd fp32 values per token, [FDSA] §二)
 *
 *   scores[b,s,t] = sum_h w[b,s,h] * max(0, q_idx[b,s,h,:] . Ic[b,t,:])   t <= pos
 *                 = -inf                                                   pos < t < T_cap
 *   q_idx  [B, S, n_ih, index_hd] float (after the indexer's RoPE)
 *   w      [B, S, n_ih] float
 *   Ic     [B, T_cap, index_hd] float
 *   scores [B, S, T_cap] float
 * Products and sums are fp32 (integer-valued inputs give exact scores).
 * ------------------------------------------------------------------------- */
int dsa_index_scores(int B, int S, int n_ih, int index_hd,
                     const float* q_idx, const float* w, const float* Ic, int T_cap,
                     const int32_t* T, float* scores, void* stream);

/* ---------------------------------------------------------------------------
 * Causal top-k key selection ([MLA-KV] §2.2: "top-keep" selection into
 * dsa_sel / dsa_nsel; the indexer only prunes once the context exceeds topk)
 *
 * For each (b,s) with pos + 1 <= topk all keys 0..pos are kept; otherwise the
 * topk keys with the largest scores[b,s,t], t <= pos, where the lower index
 * wins a tie and -0.0 equals +0.0.  Scores must not be NaN.
 *   scores [B, S, T_cap] float (entries past pos are ignored)
 *   sel    [B, S, topk] int32: kept indices in ascending order, then -1
 *   nsel   [B, S] int32: number kept (min(pos + 1, topk))
 * ------------------------------------------------------------------------- */
size_t dsa_topk_select_workspace_size(int B, int S, int T_cap, int topk);
int dsa_topk_select(int B, int S, const float* scores, int T_cap, const int32_t* T, int topk,
                    int32_t* sel, int32_t* nsel, void* workspace, size_t workspace_bytes,
                    void* stream);

/* ---------------------------------------------------------------------------
 * Cache append ([MLA-KV] §2.1, KV path: the kv_a output comp of each new
 * token -> the first kv_lora values through RMSNorm(kv_a_ln) into Lc, the
 * last qk_rope values through the RoPE shared by all heads into Rc)
 *
 * The S new tokens of sequence b sit at pos = T[b] - S + s (T counts them):
 *   Lc[b,pos,:] = comp[b,s,0:kv_lora] / sqrt(mean(comp^2) + rms_eps) * kv_a_ln
 *   Rc[b,pos,:] = RoPE(comp[b,s,kv_lora:kv_lora+qk_rope], pos)  (pairs (x[2j],x[2j+1])
 *                 -> y[j], y[qk_rope/2+j], angle pos * rope_base^(-2j/qk_rope))
 *   comp    [B, S, kv_lora + qk_rope]   dtype
 *   kv_a_ln [kv_lora]                   dtype
 *   Lc      [B, T_cap, kv_lora]         dtype: only the rows pos are written
 *   Rc      [B, T_cap, qk_rope]         dtype: likewise
 * Arithmetic in fp32 (the angle reduced in double), rounded once to dtype.
 * Sequences with T[b] outside [S, T_cap] are left untouched and raise
 * MLA_DEV_BAD_LENGTH.  Uses d->kv_lora, d->qk_rope and d->rope_base only;
 * qk_rope above 256 returns MLA_ERR_UNSUPPORTED.
 * ------------------------------------------------------------------------- */
int mla_cache_append(const mla_dims* d, int dtype, int B, int S, const void* comp, const void* kv_a_ln,
                     float rms_eps, int T_cap, const int32_t* T, void* Lc, void* Rc, void* stream);
/* The same rows written into the paged pools (layout as for mla_decode_paged). */
int mla_cache_append_paged(const mla_dims* d, int dtype, int B, int S, const void* comp, const void* kv_a_ln,
                           float rms_eps, void* Lc_pages, void* Rc_pages, int num_pages, int page_size,
                           const int32_t* block_table, int max_pages, const int32_t* T, void* stream);

/* ---------------------------------------------------------------------------
 * Indexer key append ([MLA-KV] §2.2: the indexer key of each new token goes
 * through layernorm (eps 1e-6) and RoPE into Ic; Ic is fp32, [FDSA] §二)
 *
 *   Ic[b,pos,:] = (k - mean) / sqrt(var + ln_eps) * ln_w + ln_b, k = k_idx[b,s,:],
 *                 then its last rope_dim values rotated as in mla_cache_append
 *   k_idx [B, S, index_hd] float, ln_w [index_hd] float, ln_b [index_hd] float or NULL
 *   Ic    [B, T_cap, index_hd] float: only the rows pos = T[b] - S + s are written
 * rope_dim: even, 0 .. index_hd (0: no rotation), at most 256 (else
 * MLA_ERR_UNSUPPORTED); rope_base <= 0 means 10000.  Bad lengths as above.
 * ------------------------------------------------------------------------- */
int dsa_index_key_append(int B, int S, int index_hd, int rope_dim, const float* k_idx, const float* ln_w,
                         const float* ln_b, float ln_eps, float rope_base, int T_cap, const int32_t* T,
                         float* Ic, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H */
