"""Plain, slow fp64 CPU oracle for the MLA latent-KV hot path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import or run anything in this
package.  The CUDA library never calls it and shares no code with it.

Sources, cited by page title and section:

* [MLA-KV] the page "MLA 注意力与 KV 缓存" (colibri-analysis 06):
  §1 "压缩 KV-cache 的核心思想" (latent cache Lc + shared rotated key Rc),
  §2 "attention 的数据流" (dims qh, kvb_dim, Tk = pos_base + S),
  §2.1 (interleaved partial RoPE ``rope_interleave`` on the qk_rope tail),
  §2.2 "DSA lightning indexer" (ReLU-gated head-weighted scores, causal
  top-2048 keys, the keep-all check),
  §2.3 "两条注意力路径：吸收 vs 非吸收" (absorbed decode via qabs and clat;
  non-absorbed prefill via one kv_b GEMM).
* [FDSA] the page "第 7 章 · 03 token 精确前向验证与 faithful DSA", §二 (the
  indexer key cache Ic holds index_hd fp32 values per token).

Every function takes numpy arrays, widens them to float64 and computes the
plain definition; none of them blocks, fuses or reorders beyond what the
definition states.  Readings of points the pages leave open are stated in
each docstring.

Parity status of each function (what pins it, see tests/test_oracle_pins.py):

* rope_interleave       - complex-multiply brute force, textbook cos/sin values,
                          pos=0 identity, relative-position invariance.
* attend_dense          - brute-force Python loops; T=1 and uniform closed forms;
                          hand-derived two-token example.
* attend_absorbed       - equals attend_dense (associativity, [MLA-KV] §2.3).
* prefill_nonabsorbed   - equals dense decode at every query position.
* index_scores          - hand-worked integer example; brute-force loops.
* topk_select           - brute-force full sort with the (score desc, index asc)
                          comparator; keep-all; -0.0 == +0.0 tie case.
* sparse_decode         - keep-all equals dense; a subset equals dense attention
                          over the gathered rows.
* rms_norm, layer_norm  - constant-vector closed forms, unit mean/variance of the
                          normalised values, hand-worked examples.
* cache_append,         - composed of the pinned norms and rope_interleave; rows
  index_key_append        land at pos = T[b] - S + s.
* page_row, unpage      - hand-worked block table; identity table equals the
                          contiguous layout.
* o_proj                - hand-worked 2x3 product; one-hot rows pick columns.
* e4m3_decode,          - textbook values of the format (1.0, 448, 2^-9, 2^-6,
  e4m3_encode             NaN codes); all 256 codes against torch's float8_e4m3fn;
                          ties-to-even and saturation by hand; encode(decode(c)) = c.
* dequant_latent,       - composed of the pinned e4m3 functions and cache_append;
  cache_append_fp8        codes within half a quantum of the normalised row.
"""
from .mla import (  # noqa: F401
    e4m3_decode,
    e4m3_encode,
    dequant_latent,
    cache_append_fp8,
    o_proj,
    page_row,
    unpage,
    rms_norm,
    layer_norm,
    new_token_positions,
    cache_append,
    index_key_append,
    rope_interleave,
    split_kv_b,
    attend_dense,
    attend_absorbed,
    softmax_probs,
    decode_dense,
    decode_absorbed,
    prefill_nonabsorbed,
    index_scores,
    topk_select,
    sparse_decode,
    query_positions,
)
