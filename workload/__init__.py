"""Seeded synthetic inputs for the MLA latent-KV hot path.

This module draws random tensors and nothing else: it holds none of the
method's arithmetic (no RoPE, no projection, no softmax).  Both the CUDA path
(tests, bench) and the CPU oracle (tests) receive the tensors made here, so it
is the one piece of code they share.

Workloads follow the shapes of the GLM-5.2 model described on the page
"MLA 注意力与 KV 缓存" (colibri-analysis 06), §1 (64 heads, a 512-wide latent
plus a 64-wide shared rotated key per token) and §2 (the dimensions qk_nope,
qk_rope, kv_lora, v_head of ``attention``).  Value distributions:

* tiny fp32 case: every tensor ~ N(0,1)/sqrt(fan_in), fan_in being the tensor's
  innermost dimension; DSA tensors are integers in [-4, 4] stored as fp32.
* GLM-shaped cases: Lc, Rc and q ~ N(0,1), kv_b ~ N(0, 0.02), rounded to bf16;
  DSA tensors (Ic, q_idx, w) are integers in [-4, 4] stored as fp32, so that
  every index score is an exactly representable integer.

Large tensors are drawn on the device they live on from a seeded
``torch.Generator``; small metadata (sequence lengths) always comes from a CPU
generator so that it does not depend on the device.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import torch

SEED_BASE = 0x4D4C41  # per-workload seed = SEED_BASE + workload index


@dataclasses.dataclass(frozen=True)
class Dims:
    """MLA head geometry (names follow the page's ``attention`` dimensions)."""

    H: int
    qk_nope: int
    qk_rope: int
    kv_lora: int
    v_head: int
    rope_base: float = 10000.0
    scale: Optional[float] = None  # None -> 1/sqrt(qk_nope + qk_rope)

    @property
    def qk_head(self) -> int:
        return self.qk_nope + self.qk_rope

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.qk_head)


TINY = Dims(H=4, qk_nope=16, qk_rope=8, kv_lora=32, v_head=16)
GLM = Dims(H=64, qk_nope=192, qk_rope=64, kv_lora=512, v_head=256)

# Named workloads: sizes only.  Index i uses seed SEED_BASE + i.
WORKLOADS = {
    "tiny": dict(index=0, dims=TINY, B=1, S=1, T=64, dtype="f32",
                 dsa=dict(n_ih=2, index_hd=8, topk=16)),
    "glm_decode_t4096": dict(index=1, dims=GLM, B=1, S=1, T=4096, dtype="bf16"),
    "glm_batched_b32": dict(index=2, dims=GLM, B=32, S=(1, 6), T_lo=1024, T_hi=32768,
                            T_cap=32768, dtype="bf16"),
    "glm_dsa_t65536": dict(index=3, dims=GLM, B=4, S=1, T=65536, dtype="bf16",
                           dsa=dict(n_ih=32, index_hd=128, topk=2048)),
    "glm_prefill_s2048": dict(index=4, dims=GLM, B=1, S=2048, pos_base=8192, dtype="bf16"),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g, device, dtype):
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def _small_ints(shape, g, device, lo=-4, hi=4):
    return torch.randint(lo, hi + 1, tuple(shape), generator=g, device=device,
                         dtype=torch.int32).to(torch.float32)


def seq_lengths(B: int, lo: int, hi: int, seed: int) -> List[int]:
    """Per-sequence cached lengths drawn uniformly from {lo, ..., hi} (CPU generator)."""
    g = _gen(seed, "cpu")
    return torch.randint(lo, hi + 1, (B,), generator=g).tolist()


def mla_inputs(dims: Dims, B: int, S: int, T: Sequence[int], T_cap: int, dtype: str,
               seed: int, device="cpu", tiny_scaling: Optional[bool] = None) -> Dict[str, torch.Tensor]:
    """Latent cache, query and kv_b for one MLA call.

    Returns ``q [B,S,H,qk_nope+qk_rope]`` (pre-RoPE), ``Lc [B,T_cap,kv_lora]``,
    ``Rc [B,T_cap,qk_rope]`` (keys already rotated, as stored by the cache
    writer), ``kv_b [H, qk_nope+v_head, kv_lora]`` (per head: the qk_nope rows
    of W_UK, then the v_head rows of W_UV) and ``T [B]`` int32.
    Rows of the cache at positions >= T[b] are filled with NaN so that a kernel
    that reads past a sequence's end is caught by the comparison.
    """
    assert len(T) == B and all(S <= t <= T_cap for t in T)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    if tiny_scaling is None:
        tiny_scaling = dtype == "f32"
    g = _gen(seed, device)
    H, Dq, Dl, Dr = dims.H, dims.qk_head, dims.kv_lora, dims.qk_rope
    Dkv = dims.qk_nope + dims.v_head
    if tiny_scaling:
        s_q, s_l, s_r, s_w = (1 / math.sqrt(Dq), 1 / math.sqrt(Dl), 1 / math.sqrt(Dr),
                              1 / math.sqrt(Dl))
    else:
        s_q, s_l, s_r, s_w = 1.0, 1.0, 1.0, 0.02
    q = _normal((B, S, H, Dq), s_q, g, device, tdt)
    Lc = _normal((B, T_cap, Dl), s_l, g, device, tdt)
    Rc = _normal((B, T_cap, Dr), s_r, g, device, tdt)
    kv_b = _normal((H, Dkv, Dl), s_w, g, device, tdt)
    for b, t in enumerate(T):
        if t < T_cap:
            Lc[b, t:] = float("nan")
            Rc[b, t:] = float("nan")
    Tt = torch.tensor(list(T), dtype=torch.int32, device=device)
    return dict(q=q, Lc=Lc, Rc=Rc, kv_b=kv_b, T=Tt)


E4M3_NAN = 0x7F  # the positive NaN code of the FP8 format


def fp8_latent_codes(B: int, T: Sequence[int], T_cap: int, kv_lora: int, seed: int, device="cpu") -> torch.Tensor:
    """A synthetic FP8 latent cache ``[B, T_cap, kv_lora]`` uint8: random E4M3
    bit patterns (uniform sign, exponent field 4..11, uniform mantissa), i.e.
    magnitudes 2^-3 .. 2^4 * 1.875 before the cache scale.  Rows at positions
    >= T[b] hold the NaN code, so that a kernel reading past a sequence's end
    is caught."""
    g = _gen(seed + 0x3000, device)
    shape = (B, T_cap, kv_lora)
    sign = torch.randint(0, 2, shape, generator=g, device=device, dtype=torch.int32) << 7
    expo = torch.randint(4, 12, shape, generator=g, device=device, dtype=torch.int32) << 3
    mant = torch.randint(0, 8, shape, generator=g, device=device, dtype=torch.int32)
    codes = (sign | expo | mant).to(torch.uint8)
    for b, t in enumerate(T):
        if t < T_cap:
            codes[b, t:] = E4M3_NAN
    return codes


def dsa_inputs(B: int, S: int, T: Sequence[int], T_cap: int, n_ih: int, index_hd: int,
               seed: int, device="cpu") -> Dict[str, torch.Tensor]:
    """Indexer query ``q_idx [B,S,n_ih,index_hd]``, head weights ``w [B,S,n_ih]``
    and indexer keys ``Ic [B,T_cap,index_hd]``: integers in [-4, 4] as fp32.
    Key rows at positions >= T[b] are NaN (never read by a correct kernel)."""
    g = _gen(seed + 0x1000, device)
    q_idx = _small_ints((B, S, n_ih, index_hd), g, device)
    w = _small_ints((B, S, n_ih), g, device)
    Ic = _small_ints((B, T_cap, index_hd), g, device)
    for b, t in enumerate(T):
        if t < T_cap:
            Ic[b, t:] = float("nan")
    return dict(q_idx=q_idx, w=w, Ic=Ic)


def append_inputs(dims: Dims, B: int, S: int, dtype: str, seed: int, device="cpu",
                  index_hd: int = 0) -> Dict[str, torch.Tensor]:
    """Inputs of the cache writers for S new tokens per sequence.

    ``comp [B,S,kv_lora+qk_rope]`` (the kv_a projection of each new token) and
    ``kv_a_ln [kv_lora]`` (gain around 1) in ``dtype``; with ``index_hd > 0``
    also the fp32 indexer keys ``k_idx [B,S,index_hd]`` (mean 0.3, so the
    LayerNorm centring matters) with ``ln_w`` and ``ln_b [index_hd]``."""
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    g = _gen(seed + 0x2000, device)
    comp = _normal((B, S, dims.kv_lora + dims.qk_rope), 1.0, g, device, tdt)
    kv_a_ln = (1.0 + _normal((dims.kv_lora,), 0.1, g, device, torch.float32)).to(tdt)
    out = dict(comp=comp, kv_a_ln=kv_a_ln)
    if index_hd > 0:
        out["k_idx"] = 0.3 + _normal((B, S, index_hd), 1.0, g, device, torch.float32)
        out["ln_w"] = 1.0 + _normal((index_hd,), 0.1, g, device, torch.float32)
        out["ln_b"] = _normal((index_hd,), 0.1, g, device, torch.float32)
    return out


def paged_layout(T: Sequence[int], page_size: int, seed: int, spare_pages: int = 3):
    """A shuffled page assignment for sequences of lengths T: returns
    ``(block_table [B, max_pages] int32, num_pages)``.  Sequence b owns
    ceil(T[b] / page_size) pages, drawn from a seeded permutation of the pool
    (which has ``spare_pages`` unused pages); table entries past a sequence's
    last page are -1."""
    need = [(t + page_size - 1) // page_size for t in T]
    max_pages = max(need)
    num_pages = sum(need) + spare_pages
    g = _gen(seed + 0x3000, "cpu")
    perm = torch.randperm(num_pages, generator=g).tolist()
    table = torch.full((len(T), max_pages), -1, dtype=torch.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = torch.tensor(perm[k:k + n], dtype=torch.int32)
        k += n
    return table, num_pages


def to_pages(cache, block_table, T: Sequence[int], page_size: int, num_pages: int, fill=float("nan")):
    """Copies rows 0..T[b]-1 of a contiguous cache [B, T_cap, D] into a pool
    [num_pages, page_size, D] at the rows the block table names; every other
    pool row holds ``fill``."""
    D = cache.shape[2]
    pool = torch.full((num_pages * page_size, D), fill, dtype=cache.dtype, device=cache.device)
    tbl = block_table.tolist()
    for b, n in enumerate(T):
        for i in range((n + page_size - 1) // page_size):
            lo, hi = i * page_size, min(n, (i + 1) * page_size)
            r0 = tbl[b][i] * page_size
            pool[r0:r0 + hi - lo] = cache[b, lo:hi]
    return pool.view(num_pages, page_size, D)


def workload_inputs(name: str, device="cpu", S: Optional[int] = None) -> Dict[str, object]:
    """All inputs of a named workload (see ``WORKLOADS``)."""
    wl = WORKLOADS[name]
    seed = SEED_BASE + wl["index"]
    dims: Dims = wl["dims"]
    B = wl["B"]
    if name == "glm_batched_b32":
        S = S if S is not None else 1
        T = seq_lengths(B, wl["T_lo"], wl["T_hi"], seed)
        T_cap = wl["T_cap"]
    elif name == "glm_prefill_s2048":
        S = wl["S"]
        T = [wl["pos_base"] + S] * B
        T_cap = T[0]
    else:
        S = wl["S"]
        T = [wl["T"]] * B
        T_cap = wl["T"]
    out: Dict[str, object] = dict(dims=dims, B=B, S=S, T_list=T, T_cap=T_cap, dtype=wl["dtype"])
    out.update(mla_inputs(dims, B, S, T, T_cap, wl["dtype"], seed, device))
    if "dsa" in wl:
        d = wl["dsa"]
        out.update(dsa_inputs(B, S, T, T_cap, d["n_ih"], d["index_hd"], seed, device))
        out["topk"] = d["topk"]
    if "pos_base" in wl:
        out["pos_base"] = wl["pos_base"]
    return out
