"""Benchmark of the MLA latent-KV hot path on GB300 (one JSON line on rank 0).

Headline workload: GLM-5.2-shaped single-sequence absorbed decode, B=1, S=1,
T=4096 (bf16 cache, fp32 accumulate).  One step = one mla_decode_absorbed
call (query RoPE, absorb through W_UK, scores over Lc/Rc, softmax, latent
context, W_UV lift).

Timing protocol: one step's inputs (34 MB at T=4096) fit in the 129 MB L2,
so the bench keeps C copies of every input, C * step bytes >= 4 x L2, and
step i reads copy i mod C: each step's cache, weights and query come from
HBM, as in a decode that runs layer after layer with each layer's own
weights and cache.  The K timed steps are one CUDA graph replayed once
between two CUDA events (per step = total / K).  Two more figures come with
every line: each step timed alone after a 256 MiB L2 flush write (which also
evicts the kernels' instructions, and adds the graph-launch overhead to every
step), and K back-to-back steps on one copy (warm L2).  A second,
instrumented replay records CUDA events between the library's kernels
(mla_set_kernel_events) to attribute time per kernel, and the roofline object
describes the dominant kernel.

The default run also measures the other workloads of the hot path ("rows"):
batched decode B=32 with S=1 and S=6, DSA (indexer + top-2048 + sparse
decode) at B=4, T=65536, the non-absorbed prefill S=2048 at pos_base=8192 and
the cache writers (latent + indexer key rows of 32 x 6 new tokens) and the
batched decode over a shuffled 128-row page pool, plus the T sweep 4k..64k of
the headline metric.

Multi-GPU (torchrun): replicas -- every rank runs the same workload on its own
GPU with no collective on the data path; value = all ranks' tokens / the
slowest rank's time (weak scaling).

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode tokens/s and latent-cache HBM GB/s (% roofline) at T=4k–64k, 1 GB300"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20
ROTATE_BYTES = 4 * L2_BYTES  # input copies cycled so that a step never finds its inputs in L2
COPIES_MEM_BYTES = 24 << 30  # device memory the input copies of one workload may take
ROW_WORKLOADS = ("glm_batched_b32_s1", "glm_batched_b32_s6", "glm_dsa_t65536", "glm_prefill_s2048",
                 "glm_append_b32_s6", "glm_paged_b32_s1", "glm_dsa_t65536_l4", "glm_decode_oproj_t4096",
                 "glm_batched_b32_s1_fp8", "glm_decode_t4096_fp8", "glm_decode_t65536_fp8", "glm_dsa_t65536_l4_oproj")
OPROJ_HIDDEN = 6144  # model width of the projection row: a size chosen here, the pages print none
FP8_LAT_SCALE = 0.05  # scale of the synthetic FP8 latent cache (codes of magnitude 2^-3 .. 30)
APPEND_RMS_EPS = 1e-6
# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of a
# workload's dominant kernel, from one ncu capture of that kernel on this
# workload, with the digest (kernel_digest()) of the sources that kernel was
# built from.  An entry whose sources have changed since is stale, and the
# roofline reports its traffic as null.
NCU_TRAFFIC = {
    ("glm_decode_t4096", "attention"): (4891904, "b5c89e90e54c811b"),
    ("glm_decode_t16384", "attention"): (19051264, "b5c89e90e54c811b"),
    ("glm_decode_t65536", "attention"): (77918720, "b5c89e90e54c811b"),
    ("glm_batched_b32_s1", "attention"): (582998784, "b5c89e90e54c811b"),
    ("glm_batched_b32_s6", "attention"): (622450176, "b5c89e90e54c811b"),
    ("glm_paged_b32_s1", "attention"): (582960640, "b5c89e90e54c811b"),
    ("glm_dsa_t65536", "index_scores"): (139196928, "d8d0b28c3c50688c"),
    ("glm_dsa_t65536_l4", "attention"): (9864448, "b5c89e90e54c811b"),
    ("glm_prefill_s2048", "flash_attention"): (797446912, "f81080760d23a01a"),
    ("glm_append_b32_s6", "cache_append"): (243200, "cce2f582d5b0591c"),
    ("glm_append_b32_s6", "index_key_append"): (115968, "cce2f582d5b0591c"),
    ("glm_batched_b32_s1_fp8", "attention"): (325867520, "b5c89e90e54c811b"),
    ("glm_decode_t4096_fp8", "attention"): (2937088, "b5c89e90e54c811b"),
    ("glm_decode_t65536_fp8", "attention"): (42172416, "b5c89e90e54c811b"),
    ("glm_decode_oproj_t4096", "oproj_gemv"): (205005312, "1888d6993a2c0d56"),
    ("glm_dsa_t65536_l4_oproj", "oproj_gemv"): (204694528, "1888d6993a2c0d56"),
}
# Library sources each timed kernel is built from, besides the shared headers.
KERNEL_SOURCES = {
    "attention": ("decode_tc.cu", "attn_core.cuh"), "absorb": ("decode_tc.cu",), "combine": ("decode_tc.cu",),
    "merge": ("decode_tc.cu",), "plan_rope": ("decode_tc.cu",), "quant_q": ("decode_tc.cu",),
    "gather": ("decode_tc.cu",), "absorb_gemm": ("gemm_tc.cu",), "up_gemm": ("gemm_tc.cu",),
    "index_scores": ("index_tc.cu", "dsa.cu"), "topk_select": ("dsa.cu",), "kv_gemm": ("gemm_tc.cu",),
    "flash_attention": ("prefill_tc.cu",), "cache_append": ("cache_append.cu",),
    "index_key_append": ("cache_append.cu",), "oproj_gemv": ("oproj.cu",),
}
SHARED_SOURCES = ("common.cuh", "sm100.cuh", "internal.h", "tmap.h", "decode_tc.h", "gemm_tc.h")


def kernel_digest(kernel):
    """sha256 (first 16 hex digits) of the library sources a kernel is built from."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_latent_kv_06_gb300", "csrc")
    for f in sorted(set(SHARED_SOURCES + KERNEL_SOURCES.get(kernel, ()))):
        path = os.path.join(csrc, f)
        if os.path.exists(path):
            h.update(f.encode())
            with open(path, "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(name, kernel):
    entry = NCU_TRAFFIC.get((name, kernel))
    if entry is None or kernel not in KERNEL_SOURCES or entry[1] != kernel_digest(kernel):
        return None
    return entry[0]


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            return json.load(f), "measured"
    except OSError:
        return FALLBACK, "fallback"


# ------------------------------------------------------------------ workloads
def build_workload(name, device):
    """Inputs, the step as a list of API calls, and per-kernel algorithmic work."""
    import torch
    import mla_latent_kv_06_gb300 as mla
    from workload import GLM, mla_inputs, workload_inputs, SEED_BASE

    fp8 = name.endswith("_fp8")  # the same workload over the FP8 latent cache
    if fp8:
        name = name[:-len("_fp8")]
    if name.startswith("glm_decode_t"):
        T = int(name[len("glm_decode_t"):])
        if name == "glm_decode_t4096":
            x = workload_inputs(name, device)
        else:
            x = dict(dims=GLM, B=1, S=1, T_list=[T], T_cap=T, dtype="bf16")
            x.update(mla_inputs(GLM, 1, 1, [T], T, "bf16", SEED_BASE + 1, device))
        kind = "decode"
    elif name.startswith("glm_batched_b32_s"):
        x = workload_inputs("glm_batched_b32", device, S=int(name[len("glm_batched_b32_s"):]))
        kind = "decode"
    elif name in ("glm_dsa_t65536", "glm_dsa_t65536_l4", "glm_dsa_t65536_l4_oproj"):
        x = workload_inputs("glm_dsa_t65536", device)
        x["layers"] = [x]
        if name.endswith("_oproj"):  # each layer's output projection too
            g = torch.Generator(device=device)
            g.manual_seed(SEED_BASE + 9)
            x["w_o"] = [(torch.randn(OPROJ_HIDDEN, 64 * 256, generator=g, device=device) * 0.02).to(torch.bfloat16)
                        for _ in range(4)]
        if "_l4" in name:  # three more layers reuse the first layer's selection
            for layer in range(1, 4):
                y = mla_inputs(x["dims"], x["B"], x["S"], x["T_list"], x["T_cap"], "bf16", SEED_BASE + 10 + layer,
                               device)
                x["layers"].append(y)
        kind = "dsa"
    elif name == "glm_prefill_s2048":
        x = workload_inputs(name, device)
        kind = "prefill"
    elif name == "glm_append_b32_s6":
        x = workload_inputs("glm_batched_b32", device, S=6)
        kind = "append"
    elif name == "glm_decode_oproj_t4096":
        x = workload_inputs("glm_decode_t4096", device)
        g = torch.Generator(device=device)
        g.manual_seed(SEED_BASE + 7)
        x["w_o"] = (torch.randn(OPROJ_HIDDEN, 64 * 256, generator=g, device=device) * 0.02).to(torch.bfloat16)
        kind = "decode_oproj"
    elif name == "glm_paged_b32_s1":
        from workload import paged_layout, to_pages
        x = workload_inputs("glm_batched_b32", device, S=1)
        table, num_pages = paged_layout(x["T_list"], 128, SEED_BASE + 6)
        x["table"] = table.to(device)
        x["Lc"] = to_pages(x["Lc"], table, x["T_list"], 128, num_pages)
        x["Rc"] = to_pages(x["Rc"], table, x["T_list"], 128, num_pages)
        kind = "decode"
    else:
        raise SystemExit(f"unknown workload {name}")

    d = x["dims"]
    B, S = x["B"], x["S"]
    R = B * S
    T_list = x["T_list"]
    row = 2 * (d.kv_lora + d.qk_rope)                      # latent-cache bytes per key
    if fp8:
        from workload import fp8_latent_codes
        assert kind == "decode" and "table" not in x
        x["Lc8"] = fp8_latent_codes(B, T_list, x["T_cap"], d.kv_lora, SEED_BASE + 8, device)
        del x["Lc"]
        row = d.kv_lora + 2 * d.qk_rope                    # E4M3 latent, bf16 rope key
    w_uk = 2 * d.H * d.qk_nope * d.kv_lora
    w_uv = 2 * d.H * d.v_head * d.kv_lora
    q_bytes = 2 * R * d.H * d.qk_head
    out_bytes = 4 * R * d.H * d.v_head
    qcat = 2 * R * d.H * (d.kv_lora + d.qk_rope)
    out = torch.empty(B, S, d.H, d.v_head, dtype=torch.float32, device=device)
    info = {"tokens": R, "B": B, "S": S, "T_list": T_list}

    if kind == "decode" and "table" in x:  # shuffled 128-row pages of one pool
        need = mla.lib().mla_decode_paged_workspace_size(mla.ctypes.byref(mla.make_dims(d)), mla.MLA_BF16, B, S,
                                                         x["table"].shape[1], 128)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
        calls = [lambda: mla.decode_paged(x["q"], x["Lc"], x["Rc"], x["table"], x["T"], x["kv_b"], d, out=out,
                                          workspace=ws)]
    elif kind == "decode" and fp8:
        need = mla.lib().mla_decode_fp8_workspace_size(mla.ctypes.byref(mla.make_dims(d)), B, S, x["T_cap"])
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
        calls = [lambda: mla.decode_fp8(x["q"], x["Lc8"], x["Rc"], x["T"], x["kv_b"], d, FP8_LAT_SCALE, out=out,
                                        workspace=ws)]
    elif kind == "decode":
        need = mla.decode_workspace_size(d, mla.MLA_BF16, B, S, x["T_cap"])
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
        calls = [lambda: mla.decode_absorbed(x["q"], x["Lc"], x["Rc"], x["T"], x["kv_b"], d, out=out, workspace=ws)]
    if kind == "decode":
        cache = row * sum(T_list)  # every cached key read once per sequence
        info.update(cache_bytes=cache, alg_bytes=cache + w_uk + w_uv + q_bytes + out_bytes)
        clat = 2 * R * d.H * d.kv_lora
        # S > 1: every key tile serves S query tokens, so the attention is bound by the tensor pipe
        pairs = sum(S * t - S * (S - 1) // 2 for t in T_list)
        attn_flops = 2 * d.H * (d.kv_lora + d.qk_rope + d.kv_lora) * pairs
        if S > 1:
            info["flops"] = attn_flops
        work = {"absorb": ("hbm", w_uk + q_bytes), "absorb_gemm": ("hbm", w_uk + q_bytes + qcat),
                "plan_rope": ("hbm", q_bytes),
                "attention": ("tensor", attn_flops) if S > 1 else ("hbm", cache + qcat),
                "combine": ("hbm", w_uv + out_bytes), "merge": ("hbm", clat),
                "up_gemm": ("hbm", w_uv + clat + out_bytes)}
        if fp8:
            e2e = dict(inputs=[x["q"], x["T"]], run=lambda q, T: mla.decode_fp8(
                q, x["Lc8"], x["Rc"], T, x["kv_b"], d, FP8_LAT_SCALE, out=out, workspace=ws), out=out)
        else:
            e2e = None if "table" in x else dict(inputs=[x["q"], x["T"]], run=lambda q, T: mla.decode_absorbed(
                q, x["Lc"], x["Rc"], T, x["kv_b"], d, out=out, workspace=ws), out=out)
    elif kind == "dsa":
        k = x["topk"]
        T_cap = x["T_cap"]
        sc = torch.empty(B, S, T_cap, dtype=torch.float32, device=device)
        sel = torch.empty(B, S, k, dtype=torch.int32, device=device)
        nsel = torch.empty(B, S, dtype=torch.int32, device=device)
        hidden = OPROJ_HIDDEN if "w_o" in x else 0
        need = mla.lib().mla_sparse_decode_layers_workspace_size(mla.ctypes.byref(mla.make_dims(d)), mla.MLA_BF16,
                                                                 B, S, k, hidden)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
        L = len(x["layers"])
        outs = [out] + [torch.empty_like(out) for _ in range(L - 1)]
        sws = torch.empty(max(mla.lib().dsa_select_workspace_size(B, S, x["q_idx"].shape[2], x["q_idx"].shape[3],
                                                                  T_cap, k), 1), dtype=torch.uint8, device=device)
        calls = [lambda: mla.select(x["q_idx"], x["w"], x["Ic"], x["T"], k, scores=sc, sel=sel, nsel=nsel,
                                    workspace=sws)]
        if L == 1:
            calls.append(lambda: mla.sparse_decode(x["q"], x["Lc"], x["Rc"], x["T"], x["kv_b"], sel, nsel, d, out=out,
                                                   workspace=ws))
        else:  # one call for the layers that share the selection
            layers = [(y["q"], y["Lc"], y["Rc"], y["kv_b"]) for y in x["layers"]]
            ys = [torch.empty(R, hidden, dtype=torch.float32, device=device) for _ in range(L)] if hidden else None
            calls.append(lambda: mla.sparse_decode_layers(layers, x["T"], sel, nsel, d, outs=outs, w_o=x.get("w_o"),
                                                          ys=ys, workspace=ws))
        info["tokens"] = R * L  # one query token per layer
        ic = 4 * x["Ic"].shape[2] * sum(T_list)
        scores = 4 * R * T_cap
        gathered = row * R * k
        clat = 2 * R * d.H * d.kv_lora
        proj = (2 * hidden * d.H * d.v_head + out_bytes + 4 * R * hidden) if hidden else 0  # W_O, x, y per layer
        info.update(cache_bytes=gathered * L,
                    alg_bytes=ic + 2 * scores + L * (gathered + w_uk + w_uv + q_bytes + out_bytes + proj))
        work = {"index_scores": ("hbm", ic + scores), "topk_select": ("hbm", scores + 4 * R * k),
                "gather": ("hbm", 2 * gathered), "absorb": ("hbm", w_uk + q_bytes),
                "attention": ("hbm", gathered + qcat), "combine": ("hbm", w_uv + out_bytes),
                "absorb_gemm": ("hbm", w_uk + q_bytes + qcat), "plan_rope": ("hbm", q_bytes),
                "merge": ("hbm", clat), "up_gemm": ("hbm", w_uv + clat + out_bytes), "oproj_gemv": ("hbm", proj)}
        e2e = None
    elif kind == "decode_oproj":
        need = mla.lib().mla_decode_oproj_workspace_size(mla.ctypes.byref(mla.make_dims(d)), mla.MLA_BF16, B, S,
                                                          x["T_cap"], OPROJ_HIDDEN)
        ws = torch.empty(need, dtype=torch.uint8, device=device)
        y = torch.empty(B, S, OPROJ_HIDDEN, dtype=torch.float32, device=device)
        calls = [lambda: mla.decode_oproj(x["q"], x["Lc"], x["Rc"], x["T"], x["kv_b"], x["w_o"], d, y=y,
                                          workspace=ws)]
        cache = row * sum(T_list)
        w_o = 2 * OPROJ_HIDDEN * d.H * d.v_head
        info.update(cache_bytes=cache, alg_bytes=cache + w_uk + w_uv + w_o + q_bytes + out_bytes + 4 * R * OPROJ_HIDDEN)
        work = {"absorb": ("hbm", w_uk + q_bytes), "attention": ("hbm", cache + qcat),
                "combine": ("hbm", w_uv + out_bytes), "oproj_gemv": ("hbm", w_o + out_bytes + 4 * R * OPROJ_HIDDEN)}
        e2e = None
    elif kind == "append":
        from workload import append_inputs
        hd, rope_dim = 128, d.qk_rope
        a = append_inputs(d, B, S, "bf16", SEED_BASE + 5, device, index_hd=hd)
        Ic = torch.zeros(B, x["T_cap"], hd, dtype=torch.float32, device=device)
        calls = [lambda: mla.cache_append(a["comp"], a["kv_a_ln"], x["T"], x["Lc"], x["Rc"], d, APPEND_RMS_EPS),
                 lambda: mla.index_key_append(a["k_idx"], a["ln_w"], a["ln_b"], x["T"], Ic, rope_dim)]
        kv_rows = 2 * 2 * R * (d.kv_lora + d.qk_rope) + 2 * d.kv_lora  # comp read, Lc/Rc rows written, kv_a_ln
        ic_rows = 2 * 4 * R * hd + 2 * 4 * hd                          # k_idx read, Ic rows written, ln_w/ln_b
        info.update(cache_bytes=R * (row + 4 * hd), alg_bytes=kv_rows + ic_rows)
        work = {"cache_append": ("hbm", kv_rows), "index_key_append": ("hbm", ic_rows)}
        e2e = None
    else:
        pos_base = x["pos_base"]
        need = mla.lib().mla_prefill_naive_workspace_size(mla.ctypes.byref(mla.make_dims(d)), mla.MLA_BF16, B, S,
                                                           pos_base)
        ws = torch.empty(need, dtype=torch.uint8, device=device)
        calls = [lambda: mla.prefill_naive(x["q"], x["Lc"], x["Rc"], x["kv_b"], d, pos_base, out=out, workspace=ws)]
        Tk = pos_base + S
        pairs = sum(pos_base + s + 1 for s in range(S))
        gemm_flops = 2 * B * Tk * d.kv_lora * d.H * (d.qk_nope + d.v_head)
        attn_flops = 2 * B * d.H * pairs * (d.qk_head + d.v_head)
        info.update(cache_bytes=row * Tk, alg_bytes=row * Tk + w_uk + w_uv + q_bytes + out_bytes,
                    flops=gemm_flops + attn_flops)
        work = {"kv_gemm": ("tensor", gemm_flops), "flash_attention": ("tensor", attn_flops)}
        e2e = dict(inputs=[x["q"]], run=lambda q: mla.prefill_naive(q, x["Lc"], x["Rc"], x["kv_b"], d, pos_base,
                                                                     out=out, workspace=ws), out=out)
    return x, calls, info, work, e2e


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except OSError:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ timing
def capture(calls, stream):
    """A CUDA graph of the step's API calls (the library's launches, PDL edges included)."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in calls:
            c()
    torch.cuda.synchronize()
    return g


def time_steps(step, K, W, flush, stream):
    """Device time (ms) of K steps, each timed alone after an L2 flush that is not timed."""
    import torch
    for _ in range(W):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def time_graph(steps, W, stream):
    """Device time (ms) of one replay of a CUDA graph holding the given steps
    back to back, after W untimed steps (a graph of the first W)."""
    import torch
    warm = capture([c for st in steps[:W] for c in st], stream)
    timed = capture([c for st in steps for c in st], stream)
    warm.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    timed.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def kernel_times(steps, K, stream):
    """Per-kernel device time (us, mean per launch) from events the library
    records around its launches, over K replays of a graph of `steps` (which
    cycle through the input copies), and launches per step."""
    import torch
    import mla_latent_kv_06_gb300 as mla
    calls = [c for st in steps for c in st]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(40)] for _ in calls]  # up to 39 launches a call
    for ev in evs:  # create the CUDA events before the capture
        for e in ev:
            e.record(stream)
    torch.cuda.synchronize()
    names = []
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c, ev in zip(calls, evs):
            mla.set_kernel_events(ev)
            c()
            names.append(mla.last_launch_names())
    mla.set_kernel_events(None)
    torch.cuda.synchronize()
    acc = {}
    for _ in range(K):
        g.replay()
        torch.cuda.synchronize()
        for nm, ev in zip(names, evs):
            for i, n in enumerate(nm):
                acc.setdefault(n, []).append(ev[i].elapsed_time(ev[i + 1]) * 1e3)
    counts = {}
    for nm in names:
        for n in nm:
            counts[n] = counts.get(n, 0) + 1
    counts = {n: v // len(steps) for n, v in counts.items()}
    return {n: statistics.mean(v) for n, v in acc.items()}, counts


def time_e2e(e2e_sets, K, W, stream):
    """Public-API call with host buffers, K steps back to back in one graph:
    every step copies its inputs from pinned host memory (one staging buffer,
    each input at a 256-byte offset, so one host-to-device copy), calls the
    library on input copy i mod C, and copies the output back to pinned host
    memory."""
    import torch
    e2e = e2e_sets[0]
    ins = [t.detach().cpu().contiguous() for t in e2e["inputs"]]
    offs, total = [], 0
    for t in ins:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev = torch.empty(total, dtype=torch.uint8, device=e2e["out"].device)
    dev_in = []
    for t, o in zip(ins, offs):
        nb = t.numel() * t.element_size()
        host[o:o + nb].copy_(t.reshape(-1).view(torch.uint8))
        dev_in.append(dev[o:o + nb].view(t.dtype).view(t.shape))
    host_out = torch.empty(e2e["out"].shape, dtype=e2e["out"].dtype).pin_memory()
    d2h = host_out.numel() * host_out.element_size()

    def one(es):
        def f():
            dev.copy_(host, non_blocking=True)
            es["run"](*dev_in)
            host_out.copy_(es["out"], non_blocking=True)
        return [f]

    steps = [one(e2e_sets[i % len(e2e_sets)]) for i in range(K)]
    return time_graph(steps, W, stream), total, d2h


def roofline(name, work, ktimes, counts, pk, pk_kind):
    """Roofline of the kernel with the largest share of the step (ktimes: mean
    us per launch; counts: launches per step)."""
    share_us = {n: v * counts.get(n, 1) for n, v in ktimes.items()}
    dom = max(share_us, key=share_us.get)
    bound, amount = work.get(dom, ("hbm", 0))
    t = ktimes[dom] * 1e-6
    if bound == "tensor":
        achieved, peak, unit = amount / t / 1e12, pk["bf16_tflops_sustained"], "TFLOP/s"
    else:
        achieved, peak, unit = amount / t / 1e9, pk["hbm_gbs"], "GB/s"
    total = sum(share_us.values())
    return {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "peak_source": pk_kind, "algorithmic_per_launch": amount,
            "kernel_us": ktimes[dom], "traffic": ncu_traffic(name, dom),
            "kernels": {n: {"us": round(v, 2), "launches": counts.get(n, 1), "share": round(share_us[n] / total, 3)}
                        for n, v in ktimes.items()}}


def rotation_copies(step_bytes, copy_bytes):
    """Input copies to cycle through so that the bytes read between two uses of
    one copy exceed 4 x L2, capped so that the copies (copy_bytes of device
    memory each) fit in COPIES_MEM_BYTES."""
    want = max(1, -(-ROTATE_BYTES // max(1, int(step_bytes))))
    return max(1, min(want, COPIES_MEM_BYTES // max(1, int(copy_bytes))))


def measure(name, dev, stream, flush, K, W, pk, pk_kind, want_e2e, extra=True):
    """K steps cycling through C input copies in one graph (the headline
    protocol); with `extra`, also one copy flushed before each step and one
    copy back to back (warm L2)."""
    import torch
    import mla_latent_kv_06_gb300 as mla
    m0 = torch.cuda.memory_allocated(dev)
    sets = [build_workload(name, dev)]
    info, work = sets[0][2], sets[0][3]
    C = rotation_copies(info["alg_bytes"], torch.cuda.memory_allocated(dev) - m0)
    for _ in range(C - 1):
        sets.append(build_workload(name, dev))
    for st in sets:
        for c in st[1]:
            c()
    torch.cuda.synchronize()
    assert mla.device_status() == 0, "device flags raised while warming up"
    total_ms = time_graph([sets[i % C][1] for i in range(K)], W, stream)
    kt, counts = kernel_times([sets[i % C][1] for i in range(max(C, 4))], 5, stream)
    assert mla.device_status() == 0, "device flags raised while timing"
    res = {"total_ms": total_ms, "copies": C, "rotation_bytes": C * info["alg_bytes"], "info": info,
           "ktimes": kt, "counts": counts,
           "roof": roofline(name, work, kt, counts, pk, pk_kind)}
    if extra:
        g = capture(sets[0][1], stream)
        res["flushed_ms"] = statistics.median(time_steps(g.replay, min(K, 20), W, flush, stream))
        res["warm_ms"] = time_graph([sets[0][1]] * K, W, stream) / K
        del g
    if want_e2e and sets[0][4] is not None:
        res["e2e"] = time_e2e([st[4] for st in sets], K, W, stream)
    del sets
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ ranks
def slowest_rank_ms(total_ms, device):
    """Max over the ranks of this job of a timed region (ms), each rank's
    region bracketed by a barrier; the identity for a single process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return total_ms
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def job_throughput(tokens_per_step, steps, world, total_ms):
    """Whole-job rate: every replica processes tokens_per_step per step (weak
    scaling); the job's time is the slowest rank's."""
    return world * tokens_per_step * steps / (total_ms / 1e3)


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(name, budget_s=12.0):
    """Time the fp64 oracle on the host cores on a bounded sample of the workload."""
    import numpy as np
    import oracle
    from workload import GLM, mla_inputs, workload_inputs, SEED_BASE

    if name.startswith("glm_decode_t") and name != "glm_decode_t4096":
        T = int(name[len("glm_decode_t"):])
        x = dict(T_list=[T], S=1)
        x.update(mla_inputs(GLM, 1, 1, [T], T, "bf16", SEED_BASE + 1, "cpu"))
    elif name.startswith("glm_batched_b32_s"):
        x = workload_inputs("glm_batched_b32", "cpu", S=int(name[len("glm_batched_b32_s"):]))
    else:
        x = workload_inputs(name, "cpu")
    f = lambda t: t.float().numpy().astype(np.float64)
    q, Lc, Rc, kvb = (f(x[k]) for k in ("q", "Lc", "Rc", "kv_b"))
    T_list, S = x["T_list"], x["S"]
    rows = [(b, s) for b in range(len(T_list)) for s in range(S)]
    done, t0 = 0, time.perf_counter()
    while True:
        b, s = rows[done % len(rows)]
        pos = T_list[b] - S + s
        if name == "glm_prefill_s2048":
            oracle.prefill_nonabsorbed(q[0], Lc[0], Rc[0], kvb, GLM.qk_nope, GLM.softmax_scale, x["pos_base"],
                                       queries=[done % S])
        else:
            oracle.attend_absorbed(q[b, s], Lc[b, :pos + 1], Rc[b, :pos + 1], kvb, GLM.qk_nope, pos,
                                   GLM.softmax_scale)
        done += 1
        el = time.perf_counter() - t0
        if el > budget_s:
            break
    return done / el, done, el


def host_threads():
    """Threads the oracle's BLAS runs on (all host cores unless limited)."""
    try:
        from threadpoolctl import threadpool_info
        import numpy  # noqa: F401  (loads BLAS)
        n = [dd.get("num_threads") for dd in threadpool_info() if dd.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def host_cpu():
    """Host CPU model (lscpu, else /proc/cpuinfo) and core count (nproc)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                fields = dict(ln.split(":", 1) for ln in f if ":" in ln)
            fields = {k.strip(): v.strip() for k, v in fields.items()}
            model = fields.get("model name") or " ".join(
                f"{k} {fields[k]}" for k in ("CPU implementer", "CPU part") if k in fields) or None
        except OSError:
            pass
    try:
        nproc = int(subprocess.run(["nproc"], capture_output=True, text=True, timeout=10).stdout.strip())
    except (OSError, ValueError, subprocess.SubprocessError):
        nproc = os.cpu_count() or 1
    return {"cpu_model": model, "nproc": nproc}


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mla", "reference"], default="mla")
    ap.add_argument("--workload", default="glm_decode_t4096")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-rows", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args()
    W = max(args.warmup, 3)
    K = args.steps

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        tok_s, n, el = oracle_sample(args.workload, budget_s=min(60.0, max(5.0, 2.0 * K)))
        cores = host_threads()
        hc = host_cpu()
        line = {"impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": K, "warmup": W, "ms_per_step": 1e3 / tok_s, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": args.workload},
                "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "cpu_model": hc["cpu_model"], "nproc": hc["nproc"],
                                 "sample": f"{n} query tokens x 64 heads of {args.workload} in {el:.1f} s"},
                "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    import mla_latent_kv_06_gb300 as mla
    mla.load()
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    pk, pk_kind = peaks()

    with torch.cuda.stream(stream):
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        clocks = ClockSampler(local)
        clocks.start()
        t_wall = time.perf_counter()
        res = measure(args.workload, dev, stream, flush, K, W, pk, pk_kind, want_e2e=True)
        t_wall = time.perf_counter() - t_wall
        clk = clocks.stop()
        total_ms = slowest_rank_ms(res["total_ms"], dev)
        info = res["info"]
        ms_per_step = total_ms / K
        value = job_throughput(info["tokens"], K, world, total_ms)
        step_s = ms_per_step / 1e3
        if rank == 0:
            T_list = info["T_list"]
            line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
                    "warmup": W, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                    "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, GLM-5.2-shaped)",
                    "config": {"workload": args.workload, "B": info["B"], "S": info["S"],
                               "T": T_list if len(T_list) <= 4 else f"sum {sum(T_list)}",
                               "heads": 64, "kv_lora": 512, "qk_rope": 64, "qk_nope": 192, "v_head": 256,
                               "parallelism": f"replicas x{world}",
                               "l2": (f"inputs larger than L2: {res['copies']} copies of every input, step i reads "
                                      f"copy i mod {res['copies']} ({res['rotation_bytes'] / 1e6:.0f} MB read between "
                                      f"two uses of a copy, L2 129 MB)"),
                               "launch": f"one CUDA graph of the {K} timed steps back to back"},
                    "latent_cache_gbs": info["cache_bytes"] / step_s / 1e9,
                    "hbm_gbs_algorithmic": info["alg_bytes"] / step_s / 1e9,
                    "step_frac_of_measured_hbm": info["alg_bytes"] / step_s / 1e9 / pk["hbm_gbs"],
                    "step_frac_of_8tbs": info["alg_bytes"] / step_s / 8e12,
                    "roofline": res["roof"], "clocks": clk,
                    "gpu_launches": sum(res["counts"].values()) * K,
                    "flushed_single_step_ms": res["flushed_ms"], "warm_l2_step_ms": res["warm_ms"],
                    "wall_s_timed_region": t_wall}
            if "e2e" in res:
                ems, h2d, d2h = res["e2e"]
                line["e2e"] = {"value": info["tokens"] * K / (ems / 1e3) * world, "unit": "tokens/s",
                               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ems / K}
            else:
                line["e2e"] = None
            if args.workload == "glm_decode_t4096" and not args.no_sweep:
                sweep = {}
                for T in (4096, 8192, 16384, 32768, 65536):
                    r = measure(f"glm_decode_t{T}", dev, stream, flush, 100, 5, pk, pk_kind, want_e2e=False)
                    t = r["total_ms"] / 100 / 1e3
                    sweep[str(T)] = {"tokens_s": 1 / t, "us": t * 1e6, "copies": r["copies"],
                                     "bytes_between_reuses": r["rotation_bytes"],
                                     "flushed_single_step_us": r["flushed_ms"] * 1e3,
                                     "warm_l2_us": r["warm_ms"] * 1e3,
                                     "latent_cache_gbs": r["info"]["cache_bytes"] / t / 1e9,
                                     "hbm_gbs_algorithmic": r["info"]["alg_bytes"] / t / 1e9,
                                     "frac_of_measured_hbm": r["info"]["alg_bytes"] / t / 1e9 / pk["hbm_gbs"],
                                     "dominant": r["roof"]["kernel"]}
                line["t_sweep"] = sweep
            if args.workload == "glm_decode_t4096" and not args.no_rows:
                rows = {}
                for wl in ROW_WORKLOADS:
                    r = measure(wl, dev, stream, flush, 20, 3, pk, pk_kind, want_e2e=False)
                    t = r["total_ms"] / 20 / 1e3
                    rows[wl] = {"us_per_step": t * 1e6, "tokens_s": r["info"]["tokens"] / t, "copies": r["copies"],
                                "bytes_between_reuses": r["rotation_bytes"],
                                "flushed_single_step_us": r["flushed_ms"] * 1e3, "warm_l2_us": r["warm_ms"] * 1e3,
                                "hbm_gbs_algorithmic": r["info"]["alg_bytes"] / t / 1e9,
                                "roofline": {k: r["roof"][k] for k in ("kernel", "bound", "achieved", "unit", "frac",
                                                                       "traffic", "algorithmic_per_launch",
                                                                       "kernels")}}
                    if "flops" in r["info"]:
                        rows[wl]["tflops"] = r["info"]["flops"] / t / 1e12
                    if wl.endswith("_fp8"):
                        rows[wl]["cache"] = "E4M3 latent codes (one scale), bf16 rope key"
                line["rows"] = rows
            if not args.no_cpu:
                tok_s, n, el = oracle_sample(args.workload)
                hc = host_cpu()
                line["cpu_baseline"] = {"value": tok_s, "unit": "tokens/s", "cores": host_threads(),
                                        "kind": "oracle", "cpu_model": hc["cpu_model"], "nproc": hc["nproc"],
                                        "sample": f"{n} query tokens x 64 heads of {args.workload} in {el:.1f} s"}
            print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
