"""Benchmark of the MLA latent-KV hot path on GB300 (one JSON line on rank 0).

Default workload: GLM-5.2-shaped single-sequence absorbed decode, B=1, S=1,
T=4096 (bf16 cache, fp32 accumulate).  One step = one mla_decode_absorbed
call (query RoPE, absorb through W_UK, scores over Lc/Rc, softmax, latent
context, W_UV lift).  L2 is flushed (256 MiB write) before every timed step,
outside the timed interval, because the step's inputs fit in L2.

Other workloads (--workload): glm_decode_t<T>, glm_batched_b32_s1,
glm_batched_b32_s6, glm_dsa_t65536 (indexer + top-2048 + sparse decode),
glm_prefill_s2048 (non-absorbed prefill).

Multi-GPU (torchrun): replicas only -- every rank runs the same workload on
its own GPU, no collective on the data path; value = all ranks' tokens / the
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


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except OSError:
        return FALLBACK, "fallback"


# ------------------------------------------------------------------ workloads
def build_workload(name, device):
    """Inputs + a closure running one step + the step's algorithmic accounting."""
    import torch
    import mla_latent_kv_06_gb300 as mla
    from workload import GLM, WORKLOADS, mla_inputs, workload_inputs, SEED_BASE

    if name.startswith("glm_decode_t"):
        T = int(name[len("glm_decode_t"):])
        if name == "glm_decode_t4096":
            x = workload_inputs(name, device)
        else:
            x = dict(dims=GLM, B=1, S=1, T_list=[T], T_cap=T, dtype="bf16")
            x.update(mla_inputs(GLM, 1, 1, [T], T, "bf16", SEED_BASE + 1, device))
        kind = "decode"
    elif name.startswith("glm_batched_b32_s"):
        S = int(name[len("glm_batched_b32_s"):])
        x = workload_inputs("glm_batched_b32", device, S=S)
        kind = "decode"
    elif name == "glm_dsa_t65536":
        x = workload_inputs(name, device)
        kind = "dsa"
    elif name == "glm_prefill_s2048":
        x = workload_inputs(name, device)
        kind = "prefill"
    else:
        raise SystemExit(f"unknown workload {name}")

    dims = x["dims"]
    B, S = x["B"], x["S"]
    T_list = x["T_list"]
    tokens = B * S
    w_bytes = 2 * dims.H * (dims.qk_nope + dims.v_head) * dims.kv_lora
    row = 2 * (dims.kv_lora + dims.qk_rope)
    q_bytes = 2 * B * S * dims.H * dims.qk_head
    out_bytes = 4 * B * S * dims.H * dims.v_head
    acct = {"tokens": tokens}
    out = torch.empty(B, S, dims.H, dims.v_head, dtype=torch.float32, device=device)

    if kind == "decode":
        need = mla.decode_workspace_size(dims, mla.MLA_BF16, B, S, x["T_cap"])
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)

        def step():
            mla.decode_absorbed(x["q"], x["Lc"], x["Rc"], x["T"], x["kv_b"], dims, out=out, workspace=ws)

        cache = row * sum(T_list)
        acct.update(cache_bytes=cache, alg_bytes=cache + w_bytes + q_bytes + out_bytes + 4 * B,
                    flops=2 * dims.H * sum(sum(T - S + s + 1 for s in range(S)) * (dims.kv_lora * 2 + dims.qk_rope)
                                           for T in T_list)
                    + 2 * dims.H * B * S * (dims.qk_nope + dims.v_head) * dims.kv_lora,
                    bound="hbm", kernels_per_step=mla_kernels_per_call("decode", dims, B, S))
        e2e = dict(inputs=[x["q"], x["T"]], run=lambda q, T: mla.decode_absorbed(
            q, x["Lc"], x["Rc"], T, x["kv_b"], dims, out=out, workspace=ws), out=out)
    elif kind == "dsa":
        k = x["topk"]
        sc = torch.empty(B, S, x["T_cap"], dtype=torch.float32, device=device)
        sel = torch.empty(B, S, k, dtype=torch.int32, device=device)
        nsel = torch.empty(B, S, dtype=torch.int32, device=device)
        need = mla.lib().mla_sparse_decode_workspace_size(
            mla.ctypes.byref(mla.make_dims(dims)), mla.MLA_BF16, B, S, k)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)

        def step():
            mla.index_scores(x["q_idx"], x["w"], x["Ic"], x["T"], out=sc)
            mla.topk_select(sc, x["T"], k, sel=sel, nsel=nsel)
            mla.sparse_decode(x["q"], x["Lc"], x["Rc"], x["T"], x["kv_b"], sel, nsel, dims, out=out,
                              workspace=ws)

        ic_bytes = 4 * x["Ic"].shape[2] * sum(T_list)
        gathered = row * B * S * k
        acct.update(cache_bytes=gathered, alg_bytes=ic_bytes + 2 * 4 * B * S * x["T_cap"] + gathered + w_bytes
                    + q_bytes + out_bytes, flops=0, bound="hbm",
                    kernels_per_step=2 + mla_kernels_per_call("sparse", dims, B, S))
        e2e = dict(inputs=[x["q"], x["q_idx"], x["w"], x["T"]], run=None, out=out)
    else:
        pos_base = x["pos_base"]
        need = mla.lib().mla_prefill_naive_workspace_size(
            mla.ctypes.byref(mla.make_dims(dims)), mla.MLA_BF16, B, S, pos_base)
        ws = torch.empty(need, dtype=torch.uint8, device=device)

        def step():
            mla.prefill_naive(x["q"], x["Lc"], x["Rc"], x["kv_b"], dims, pos_base, out=out, workspace=ws)

        Tk = pos_base + S
        pairs = sum(pos_base + s + 1 for s in range(S))
        acct.update(cache_bytes=row * Tk, alg_bytes=row * Tk + w_bytes + q_bytes + out_bytes,
                    flops=2 * Tk * dims.kv_lora * dims.H * (dims.qk_nope + dims.v_head)
                    + 2 * dims.H * pairs * (dims.qk_head + dims.v_head),
                    bound="tensor", kernels_per_step=2)
        e2e = dict(inputs=[x["q"]], run=None, out=out)
    return x, step, acct, e2e


def mla_kernels_per_call(kind, dims, B, S):
    """Kernels one API call launches (queried from the library)."""
    import mla_latent_kv_06_gb300 as mla
    return mla.kernels_per_call(kind, dims, B, S)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region."""

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
def graph_of(step, stream):
    """Capture one step into a CUDA graph (the library's launches, PDL edges included)."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    torch.cuda.synchronize()
    return g.replay


def time_steps(step, K, W, flush, stream):
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


def time_e2e(e2e, K, W, flush, stream):
    """Public-API call with host buffers: pinned H2D of the step inputs, the call, D2H of out."""
    import torch
    host_in = [t.detach().cpu().pin_memory() for t in e2e["inputs"]]
    dev_in = [torch.empty_like(t) for t in e2e["inputs"]]
    host_out = torch.empty(e2e["out"].shape, dtype=e2e["out"].dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out.numel() * host_out.element_size()

    def one():
        for d, h in zip(dev_in, host_in):
            d.copy_(h, non_blocking=True)
        e2e["run"](*dev_in)
        host_out.copy_(e2e["out"], non_blocking=True)

    ms = time_steps(one, K, W, flush, stream)
    return ms, h2d, d2h


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(name, budget_s=12.0):
    """Time the fp64 oracle on the host cores on a bounded sample of the workload."""
    import numpy as np
    import oracle
    from workload import WORKLOADS, GLM, mla_inputs, workload_inputs, SEED_BASE

    x = build_workload_cpu(name)
    q, Lc, Rc, kvb = (x[k] for k in ("q", "Lc", "Rc", "kv_b"))
    T_list, S = x["T_list"], x["S"]
    B = len(T_list)
    rows = [(b, s) for b in range(B) for s in range(S)]
    done, t0 = 0, time.perf_counter()
    while True:
        b, s = rows[done % len(rows)]
        pos = T_list[b] - S + s
        if x["kind"] == "prefill":
            oracle.prefill_nonabsorbed(q[0], Lc[0], Rc[0], kvb, GLM.qk_nope, GLM.softmax_scale,
                                       x["pos_base"], queries=[done % S])
        else:
            oracle.attend_absorbed(q[b, s], Lc[b, :pos + 1], Rc[b, :pos + 1], kvb, GLM.qk_nope, pos,
                                   GLM.softmax_scale)
        done += 1
        el = time.perf_counter() - t0
        if el > budget_s or done >= 4 * len(rows):
            break
    return done / el, done, el


def build_workload_cpu(name):
    """fp64 numpy copies of a workload's MLA inputs (CPU generator)."""
    import numpy as np
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
    out = {k: f(x[k]) for k in ("q", "Lc", "Rc", "kv_b")}
    out.update(T_list=x["T_list"], S=x["S"], kind="prefill" if name == "glm_prefill_s2048" else "decode",
               pos_base=x.get("pos_base", 0))
    return out


def host_threads():
    try:
        from threadpoolctl import threadpool_info
        import numpy  # noqa: F401  (loads BLAS)
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count() or 1


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mla", "reference"], default="mla")
    ap.add_argument("--workload", default="glm_decode_t4096")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time plain API calls instead of graph replays")
    args = ap.parse_args()
    W = max(args.warmup, 3)
    K = args.steps

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        tok_s, n, el = oracle_sample(args.workload, budget_s=max(5.0, 2.0 * K))
        cores = host_threads()
        line = {"impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": K, "warmup": W, "ms_per_step": 1e3 / tok_s, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": args.workload},
                "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
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
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    x, step, acct, e2e = build_workload(args.workload, dev)
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    assert mla.device_status() == 0
    # Timed steps replay a CUDA graph of the step so that host-side launch
    # cost (ctypes marshalling, tensor-map encoding) stays out of device time;
    # the e2e figure below goes through the plain API call instead.
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        replay = graph_of(step, cap) if not args.no_graph else step
    timed_step = replay

    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_wall = time.perf_counter()
    ms = time_steps(timed_step, K, W, flush, stream)
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    total_ms = sum(ms)
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
        dist.barrier()
    ms_per_step = total_ms / K
    value = world * acct["tokens"] * K / (total_ms / 1e3)

    pk, pk_kind = peaks()
    line = None
    if rank == 0:
        step_s = ms_per_step / 1e3
        if acct["bound"] == "hbm":
            achieved = acct["alg_bytes"] / step_s / 1e9
            peak = pk["hbm_gbs"]
            unit = "GB/s"
        else:
            achieved = acct["flops"] / step_s / 1e12
            peak = pk["bf16_tflops_sustained"]
            unit = "TFLOP/s"
        roof = {"bound": acct["bound"], "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "peak_source": pk_kind,
                "kernel": "whole step" if acct["kernels_per_step"] > 1 else "the step's one kernel",
                "alg_bytes_per_launch": acct["alg_bytes"], "traffic": None}
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
                "warmup": W, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": args.workload, "B": x["B"], "S": x["S"],
                           "T": x["T_list"] if len(x["T_list"]) <= 4 else f"sum {sum(x['T_list'])}",
                           "heads": 64, "kv_lora": 512, "qk_rope": 64, "qk_nope": 192, "v_head": 256,
                           "parallelism": f"replicas x{world}",
                           "l2": "256 MiB flush write before every timed step (outside the timed interval)",
                           "launch": "plain API calls" if args.no_graph else "CUDA graph replay of one API call"},
                "latent_cache_gbs": acct["cache_bytes"] / step_s / 1e9,
                "hbm_gbs_algorithmic": acct["alg_bytes"] / step_s / 1e9,
                "hbm_frac_of_8tbs": acct["alg_bytes"] / step_s / 8e12,
                "roofline": roof, "clocks": clk,
                "gpu_launches": acct["kernels_per_step"] * K,
                "step_ms_min": min(ms), "step_ms_median": statistics.median(ms),
                "wall_s_timed_region": t_wall}
    # end-to-end through the public API with host buffers
    if e2e.get("run") is not None:
        ems, h2d, d2h = time_e2e(e2e, K, W, flush, stream)
        if rank == 0:
            ev = acct["tokens"] * K / (sum(ems) / 1e3) * world
            line["e2e"] = {"value": ev, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                           "d2h_bytes_per_step": d2h, "ms_per_step": sum(ems) / K}
    elif rank == 0:
        line["e2e"] = None
    # T sweep of the metric (4k..64k) for the decode headline
    if rank == 0 and args.workload == "glm_decode_t4096" and not args.no_sweep:
        sweep = {}
        del x, step
        for T in (4096, 8192, 16384, 32768, 65536):
            xs, st_, ac, _ = build_workload(f"glm_decode_t{T}", dev)
            st_()
            with torch.cuda.stream(cap):
                rp = graph_of(st_, cap) if not args.no_graph else st_
            m = time_steps(rp, 20, 3, flush, stream)
            t = statistics.median(m) / 1e3
            sweep[str(T)] = {"tokens_s": 1 / t, "us": t * 1e6, "latent_cache_gbs": ac["cache_bytes"] / t / 1e9,
                             "hbm_gbs_algorithmic": ac["alg_bytes"] / t / 1e9,
                             "frac_of_measured_hbm": ac["alg_bytes"] / t / 1e9 / pk["hbm_gbs"]}
            del xs, st_
        line["t_sweep"] = sweep
    if rank == 0 and not args.no_cpu:
        tok_s, n, el = oracle_sample(args.workload)
        line["cpu_baseline"] = {"value": tok_s, "unit": "tokens/s", "cores": host_threads(), "kind": "oracle",
                                "sample": f"{n} query tokens x 64 heads of {args.workload} in {el:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
