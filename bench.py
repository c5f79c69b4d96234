"""Benchmark of the speculative-decoding verification step on GB300.

One step = one spec_verify call over one batch of the headline workload
(default c4: B=256 requests, gamma=4, V=151936, bf16 logits, T=1; the
largest-vocabulary workload, 700 MB of logits per step).  The metric is
verified draft positions per second (B * gamma per step) with the achieved
HBM bandwidth reported in `roofline`.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c4]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

Inputs are synthetic (seeded Philox, see speculative_decoding_verification_09_gb300/synth.py),
generated on the host and copied to the device once; three input sets rotate
so every step reads its 700 MB from HBM (3 x 700 MB >> 129 MB L2).
Multi-GPU (torchrun): every rank verifies its own batch (independent
requests, no collective on the data path); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_verification_09_gb300 import synth  # noqa: E402

METRIC = "verified draft positions/sec and achieved HBM GB/s (fraction of GB300 peak)"
NOMINAL_HBM_GBS = 7900.0
UNIT = "positions/s"
KERNEL_SRC = os.path.join(ROOT, "speculative_decoding_verification_09_gb300", "csrc",
                          "specverify.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_c4.txt")
WORKLOADS = {f"c{i}": i for i in synth.CONFIGS}


def code_hash(src: str) -> str:
    """sha256/16 of C/CUDA source with comments and blank lines removed."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    code = "\n".join(line.rstrip() for line in src.splitlines() if line.strip())
    return hashlib.sha256(code.encode("utf-8")).hexdigest()[:16]


def kernel_hash() -> str:
    """The kernel code's hash, so that an edit of a comment does not void the
    recorded counters but any change of code does."""
    with open(KERNEL_SRC, encoding="utf-8") as f:
        return code_hash(f.read())


def read_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def read_traffic() -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel source as it is now (else None)."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_code_sha256_16") != kernel_hash():
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
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
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_set_index(rank: int, s: int) -> int:
    """Input set s of a rank: every rank verifies its own requests (weak
    scaling, no data shared between ranks)."""
    return 1000 * rank + s


def max_over_ranks(x: float, dist_mod, device) -> float:
    """The job's time is the slowest rank's: MAX all-reduce of one float
    (NCCL on the GPU path; any backend works)."""
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step: int, world: int, steps: int, total_ms: float) -> float:
    """Whole-job units per second: every rank's units over the slowest rank's time."""
    return units_per_rank_step * world * steps / (total_ms / 1e3)


def oracle_positions_per_s(inp: synth.Inputs, n_req: int, threads: int,
                           keep: list | None = None) -> tuple[float, float]:
    """Time the oracle on the first n_req requests (the cpu_baseline leg);
    its result is appended to `keep` when given."""
    import oracle
    sl = slice(0, n_req)
    t0 = time.perf_counter()
    ref = oracle.verify(inp.Lt[sl], inp.Ld[sl], inp.x[sl], inp.u_acc[sl], inp.u_res[sl],
                        inp.temp[sl], inp.dtype, nthreads=threads)
    dt = time.perf_counter() - t0
    if keep is not None:
        keep.append(ref)
    return n_req * inp.gamma / dt, dt


def parity_counts(inp: synth.Inputs, tokens: np.ndarray, n: np.ndarray, ref: dict,
                  greedy: bool) -> dict:
    """The GPU's outputs for the first requests of an input set against the
    oracle's (computed in the cpu_baseline leg): flagged near-ties (accept
    tests within 1e-6 of u, draws within 1e-6 of a CDF edge, vanished
    residuals), requests that differ, and those that differ without a flag."""
    import oracle
    B = tokens.shape[0]
    flags = ref["flags"][:B]
    same = np.all(tokens == ref["tokens"][:B], axis=1) & (n == ref["n"][:B])
    inv = (flags & oracle.INVALID_ANY) != 0
    near = (flags & oracle.NEAR_ANY) != 0
    near_pos = 0 if greedy else int(((flags & oracle.NEAR_ACCEPT) != 0).sum()
                                    + ((flags & oracle.NEAR_SAMPLE) != 0).sum()
                                    + ((flags & oracle.DEGENERATE) != 0).sum())
    return {"requests": int(B), "positions": int(B * inp.gamma), "near_ties": near_pos,
            "near_tie_requests": int(near.sum()),
            "near_tie_rate": near_pos / max(1, B * inp.gamma),
            "mismatches": int((~inv & ~same).sum()),
            "unflagged_mismatches": int((~inv & ~same & ~near).sum())}


def run_reference(args) -> None:
    """The reference arm: the fp64 CPU oracle as it stands, on the host cores,
    timed on bounded samples of the same workload."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    cid = WORKLOADS[args.workload]
    n_req = args.ref_requests
    inp = synth.make_inputs(cid, B=n_req)
    cores = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle_positions_per_s(inp, n_req, cores)
    times = []
    for _ in range(args.steps):
        times.append(oracle_positions_per_s(inp, n_req, cores)[1])
    t = float(np.mean(times))
    value = n_req * inp.gamma / t
    cfg = synth.CONFIGS[cid]
    sample = f"first {n_req} of {cfg['B']} requests of {cfg['name']} per step, fp64, {cores} threads"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": cfg["name"], "B": cfg["B"],
                                        "gamma": cfg["gamma"], "V": cfg["V"],
                                        "sample_requests_per_step": n_req},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def measure_draft_side(binding, torch, dev, stream, sets, host_sets, B, g, V, ws, out_tok, out_n,
                       status, steps, warmup, peak) -> dict:
    """The steps beside verification on the same workload, each timed alone
    over `steps` calls (input sets rotating, CUDA events on the stream):
    sv_draft_sample over the B * gamma draft rows, and spec_verify_cached
    with the normalisers it produced (the draft rows are then not streamed)."""
    es = synth.ELEM_BYTES[host_sets[0].dtype]
    u = [torch.from_numpy(synth.draft_uniforms(B, g, 7000 + i)).to(dev) for i in range(len(sets))]
    tok = [torch.empty(B, g, dtype=torch.int32, device=dev) for _ in sets]
    stats = [torch.empty(B, g, 2, dtype=torch.float32, device=dev) for _ in sets]
    dws = binding.make_draft_workspace(B, g, V, dev)

    def draft(i):
        binding.sv_draft_sample(sets[i]["Ld"], u[i], sets[i]["temp"], tok[i], stats[i], dws,
                                dev_status=status, stream=stream)

    def cached(i):
        t = sets[i]
        binding.spec_verify_cached(t["Lt"], t["Ld"], tok[i], stats[i], t["u_acc"], t["u_res"],
                                   t["temp"], out_tok, out_n, ws, dev_status=status,
                                   stream=stream)

    def timed(fn):
        for i in range(warmup):
            fn(i % len(sets))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a.record(stream)
        for i in range(steps):
            fn(i % len(sets))
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / steps

    for i in range(len(sets)):  # every set's draft tokens and normalisers exist before timing
        draft(i)
    d_ms = timed(draft)
    c_ms = timed(cached)
    d_bytes = B * g * V * es
    c_bytes = B * (g + 1) * V * es
    return {
        "sv_draft_sample": {
            "ms_per_call": d_ms, "rows_per_s": B * g / (d_ms / 1e3),
            "logit_bytes": d_bytes, "call_gbs": d_bytes / (d_ms / 1e3) / 1e9,
            "frac_of_peak": d_bytes / (d_ms / 1e3) / 1e9 / peak, "kernels": 2},
        "spec_verify_cached": {
            "ms_per_call": c_ms, "positions_per_s": B * g / (c_ms / 1e3),
            "streamed_logit_bytes": c_bytes, "call_gbs": c_bytes / (c_ms / 1e3) / 1e9,
            "kernels": 4},
        "timing": f"{steps} calls each after {warmup} warm-up calls, CUDA events around the "
                  "loop, input sets rotating; not part of the headline value",
    }


KV_MODEL = dict(layers=24, kv_heads=16, head_dim=128, elem_bytes=2, sink=4, window=256)


def measure_kv_side(binding, torch, dev, stream, B, g, num_accepted, steps, warmup, peak,
                    window: int) -> dict:
    """The KV steps after verification, each timed alone over `steps` calls
    (CUDA events on the stream): committing the accepted entries of a
    1.8B-class target (24 layers x 16 KV heads, head dim 128, bf16; 4 sink
    slots and a ring of 256) with the verification's own accepted counts, the
    valid-slot lists, and a draft block-table window (W = 2048, block 128,
    K = gamma, lengths up to 32768)."""
    m = KV_MODEL
    LH, D, S, W, R = m["layers"] * m["kv_heads"], m["head_dim"], m["sink"], window, g + 1
    pools = [torch.zeros(B, LH, S + W, D, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    staged = [torch.randn(B, LH, R, D, generator=gen, device=dev).to(torch.bfloat16)
              for _ in range(2)]
    pos = torch.zeros(B, dtype=torch.int32, device=dev)
    slots = torch.empty(B, S + W, dtype=torch.int32, device=dev)
    lens = torch.empty(B, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    blk, Wd = 128, 2048
    full = 32768 // blk
    seq = torch.randint(1, 32768, (B,), generator=gen, device=dev, dtype=torch.int32)
    table = torch.randint(1, 1 << 30, (B, full), generator=gen, device=dev, dtype=torch.int32)
    cols = binding.sv_window_cols(Wd, blk)
    wseq = torch.empty(B, dtype=torch.int32, device=dev)
    wtab = torch.empty(B, cols, dtype=torch.int32, device=dev)

    def commit(i):
        binding.sv_kv_commit(pools[0], pools[1], staged[0], staged[1], num_accepted, pos, S, W,
                             dev_status=st, stream=stream)

    def valid(i):
        binding.sv_kv_valid_slots(pos, S, W, slots, lens, dev_status=st, stream=stream)

    def window(i):
        binding.sv_window_block_table(seq, table, Wd, blk, g, wseq, wtab, dev_status=st,
                                      stream=stream)

    def timed(fn):
        for i in range(warmup):
            fn(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a.record(stream)
        for i in range(steps):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / steps

    c_ms, v_ms, w_ms = timed(commit), timed(valid), timed(window)
    entries = int((num_accepted.clamp(min=-1) + 1).sum().item())
    moved = entries * LH * D * m["elem_bytes"] * 2 * 2  # K and V, read and written
    st_v = int(st.item())
    del pools, staged
    return {
        "model": f"{m['layers']} layers x {m['kv_heads']} KV heads x {D}, bf16, sink {S}, "
                 f"ring {W}, B {B}, R {R}",
        "sv_kv_commit": {"ms_per_call": c_ms, "entries_per_call": entries,
                         "algorithmic_bytes": moved,
                         "achieved_gbs": moved / (c_ms / 1e3) / 1e9,
                         "frac_of_peak": moved / (c_ms / 1e3) / 1e9 / peak, "kernels": 2},
        "sv_kv_valid_slots": {"ms_per_call": v_ms, "slots": B * (S + W)},
        "sv_window_block_table": {"ms_per_call": w_ms, "B": B, "window": Wd, "block": blk,
                                  "cols": cols},
        "status": st_v,
    }


def measure_streams(binding, torch, dev, sets, B, g, V, greedy, calls=60) -> dict:
    """Throughput when consecutive calls alternate over S streams, each with
    its own workspace and outputs (calls that may overlap need separate
    workspaces), so one call's latency-bound tail runs beside the next call's
    streaming reduce.  Not the headline: every call still takes its full
    single-call latency."""
    out = {}
    for S in (2, 3):
        streams = [torch.cuda.Stream(dev) for _ in range(S)]
        wss = [binding.make_workspace(B, g, V, dev) for _ in range(S)]
        bufs = [(torch.empty(B, g + 1, dtype=torch.int32, device=dev),
                 torch.empty(B, dtype=torch.int32, device=dev),
                 torch.zeros(1, dtype=torch.int32, device=dev)) for _ in range(S)]

        def call(i):
            j, t = i % S, sets[i % len(sets)]
            tok, n, st = bufs[j]
            if greedy:
                binding.spec_verify_greedy(t["Lt"], t["x"], tok, n, wss[j], st, streams[j])
            else:
                binding.spec_verify(t["Lt"], t["Ld"], t["x"], t["u_acc"], t["u_res"], t["temp"],
                                    tok, n, wss[j], st, streams[j])

        for i in range(2 * S):
            call(i)
        torch.cuda.synchronize(dev)
        main = torch.cuda.current_stream(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(main)
        for st_ in streams:
            st_.wait_event(a)
        for i in range(calls):
            call(i)
        for st_ in streams:
            e = torch.cuda.Event()
            e.record(st_)
            main.wait_event(e)
        b.record(main)
        torch.cuda.synchronize(dev)
        ms = a.elapsed_time(b) / calls
        out[f"{S}_streams"] = {"ms_per_call": ms, "positions_per_s": B * g / (ms / 1e3),
                               "status": [int(x[2].item()) for x in bufs]}
    out["timing"] = (f"{calls} calls alternating over the streams, CUDA events on the "
                     "launching stream around all of them; input sets rotating")
    return out


def measure_tree_side(binding, torch, dev, stream, steps, warmup, peak, sets=3) -> dict:
    """Token-tree verification (sv_tree_verify) on its workload: 64 requests,
    22-node trees (3, 2, 1, 1 children per level), V = 151936 bf16.  `sets`
    device copies of one batch at distinct addresses rotate between calls,
    so no call finds its rows in L2.  The algorithmic bytes of a call are the
    rows its walks must read once: each visited node's target row and the
    draft row of each visited node with children."""
    cfg = synth.TREE_WORKLOAD
    parent = synth.tree_parents(cfg["branching"])
    ti = synth.make_tree_inputs(cfg, parent)
    B, N, V = ti.B, ti.N, ti.V

    def dev_set():
        t = {k: torch.from_numpy(np.ascontiguousarray(getattr(ti, k))).to(dev)
             for k in ("Lt", "Ld", "parent", "tokens", "u_acc", "u_res", "temp")}
        t["Lt"], t["Ld"] = t["Lt"].view(torch.bfloat16), t["Ld"].view(torch.bfloat16)
        return t

    ds = [dev_set() for _ in range(sets)]
    tok = torch.empty(B, N, dtype=torch.int32, device=dev)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    nodes = torch.empty(B, N, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def call(i):
        t = ds[i % sets]
        binding.sv_tree_verify(t["Lt"], t["Ld"], t["parent"], t["tokens"], t["u_acc"],
                               t["u_res"], t["temp"], tok, n, nodes, st, stream)

    for i in range(warmup):
        call(i)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    a.record(stream)
    for i in range(steps):
        call(i)
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / steps
    n_h, nodes_h = n.cpu().numpy(), nodes.cpu().numpy()
    has_child = np.zeros(N, bool)
    has_child[parent[1:]] = True
    row = V * 2
    rows = 0
    for r in range(B):
        for v in [0] + [int(c) for c in nodes_h[r, :n_h[r]]]:
            rows += 1 + int(has_child[v])
    moved = rows * row
    del ds
    return {"workload": cfg["name"], "B": B, "N": N, "V": V, "ms_per_call": ms,
            "requests_per_s": B / (ms / 1e3), "accepted_per_request": float(n_h.mean()),
            "emitted_tokens_per_s": float((n_h + 1).sum()) / (ms / 1e3),
            "rows_read_per_call": rows, "algorithmic_bytes": moved,
            "all_rows_bytes": int((ti.Lt.nbytes + ti.Ld.nbytes)),
            "achieved_gbs": moved / (ms / 1e3) / 1e9,
            "frac_of_peak": moved / (ms / 1e3) / 1e9 / peak,
            "l2": f"{sets} device copies at distinct addresses, rotated", "kernels": 1,
            "status": int(st.item())}


def dev_tensors(torch, dev, inp: synth.Inputs) -> dict:
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(inp, k))).to(dev)
         for k in ("Lt", "Ld", "x", "u_acc", "u_res", "temp")}
    if inp.dtype == synth.BF16:
        t["Lt"], t["Ld"] = t["Lt"].view(torch.bfloat16), t["Ld"].view(torch.bfloat16)
    return t


def call_stats(ms: np.ndarray) -> dict:
    return {"median": float(np.median(ms)), "p10": float(np.percentile(ms, 10)),
            "p90": float(np.percentile(ms, 90)), "calls": int(ms.size)}


def measure_workload(binding, torch, dev, stream, cid: int, steps: int, warmup: int, peak: float,
                     sets: int = 3, parity_requests: int = 256) -> tuple[dict, dict]:
    """Another workload at its own size, measured in the same run as the
    headline: `steps` calls back to back between two events (call_ms), the
    reduce kernel alone with an event on each side (reduce_ms), and per-call
    times of max(steps, 50) calls each between its own two events; `sets`
    input sets rotate.  Also returns the outputs for the first requests of
    input set 0, for the parity count of the cpu_baseline leg."""
    cfg = synth.CONFIGS[cid]
    B, g, V = cfg["B"], cfg["gamma"], cfg["V"]
    greedy = cfg["kind"] == "greedy"
    host = [synth.make_inputs(cid, set_index=s) for s in range(sets)]
    lb = host[0].Lt.nbytes if greedy else host[0].logit_bytes
    ds = [dev_tensors(torch, dev, h) for h in host]
    ws = binding.make_workspace(B, g, V, dev)
    tok = torch.empty(B, g + 1, dtype=torch.int32, device=dev)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(t):
        if greedy:
            binding.spec_verify_greedy(t["Lt"], t["x"], tok, n, ws, st, stream)
        else:
            binding.spec_verify(t["Lt"], t["Ld"], t["x"], t["u_acc"], t["u_res"], t["temp"], tok,
                                n, ws, st, stream)

    for i in range(max(3, warmup)):
        step(ds[i % sets])
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        step(ds[i % sets])
    b.record(stream)
    torch.cuda.synchronize(dev)
    call_ms = a.elapsed_time(b) / steps
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for es in kev:  # torch creates an event on its first record
        for e in es:
            e.record(stream)
    torch.cuda.synchronize(dev)
    for i, es in enumerate(kev):
        binding.sv_set_stage_events(es)
        step(ds[i % sets])
    binding.sv_set_stage_events([])
    torch.cuda.synchronize(dev)
    reduce_ms = float(np.mean([es[0].elapsed_time(es[1]) for es in kev]))
    nl = max(steps, 50)
    lev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(nl)]
    for i, (e0, e1) in enumerate(lev):
        e0.record(stream)
        step(ds[i % sets])
        e1.record(stream)
    torch.cuda.synchronize(dev)
    lat = np.array([e0.elapsed_time(e1) for e0, e1 in lev])
    status = int(st.item())
    step(ds[0])
    torch.cuda.synchronize(dev)
    k = min(B, parity_requests)
    out = dict(inp=host[0], tokens=tok[:k].cpu().numpy(), n=n[:k].cpu().numpy(), greedy=greedy)
    res = {"workload": cfg["name"], "B": B, "gamma": g, "V": V, "greedy": greedy,
           "dtype": cfg["dtype"], "logit_bytes": int(lb), "call_ms": call_ms,
           "positions_per_s": B * g / (call_ms / 1e3), "call_gbs": lb / (call_ms / 1e3) / 1e9,
           "call_frac_of_peak": lb / (call_ms / 1e3) / 1e9 / peak, "reduce_ms": reduce_ms,
           "reduce_frac_of_peak": lb / (reduce_ms / 1e3) / 1e9 / peak,
           "per_call_ms": call_stats(lat), "status": status,
           "timing": f"{steps} calls back to back between two events; reduce with an event "
                     f"on each side; {nl} calls each between its own events; "
                     f"{sets} input sets rotating"}
    del ds, ws
    return res, out


def run_tree_only(args) -> None:
    """Token-tree verification alone (for profiling captures): one JSON dict."""
    import torch

    from speculative_decoding_verification_09_gb300 import binding
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    binding.lib()
    peak, _ = read_peaks()
    print(json.dumps(measure_tree_side(binding, torch, dev, torch.cuda.current_stream(dev),
                                       args.steps, args.warmup, peak, sets=args.tree_sets)))


def run_ours(args) -> None:
    import torch

    from speculative_decoding_verification_09_gb300 import binding

    ws_n, rank, local = dist_env()
    pg = None
    if ws_n > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        pg = dist
    dev = torch.device("cuda", local if ws_n > 1 else 0)
    torch.cuda.set_device(dev)
    cid = WORKLOADS[args.workload]
    cfg = synth.CONFIGS[cid]
    B, g, V = cfg["B"], cfg["gamma"], cfg["V"]
    if args.batch:  # a smaller batch of the same workload (profiling captures)
        B = args.batch
    greedy = cfg["kind"] == "greedy"
    stream = torch.cuda.current_stream(dev)

    # input sets: host copies (pinned, for the end-to-end leg) and device copies
    host_sets = [synth.make_inputs(cid, set_index=rank_set_index(rank, s), B=B)
                 for s in range(args.sets)]
    logit_bytes = host_sets[0].Lt.nbytes if greedy else host_sets[0].logit_bytes

    sets = [dev_tensors(torch, dev, h) for h in host_sets]
    out_tok = torch.empty(B, g + 1, dtype=torch.int32, device=dev)
    out_n = torch.empty(B, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = binding.make_workspace(B, g, V, dev)
    if args.chunk:
        binding.sv_set_tuning(args.chunk)
    binding.sv_set_tail(args.tail)

    def step(t):
        if greedy:
            binding.spec_verify_greedy(t["Lt"], t["x"], out_tok, out_n, ws, status, stream)
        else:
            binding.spec_verify(t["Lt"], t["Ld"], t["x"], t["u_acc"], t["u_res"], t["temp"],
                                out_tok, out_n, ws, status, stream)

    for i in range(args.warmup):
        step(sets[i % len(sets)])
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    clocks = ClockSampler(dev.index if dev.index is not None else 0)

    def soak(seconds):  # back-to-back calls of the same workload (clocks under load)
        t_end = time.perf_counter() + seconds
        i = 0
        while time.perf_counter() < t_end:
            for _ in range(20):
                step(sets[i % len(sets)])
                i += 1
            torch.cuda.synchronize(dev)

    if not args.no_clocks:
        clocks.start()
        soak(0.3)
    # two events around the K back-to-back steps (an event between two calls
    # would keep the next call's first kernel from being placed early)
    ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # the reduce kernel's duration: a second loop of the same steps in which the
    # library records an event before its first kernel and one after the
    # reduce kernel (an event between two kernels stops the next one from
    # being launched early, so the headline loop has none)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fused = not greedy and (args.tail == 2 or (args.tail == 0 and min(8, sms // B) >= 2))
    if greedy:
        kernel_names = ["reduce", "decide"]
    elif fused:  # small batches: one fused kernel after the reduce
        kernel_names = ["reduce", "finish"]
    else:
        kernel_names = ["reduce", "decide", "residual", "draw"]
    n_kern = len(kernel_names)

    def make_events(n):
        es = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in es:  # create them
            e.record(stream)
        return es

    kev = [make_events(2) for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    t_wall = time.perf_counter()
    ev_a.record(stream)
    for i in range(args.steps):
        step(sets[i % len(sets)])
    ev_b.record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall
    if pg:
        pg.barrier()
    for i in range(args.steps):
        binding.sv_set_stage_events(kev[i])
        step(sets[i % len(sets)])
    binding.sv_set_stage_events([])
    torch.cuda.synchronize(dev)
    reduce_ms = float(np.mean([es[0].elapsed_time(es[1]) for es in kev]))
    # breakdown over all kernels, from a few extra (untimed) calls with an
    # event between every two kernels
    bev = [make_events(n_kern + 1) for _ in range(5)]
    for i, es in enumerate(bev):
        binding.sv_set_stage_events(es)
        step(sets[i % len(sets)])
    binding.sv_set_stage_events([])
    torch.cuda.synchronize(dev)
    stage_ms = {nm: float(np.mean([es[j].elapsed_time(es[j + 1]) for es in bev]))
                for j, nm in enumerate(kernel_names)}
    # single-call latency distribution: K more calls, each bracketed by its
    # own events (which keep calls from overlapping, unlike the timed loop)
    lev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(max(args.steps, 50))]
    for i, (a_, b_) in enumerate(lev):
        a_.record(stream)
        step(sets[i % len(sets)])
        b_.record(stream)
    torch.cuda.synchronize(dev)
    lat = np.array([a_.elapsed_time(b_) for a_, b_ in lev])
    latency_ms = {"p10": float(np.percentile(lat, 10)), "p50": float(np.percentile(lat, 50)),
                  "p90": float(np.percentile(lat, 90)), "calls": int(lat.size)}
    if not args.no_clocks:
        soak(0.1)
    clk = clocks.stop() if not args.no_clocks else None
    if clk is not None:
        clk["window"] = ("0.3 s of back-to-back calls of the same workload before the timed "
                         "steps, the timed steps, the stage and per-call timings, 0.1 s of "
                         "calls after; samples every 20 ms")
    total_ms = ev_a.elapsed_time(ev_b)
    peak, peak_kind = read_peaks()
    multi_stream = None if args.no_multi_stream else measure_streams(
        binding, torch, dev, sets, B, g, V, greedy)
    draft_side = None if (greedy or args.no_draft_side) else measure_draft_side(
        binding, torch, dev, stream, sets, host_sets, B, g, V, ws, out_tok, out_n, status,
        args.steps, args.warmup, peak)
    tree_side = None
    if not args.no_tree_side:
        tree_side = measure_tree_side(binding, torch, dev, stream, args.steps, args.warmup, peak)
    kv_side = None
    if not args.no_kv_side:
        step(sets[0])  # the accepted counts of one verification drive the commit
        kv_side = measure_kv_side(binding, torch, dev, stream, B, g, out_n.clone(), args.steps,
                                  args.warmup, peak, args.kv_window)

    if pg:
        total_ms = max_over_ranks(total_ms, pg, dev)
    st = int(status.item())
    ms_step = total_ms / args.steps
    value = job_throughput(B * g, ws_n, args.steps, total_ms)
    launch_ms = total_ms / args.steps
    # the dominant kernel is the streaming reduce: it reads every logit once
    achieved = logit_bytes / (reduce_ms / 1e3) / 1e9

    # end to end: pinned host inputs -> device, verify, results -> host, every step
    e2e = None
    if not args.no_e2e:
        h = host_sets[0]
        pinned = {k: torch.from_numpy(np.ascontiguousarray(getattr(h, k))).pin_memory()
                  for k in ("Lt", "Ld", "x", "u_acc", "u_res", "temp")}
        d = {k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in pinned.items()}
        tok_h = torch.empty(B, g + 1, dtype=torch.int32).pin_memory()
        n_h = torch.empty(B, dtype=torch.int32).pin_memory()
        keys = ("Lt", "x") if greedy else ("Lt", "Ld", "x", "u_acc", "u_res", "temp")
        h2d = sum(pinned[k].numel() * pinned[k].element_size() for k in keys)
        d2h = tok_h.numel() * 4 + n_h.numel() * 4

        # the batch in chunks of requests: chunk j's inputs are copied on a copy
        # stream while chunk j - 1 is verified (requests are independent)
        nsub = max(1, min(args.e2e_chunks, B))
        bs = (B + nsub - 1) // nsub
        copy_st = torch.cuda.Stream(dev)
        ws_sub = binding.make_workspace(bs, g, V, dev)

        def e2e_step():
            go = torch.cuda.Event()
            go.record(stream)  # this step's copies follow the previous step's verification
            copy_st.wait_event(go)
            for j in range(0, B, bs):
                sl = slice(j, min(B, j + bs))
                ready = torch.cuda.Event()
                with torch.cuda.stream(copy_st):
                    for k in keys:
                        d[k][sl].copy_(pinned[k][sl], non_blocking=True)
                    ready.record(copy_st)
                stream.wait_event(ready)
                t = {k: v[sl] for k, v in d.items()}
                if h.dtype == synth.BF16:
                    t["Lt"], t["Ld"] = t["Lt"].view(torch.bfloat16), t["Ld"].view(torch.bfloat16)
                if greedy:
                    binding.spec_verify_greedy(t["Lt"], t["x"], out_tok[sl], out_n[sl], ws_sub,
                                               status, stream)
                else:
                    binding.spec_verify(t["Lt"], t["Ld"], t["x"], t["u_acc"], t["u_res"],
                                        t["temp"], out_tok[sl], out_n[sl], ws_sub, status, stream)
                tok_h[sl].copy_(out_tok[sl], non_blocking=True)
                n_h[sl].copy_(out_n[sl], non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        k_e2e = max(3, min(args.steps, 10))
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(k_e2e):
            e2e_step()
        b_.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = a.elapsed_time(b_) / k_e2e
        e2e = {"value": B * g / (e_ms / 1e3), "unit": UNIT, "ms_per_step": e_ms,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "chunks": nsub,
               "path": "pinned host inputs copied in chunks of requests on a copy stream, "
                       "each chunk verified as it lands, results copied back"}

    # the other workloads at their own sizes, after the headline (one GPU)
    workloads, wl_out = None, {}
    if rank == 0 and ws_n == 1 and not args.no_workloads and not args.batch:
        workloads = {}
        for c2 in sorted(synth.CONFIGS):
            if c2 == cid:
                continue
            res, out = measure_workload(binding, torch, dev, stream, c2, args.steps, args.warmup,
                                        peak)
            workloads[f"c{c2}"] = res
            wl_out[f"c{c2}"] = out
            torch.cuda.empty_cache()

    # the headline's outputs for the first requests of input set 0 (parity count)
    n_req = min(B, args.cpu_requests)
    step(sets[0])
    torch.cuda.synchronize(dev)
    head_tok, head_n = out_tok[:n_req].cpu().numpy(), out_n[:n_req].cpu().numpy()

    cpu, parity = None, None
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        import oracle
        cores = os.cpu_count() or 1
        # repeat the bounded sample until about cpu_seconds of work were timed
        passes, dt, keep = 0, 0.0, []
        while passes == 0 or dt < args.cpu_seconds:
            dt += oracle_positions_per_s(host_sets[0], n_req, cores, keep if passes == 0 else None)[1]
            passes += 1
        v = passes * n_req * g / dt
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"first {n_req} of {B} requests of {cfg['name']} (set 0), fp64, "
                         f"{cores} threads, {passes} passes, {dt:.1f} s wall"}
        # the GPU's outputs against the oracle's on the same requests: flagged
        # near-ties and differing requests, headline and the other workloads
        h0 = host_sets[0]
        if greedy:
            keep = [oracle.greedy(h0.Lt[:n_req], h0.x[:n_req], h0.dtype)]
        parity = {cfg["name"]: parity_counts(h0, head_tok, head_n, keep[0], greedy)}
        for key, o in wl_out.items():
            inp, k = o["inp"], o["tokens"].shape[0]
            if o["greedy"]:
                ref = oracle.greedy(inp.Lt[:k], inp.x[:k], inp.dtype)
            else:
                ref = oracle.verify(inp.Lt[:k], inp.Ld[:k], inp.x[:k], inp.u_acc[:k],
                                    inp.u_res[:k], inp.temp[:k], inp.dtype, nthreads=cores)
            parity[synth.CONFIGS[int(key[1:])]["name"]] = parity_counts(inp, o["tokens"], o["n"],
                                                                          ref, o["greedy"])
        tot_pos = sum(p_["positions"] for p_ in parity.values())
        parity["all"] = {"positions": tot_pos,
                         "near_ties": sum(p_["near_ties"] for p_ in parity.values()),
                         "mismatches": sum(p_["mismatches"] for p_ in parity.values()),
                         "unflagged_mismatches": sum(p_["unflagged_mismatches"]
                                                     for p_ in parity.values())}
        parity["rule"] = ("GPU outputs vs the fp64 oracle on the first requests of input set 0 "
                          "of each workload (the cpu_baseline leg's own oracle runs); near_ties "
                          "counts accept tests within 1e-6 of u, draws within 1e-6 of a CDF "
                          "edge and vanished residuals; a mismatch is a request whose tokens "
                          "or count differ")

    if rank != 0:
        return
    traffic = read_traffic() if (cid == 4 and not args.batch and args.tail != 2) else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if cfg["dtype"] == "bf16" else "f32",
        "data": "synthetic",
        "config": {"workload": cfg["name"], "B": B, "gamma": g, "V": V, "greedy": greedy,
                   "logit_bytes_per_step": int(logit_bytes),
                   "l2": f"{args.sets} rotating input sets of {logit_bytes / 1e6:.0f} MB "
                         f"(each larger than the 129 MB L2)"},
        "roofline": {"bound": "hbm", "kernel": "reduce", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_source": peak_kind, "kernel_ms": reduce_ms,
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "nominal": "GB300 HBM3e 7.9 TB/s (datasheet figure, context only)",
                     "algorithmic_bytes": int(logit_bytes),
                     "timing": f"CUDA events around the reduce kernel over {args.steps} calls "
                               "right after the timed loop (same inputs)"},
        "stages_ms_extra_calls": stage_ms, "call_ms": launch_ms,
        "single_call_latency_ms": latency_ms,
        "per_call_ms": dict(call_stats(lat), mean_of_timed_loop=launch_ms),
        "workloads": workloads, "parity": parity,
        "call_equivalent_gbs": logit_bytes / (launch_ms / 1e3) / 1e9,
        "concurrent_calls": multi_stream,
        "draft_side": draft_side, "kv_side": kv_side, "tree_side": tree_side,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": n_kern * args.steps, "clocks": clk,
        "status": st, "wall_s_timed": t_wall,
        "tuning": {"chunk": args.chunk, "tail": args.tail},
    }
    print(json.dumps(line))
    if pg:
        pg.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="c4")
    ap.add_argument("--sets", type=int, default=3)
    ap.add_argument("--batch", type=int, default=0,
                    help="requests per step (0 = the workload's own); for profiling captures")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=4,
                    help="request chunks of the end-to-end leg (copy of one overlaps the next)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-draft-side", action="store_true",
                    help="skip timing sv_draft_sample and spec_verify_cached")
    ap.add_argument("--no-kv-side", action="store_true",
                    help="skip timing the KV commit, valid slots and block-table window")
    ap.add_argument("--no-multi-stream", action="store_true",
                    help="skip timing calls that alternate over several streams")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip measuring the other workloads after the headline")
    ap.add_argument("--no-tree-side", action="store_true",
                    help="skip timing token-tree verification")
    ap.add_argument("--tree-only", action="store_true",
                    help="time token-tree verification alone (profiling captures)")
    ap.add_argument("--tree-sets", type=int, default=3)
    ap.add_argument("--kv-window", type=int, default=KV_MODEL["window"],
                    help="ring slots of the KV-commit measurement (smaller for profiling captures)")
    ap.add_argument("--cpu-requests", type=int, default=256)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="approximate seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-requests", type=int, default=32)
    ap.add_argument("--chunk", type=int, default=0, help="phase-1 chunk elements (0 = auto)")
    ap.add_argument("--tail", type=int, default=0, choices=[0, 1, 2, 3],
                    help="kernels of a sampling call: 0 automatic, 1 reduce + decide/residual/"
                         "draw, 2 reduce + fused tail, 3 one kernel")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    if args.tree_only:
        run_tree_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
