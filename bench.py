"""Benchmark: prefix-cached paged attention on one GB300 (replicas across GPUs under torchrun).

Default workload: the fork / self-consistency mixed step -- 32 layers of Llama-2-7B attention
(32 x 128 MHA, bf16), a 300k-slot pool kept full so that LRU eviction runs every step, 16
programs x 5 forks extending 200 new tokens over a cached 1500-token prefix, and 128 requests
decoding over contexts of 512..8192 tokens. One step is the whole hot path: radix match + lock,
LRU eviction, slot allocation, slot-table write, and per layer extend attention (with the K/V
scatter) and split-K decode attention (with its merge), then insert + unlock.

Prints one JSON line. `value` is extend-attention throughput in algorithmic TFLOP/s
(4 * d * Hq * (S*P + S(S+1)/2) per request and layer) over the time the extend launches take
inside the step; `decode` gives decode KV GB/s (L * (2 * Hkv * d * 2 B + 4 B) per request and
layer) over the decode launches; `prefill_tokens_skipped` the matched-token count.

--impl reference times the oracle (plain CPU C++, fp64) on the same workload and metric, a
bounded sample of units per step, on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "extend attn TFLOP/s & decode KV GB/s vs GB300 peak; prefill tokens skipped"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "source": "fallback"}


# DRAM traffic per launch from one ncu capture (`--write-traffic`), tied to the kernel sources it
# was taken on: a figure whose source file has changed since is reported as null
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_fork_mixed_step.json")
TRAFFIC_SOURCES = {"extend": "prefix_cached_paged_gb300/csrc/extend_tc.cu",
                   "decode": "prefix_cached_paged_gb300/csrc/decode.cu"}
# kernels whose launches make up one call of each entry point
TRAFFIC_KERNELS = {"extend": ("extend_tc_kernel",),
                   "decode": ("decode_plan_kernel", "decode_mma_kernel", "decode_merge_kernel")}


def source_hash(rel):
    import hashlib
    return hashlib.sha256(open(os.path.join(ROOT, rel), "rb").read()).hexdigest()


def stored_traffic():
    """{"extend": bytes per call or None, "decode": ...}; None where no capture matches the
    current kernel source."""
    out = {k: None for k in TRAFFIC_SOURCES}
    if not os.path.exists(TRAFFIC_FILE):
        return out
    d = json.load(open(TRAFFIC_FILE))
    for k, rel in TRAFFIC_SOURCES.items():
        e = d.get(k)
        if e and e.get("source_sha256") == source_hash(rel):
            out[k] = e["dram_bytes_per_call"]
    return out


def write_traffic(csv_path, command):
    """Summarise an ncu --csv capture of dram__bytes_read.sum and dram__bytes_write.sum into
    TRAFFIC_FILE: per entry point, the mean DRAM bytes of each of its kernels, summed per call."""
    import csv
    import collections
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12}
    rows = list(csv.reader(open(csv_path)))
    hi = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    h = rows[hi]
    ids, ki, mi, ui, vi = (h.index(c) for c in ("ID", "Kernel Name", "Metric Name",
                                                 "Metric Unit", "Metric Value"))
    per_launch = collections.defaultdict(lambda: [None, 0.0])
    for r in rows[hi + 1:]:
        if len(r) <= vi or r[mi] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        e = per_launch[r[ids]]
        e[0] = r[ki].split("(")[0].split("::")[-1].split("<")[0]
        e[1] += float(r[vi].replace(",", "")) * scale[r[ui]]
    by_kernel = collections.defaultdict(list)
    for name, b in per_launch.values():
        by_kernel[name].append(b)
    out = {"command": command, "metrics": "dram__bytes_read.sum + dram__bytes_write.sum"}
    for k, names in TRAFFIC_KERNELS.items():
        if all(n in by_kernel for n in names):
            out[k] = {"source_sha256": source_hash(TRAFFIC_SOURCES[k]),
                      "dram_bytes_per_call": round(sum(float(np.mean(by_kernel[n]))
                                                       for n in names)),
                      "per_kernel": {n: {"launches": len(by_kernel[n]),
                                         "mean_bytes": round(float(np.mean(by_kernel[n])))}
                                     for n in names}}
    os.makedirs(os.path.dirname(TRAFFIC_FILE), exist_ok=True)
    json.dump(out, open(TRAFFIC_FILE, "w"), indent=1)
    print(json.dumps(out))


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["source"] = "measured"
        return d
    return dict(FALLBACK_PEAKS)


# ------------------------------------------------------------------ distributed plumbing
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:   # host-only runs (tests of the replica plumbing)
            dist.init_process_group("gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workload: fork mixed step
def extend_flops(P, S, Hq, d):
    P = np.asarray(P, dtype=np.float64)
    S = np.asarray(S, dtype=np.float64)
    return float(np.sum(4.0 * d * Hq * (S * P + S * (S + 1) / 2)))


def decode_bytes(seq_len, Hkv, d, elem=2):
    return float(np.sum(np.asarray(seq_len, dtype=np.float64) * (2 * Hkv * d * elem + 4)))


def setup_fork_mixed(args):
    import torch
    from synth import workloads as W
    from tests import harness as H
    import synth
    from synth import device as sdev

    fm = W.fork_mixed_step(layers=args.layers)
    w = fm.workload
    m = w.model
    eng = H.make_engine(w, max_reqs=len(fm.decode_seqs) + 80 + 8, kv_chunk=args.kv_chunk)
    t0 = time.time()
    for ph in w.phases:
        H.run_cache_phase(eng, m, ph.seqs, keep_locked=False)
    db = eng.decode_begin([s[:-1] for s in fm.decode_seqs])
    setup_s = time.time() - t0
    assert eng.host.pool.available() == 4096, eng.host.pool.available()
    # step inputs (identical values reused by every step: values do not change the work)
    ext0 = fm.extend_seqs(0)
    P0 = 1500
    h_ext = np.concatenate([synth.prefix_hashes(m.seed, s)[P0:] for s in ext0])
    hd_ext = sdev.hashes_to_device(h_ext)
    T = len(h_ext)
    h_dec = np.array([synth.prefix_hashes(m.seed, s)[-1] for s in fm.decode_seqs], np.uint64)
    hd_dec = sdev.hashes_to_device(h_dec)
    Bd = len(fm.decode_seqs)
    dt = torch.bfloat16
    xq = torch.empty((m.layers, T, m.n_q_heads, m.head_dim), dtype=dt, device="cuda")
    xk = torch.empty((m.layers, T, m.n_kv_heads, m.head_dim), dtype=dt, device="cuda")
    xv = torch.empty_like(xk)
    dq = torch.empty((m.layers, Bd, m.n_q_heads, m.head_dim), dtype=dt, device="cuda")
    dk = torch.empty((m.layers, Bd, m.n_kv_heads, m.head_dim), dtype=dt, device="cuda")
    dv = torch.empty_like(dk)
    for layer in range(m.layers):
        sdev.fill_rows(hd_ext, synth.TENSOR_Q, layer, xq[layer])
        sdev.fill_rows(hd_ext, synth.TENSOR_K, layer, xk[layer])
        sdev.fill_rows(hd_ext, synth.TENSOR_V, layer, xv[layer])
        sdev.fill_rows(hd_dec, synth.TENSOR_Q, layer, dq[layer])
        sdev.fill_rows(hd_dec, synth.TENSOR_K, layer, dk[layer])
        sdev.fill_rows(hd_dec, synth.TENSOR_V, layer, dv[layer])
    xo = torch.empty((T, m.n_q_heads, m.head_dim), dtype=dt, device="cuda")
    do = torch.empty((Bd, m.n_q_heads, m.head_dim), dtype=dt, device="cuda")
    torch.cuda.synchronize()
    n_steps = args.warmup + args.steps + 3   # + the end-to-end steps
    seqs = [fm.extend_seqs(s) for s in range(n_steps)]
    return dict(fm=fm, w=w, m=m, eng=eng, db=db, xq=xq, xk=xk, xv=xv, dq=dq, dk=dk, dv=dv,
                xo=xo, do=do, T=T, Bd=Bd, seqs=seqs, setup_s=setup_s, ext0=ext0,
                max_total=int(db.seq_len.sum()) + Bd * (n_steps + 1))


def run_step(ctx, s, ev=None, host_t=None, e2e=None):
    """One mixed step over batch s. ev: list of (start, after-extend, after-decode) CUDA events
    per layer. e2e: host buffers (copies in and out inside the step)."""
    eng, m, db = ctx["eng"], ctx["m"], ctx["db"]
    h0 = eng.host.host_seconds
    eb = eng.extend_begin(ctx["seqs"][s], extra=ctx["Bd"])
    eng.decode_step(db, new_slots=eb.plan.extra)
    mt = ctx["max_total"]   # fixed bound: the workspace is sized once
    if e2e is not None:
        _layers_with_copies(ctx, eb, ev, e2e)
        _, dups = eng.extend_end(eb)
        if host_t is not None:
            host_t.append(eng.host.host_seconds - h0)
        return eb
    for layer in range(m.layers):
        if ev is not None:
            ev[layer][0].record()
        eng.extend_layer(eb, layer, ctx["xq"][layer], ctx["xk"][layer], ctx["xv"][layer],
                         ctx["xo"])
        if ev is not None:
            ev[layer][1].record()
        eng.decode_layer(db, layer, ctx["dq"][layer], ctx["dk"][layer], ctx["dv"][layer],
                         ctx["do"], max_total_tokens=mt)
        if ev is not None:
            ev[layer][2].record()
    _, dups = eng.extend_end(eb)
    if host_t is not None:
        host_t.append(eng.host.host_seconds - h0)
    return eb


def _layers_with_copies(ctx, eb, ev, e2e):
    """The step's layers with their inputs copied in from pinned host memory and their outputs
    copied back, overlapped with the kernels: layer l+1's inputs go up (one copy stream) while
    layer l computes, layer l's outputs come down (another copy stream, the link is full duplex)
    as soon as its kernels are done; two device buffer sets, events guard their reuse. ev[l]
    brackets layer l's extend and decode phases on the compute stream, including any time spent
    waiting for a copy; the last phase ends when the last output is on the host."""
    import torch
    eng, m, db = ctx["eng"], ctx["m"], ctx["db"]
    mt = ctx["max_total"]
    comp = torch.cuda.current_stream()
    up, down = ctx["up_stream"], ctx["down_stream"]
    dev = ctx["e2e_dev"]          # name -> [buffer 0, buffer 1]
    L = m.layers
    in_ready = [torch.cuda.Event() for _ in range(L)]
    comp_done = [torch.cuda.Event() for _ in range(L)]
    out_done = [torch.cuda.Event() for _ in range(L)]
    ev[0][0].record()
    up.wait_stream(comp)

    def upload(l):
        with torch.cuda.stream(up):
            if l >= 2:
                up.wait_event(comp_done[l - 2])     # buffer l % 2 no longer read
            for n in ("xq", "xk", "xv", "dq", "dk", "dv"):
                dev[n][l % 2].copy_(e2e[n], non_blocking=True)
            in_ready[l].record(up)

    upload(0)
    for l in range(L):
        if l + 1 < L:
            upload(l + 1)
        if l > 0:
            ev[l][0].record()
        comp.wait_event(in_ready[l])
        if l >= 2:
            comp.wait_event(out_done[l - 2])        # output buffer l % 2 copied back
        b = l % 2
        eng.extend_layer(eb, l, dev["xq"][b], dev["xk"][b], dev["xv"][b], dev["xo"][b])
        ev[l][1].record()
        eng.decode_layer(db, l, dev["dq"][b], dev["dk"][b], dev["dv"][b], dev["do"][b],
                         max_total_tokens=mt)
        comp_done[l].record()
        with torch.cuda.stream(down):
            down.wait_event(comp_done[l])
            e2e["xo"].copy_(dev["xo"][b], non_blocking=True)
            e2e["do"].copy_(dev["do"][b], non_blocking=True)
            out_done[l].record(down)
        if l == L - 1:
            comp.wait_event(out_done[l])
        ev[l][2].record()


def bench_ours(args, rank, world, local):
    import torch
    import prefix_cached_paged_gb300 as rc

    ctx = setup_fork_mixed(args)
    m, eng, db = ctx["m"], ctx["eng"], ctx["db"]
    for s in range(args.warmup):
        run_step(ctx, s)
    torch.cuda.synchronize()

    # ---------------- timed region (device-resident inputs)
    S = [np.asarray(ctx["seqs"][args.warmup + k]) for k in range(args.steps)]
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(m.layers)]
           for _ in range(args.steps)]
    host_t = []
    plans = []
    seq_lens = []
    launches0 = rc.launch_count()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for k in range(args.steps):
        seq_lens.append(db.seq_len.copy() + 1)
        plans.append(run_step(ctx, args.warmup + k, ev=evs[k], host_t=host_t))
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    launches = rc.launch_count() - launches0
    total_ms = start.elapsed_time(end)
    ext_ms = sum(e[l][0].elapsed_time(e[l][1]) for e in evs for l in range(m.layers))
    dec_ms = sum(e[l][1].elapsed_time(e[l][2]) for e in evs for l in range(m.layers))
    assert rc.device_status() == 0

    # algorithmic work of the timed steps
    ext_flops = 0.0
    skipped = prompt = 0
    for p in plans:
        Pl = p.plan.prefix_len.astype(np.int64)
        Sl = p.plan.lengths - Pl
        ext_flops += extend_flops(Pl, Sl, m.n_q_heads, m.head_dim) * m.layers
        skipped += int(Pl.sum())
        prompt += int(p.plan.lengths.sum())
    dec_bytes = sum(decode_bytes(sl, m.n_kv_heads, m.head_dim) * m.layers for sl in seq_lens)
    total_ms = max_over_ranks(total_ms, world)
    ext_ms_m = max_over_ranks(ext_ms, world)
    dec_ms_m = max_over_ranks(dec_ms, world)
    ext_tflops = world * ext_flops / (ext_ms_m * 1e-3) / 1e12
    dec_gbs = world * dec_bytes / (dec_ms_m * 1e-3) / 1e9

    # ---------------- end to end: inputs from pinned host memory, outputs back, every layer
    e2e = None
    if args.e2e:
        T, Bd = ctx["T"], ctx["Bd"]
        hb = {}
        for name in ("xq", "xk", "xv", "dq", "dk", "dv"):
            hb[name] = ctx[name][0].cpu().pin_memory()
        hb["xo"] = torch.empty(ctx["xo"].shape, dtype=ctx["xo"].dtype).pin_memory()
        hb["do"] = torch.empty(ctx["do"].shape, dtype=ctx["do"].dtype).pin_memory()
        ctx["up_stream"], ctx["down_stream"] = torch.cuda.Stream(), torch.cuda.Stream()
        ctx["e2e_dev"] = {n: [torch.empty_like(ctx[n][0]) for _ in range(2)]
                          for n in ("xq", "xk", "xv", "dq", "dk", "dv")}
        ctx["e2e_dev"]["xo"] = [torch.empty_like(ctx["xo"]) for _ in range(2)]
        ctx["e2e_dev"]["do"] = [torch.empty_like(ctx["do"]) for _ in range(2)]
        h2d = sum(hb[n].numel() * hb[n].element_size() for n in ("xq", "xk", "xv", "dq", "dk",
                                                                    "dv")) * m.layers
        d2h = (hb["xo"].numel() * 2 + hb["do"].numel() * 2) * m.layers
        ne = max(1, min(args.steps, 3))
        base = args.warmup + args.steps
        eevs = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)]
                 for _ in range(m.layers)] for _ in range(ne)]
        ef = 0.0
        dbb = 0.0
        torch.cuda.synchronize()
        barrier(world)
        for k in range(ne):
            sl = db.seq_len.copy() + 1
            p = run_step(ctx, base + k, ev=eevs[k], e2e=hb)
            Pl = p.plan.prefix_len.astype(np.int64)
            ef += extend_flops(Pl, p.plan.lengths - Pl, m.n_q_heads, m.head_dim) * m.layers
            dbb += decode_bytes(sl, m.n_kv_heads, m.head_dim) * m.layers
        torch.cuda.synchronize()
        e_ext = max_over_ranks(sum(e[l][0].elapsed_time(e[l][1]) for e in eevs
                                   for l in range(m.layers)), world)
        e_dec = max_over_ranks(sum(e[l][1].elapsed_time(e[l][2]) for e in eevs
                                   for l in range(m.layers)), world)
        link = host_link(hb["xq"])
        e2e = {"value": round(world * ef / (e_ext * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "decode_gbs": round(world * dbb / (e_dec * 1e-3) / 1e9, 1),
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": ne, "host_link": link,
               "note": "every layer's q/k_new/v_new (extend and decode) copied in from pinned "
                       "host memory and its outputs copied back, overlapped with the kernels "
                       "(two copy streams, double buffers); phases timed on the compute stream "
                       "including every wait for a copy, the last one until the last output "
                       "is on the host"}

    pk = peaks()
    traffic = stored_traffic()
    # decode: the bytes the stacked kernel must move (each fork group's shared context once),
    # the per-request count of the metric's definition kept as a labelled extra
    from prefix_cached_paged_gb300 import DEFAULT_KV_CHUNK
    G = m.n_q_heads // m.n_kv_heads
    uniq = sum(decode_unique_bytes(db.context_rows, db.context_len, sl, m.n_kv_heads,
                                   m.head_dim, 8 // G, args.kv_chunk or DEFAULT_KV_CHUNK)
               * m.layers for sl in seq_lens)
    # the kernels run for well under a second at a time: the burst peak applies
    ext_peak = pk["bf16_tflops"]
    # dominant kernel by time: decode (3 launches per call: plan, split-K main, merge)
    dom_is_decode = dec_ms >= ext_ms
    n_calls = args.steps * m.layers
    dec_call_ms = dec_ms / n_calls
    ext_call_ms = ext_ms / n_calls
    dec_uniq_gbs = uniq / n_calls / (dec_call_ms * 1e-3) / 1e9
    roof_dec = {"kernel": "decode_attention (plan + split-K main + merge)", "bound": "hbm",
                "achieved": round(dec_uniq_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(dec_uniq_gbs / pk["hbm_gbs"], 4),
                "traffic": traffic["decode"], "peak_source": pk["source"] + " hbm_gbs",
                "algorithmic_bytes": "unique: each fork group's shared context rows once, every "
                                     "request's own rows once (K, V of all KV heads + 4 B slot "
                                     "index per token)",
                "per_request_gbs": round(dec_gbs / world, 1),
                "per_request_note": "every request's context rows counted (L x 16388 B per "
                                    "layer); exceeds HBM because shared rows are read once"}
    if traffic["decode"]:
        roof_dec["dram_gbs"] = round(traffic["decode"] / (dec_call_ms * 1e-3) / 1e9, 1)
        roof_dec["dram_frac"] = round(roof_dec["dram_gbs"] / pk["hbm_gbs"], 4)
    per_launch_ext = ext_flops / n_calls
    roof_ext = {"kernel": "extend_attention", "bound": "tensor",
                "achieved": round(per_launch_ext / (ext_call_ms * 1e-3) / 1e12, 2),
                "peak": ext_peak, "unit": "TFLOP/s",
                "frac": round(per_launch_ext / (ext_call_ms * 1e-3) / 1e12 / ext_peak, 4),
                "traffic": traffic["extend"],
                "peak_source": pk["source"] + " bf16_tflops (burst)",
                "frac_of_sustained": round(per_launch_ext / (ext_call_ms * 1e-3) / 1e12
                                           / pk.get("bf16_tflops_sustained", ext_peak), 4)}
    cpu = cpu_baseline(ctx, args) if (rank == 0 and world == 1 and args.cpu_baseline) else None
    out = {
        "metric": METRIC, "value": round(ext_tflops, 2), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "fork_mixed_step", "layers": m.layers, "heads": "32x128 MHA",
                   "pool_slots": ctx["w"].pool_slots, "extend": "16 programs x 5 forks, P=1500, "
                   "S=200", "decode": "128 requests, ctx 512..8192 uniform",
                   "l2": "inputs larger than L2 (decode reads ~9 GB of KV per layer)",
                   "parallelism": f"replicas x{world}", "kv_chunk": args.kv_chunk or 512},
        "decode": {"unique_gbs": roof_dec["achieved"], "frac_of_hbm": roof_dec["frac"],
                   "per_request_gbs": round(dec_gbs, 1), "unit": "GB/s",
                   "dram_gbs": roof_dec.get("dram_gbs"), "dram_frac": roof_dec.get("dram_frac")},
        "prefill_tokens_skipped": {"skipped": skipped, "prompt_tokens": prompt,
                                   "hit_rate": round(skipped / max(prompt, 1), 4)},
        "evicted_tokens_per_step": int(np.mean([p.plan.evicted for p in plans])),
        "host_ms_per_step": round(1e3 * float(np.mean(host_t)), 3),
        "layers_ms_median": round(float(np.median(
            [e[0][0].elapsed_time(e[m.layers - 1][2]) for e in evs])), 3),
        "extend_ms_per_step": round(ext_ms / args.steps, 3),
        "decode_ms_per_step": round(dec_ms / args.steps, 3),
        "roofline": roof_dec if dom_is_decode else roof_ext,
        "roofline_extend": roof_ext, "roofline_decode": roof_dec,
        "clocks": clk, "gpu_launches": int(launches), "e2e": e2e,
        "cpu_baseline": cpu, "setup_s": round(ctx["setup_s"], 1),
    }
    return out


def host_link(pinned):
    """The host link the end-to-end leg goes through: NUMA nodes of the host, the GPU's node, and
    the copy rate of one contiguous pinned buffer (the e2e leg's own) each way."""
    import torch
    nodes = sorted(int(d[4:]) for d in os.listdir("/sys/devices/system/node")
                   if d.startswith("node") and d[4:].isdigit()) \
        if os.path.isdir("/sys/devices/system/node") else []
    gpu_node = None
    try:
        bus = subprocess.run(["nvidia-smi", "--query-gpu=pci.bus_id", "--format=csv,noheader",
                              f"--id={torch.cuda.current_device()}"], capture_output=True,
                             text=True, timeout=20).stdout.strip().lower()
        path = f"/sys/bus/pci/devices/{bus[4:] if len(bus.split(':')[0]) == 8 else bus}/numa_node"
        gpu_node = int(open(path).read().strip())
    except (OSError, ValueError, subprocess.SubprocessError):
        pass
    flat = pinned.view(-1)
    dev = torch.empty_like(flat, device="cuda")
    rates = {}
    for name, (dst, src) in (("h2d_gbs", (dev, flat)), ("d2h_gbs", (flat, dev))):
        for _ in range(2):
            dst.copy_(src, non_blocking=True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(5):
            dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        rates[name] = round(5 * flat.numel() * flat.element_size() / (e0.elapsed_time(e1) * 1e-3)
                            / 1e9, 1)
    del dev
    return {"numa_nodes": nodes, "gpu_numa_node": gpu_node, **rates,
            "bytes": int(flat.numel() * flat.element_size())}


def cpu_baseline(ctx, args, budget_s=None):
    """The oracle, as it stands, on a bounded sample of the step's extend units (fp64 attention
    of (request, layer, head) units on all host cores). Returns the metric in TFLOP/s."""
    import oracle
    import synth
    m = ctx["m"]
    seqs = ctx["ext0"]
    budget_s = args.cpu_budget if budget_s is None else budget_s
    threads = os.cpu_count() or 1
    rng = np.random.default_rng(7)
    units, flops = [], 0.0
    # one unit: a request's 200 queries of one head over 1700 keys; passes over the sample repeat
    # until the budget (10-30 s of CPU work by default) is spent
    n_units = threads * 8
    for _ in range(n_units):
        b, layer, h = (int(rng.integers(len(seqs))), int(rng.integers(m.layers)),
                       int(rng.integers(m.n_kv_heads)))
        s = seqs[b]
        hs = synth.prefix_hashes(m.seed, s)
        P = 1500
        q = synth.values(hs[P:], synth.TENSOR_Q, layer, [h], m.head_dim, m.dtype)
        k = synth.values(hs, synth.TENSOR_K, layer, [h], m.head_dim, m.dtype)
        v = synth.values(hs, synth.TENSOR_V, layer, [h], m.head_dim, m.dtype)
        units.append((q, k, v, P))
        flops += extend_flops([P], [len(s) - P], 1, m.head_dim)
    t0 = time.perf_counter()
    oracle.attention_units(units, m.sm_scale, 1, 1, threads)
    dt = time.perf_counter() - t0
    reps = 1
    while dt * (reps + 1) / reps < budget_s and reps < 256:
        t1 = time.perf_counter()
        oracle.attention_units(units, m.sm_scale, 1, 1, threads)
        dt += time.perf_counter() - t1
        reps += 1
    # the same oracle on one core, two units
    t1 = time.perf_counter()
    oracle.attention_units(units[:2], m.sm_scale, 1, 1, 1)
    one = time.perf_counter() - t1
    one_flops = flops * 2 / n_units
    return {"value": round(flops * reps / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "single_core_value": round(one_flops / one / 1e12, 6),
            "kind": "oracle",
            "sample": f"{n_units} extend units (request x layer x head: 200 queries over 1700 "
                      f"keys, fp64) of the fork mixed step, x{reps} passes, {dt:.1f} s"}


L2_FLUSH_BYTES = 512 << 20   # written between timed replays: larger than the 129 MB L2


def decode_unique_bytes(rows, ctx_len, seq_len, Hkv, d, group_size, chunk, elem=2):
    """Bytes decode must move at the least once requests that share a context prefix read it
    together (the stacked groups the engine forms): each group's shared rows once, every
    request's own rows once; K and V rows of all KV heads plus the 4-byte slot index per
    token. The per-request count (decode_bytes) charges shared rows once per request."""
    from prefix_cached_paged_gb300 import shared_context_groups
    row = 2 * Hkv * d * elem + 4
    indptr, members, shared = shared_context_groups(rows, ctx_len, group_size, chunk)
    L = np.asarray(seq_len, dtype=np.float64)
    total = float(L.sum())
    for g in range(len(shared)):
        mem = members[indptr[g]:indptr[g + 1]]
        total -= float(shared[g]) * (len(mem) - 1)
    return total * row


def _replay(name, steps, warmup, kv_chunk=0, stack="auto", local=0, flush=True):
    """Kernel replay on one of the single-phase workloads: the workload's setup phases run once
    through the engine, then the final batch's attention call (extend or decode) is timed
    `steps` times on the same inputs (idempotent: the same slots are rewritten), each call
    bracketed by CUDA events on the launching stream with a 512 MB write in between so that
    every call starts with nothing of its inputs in L2 (flush=True). Returns the record."""
    import torch
    import prefix_cached_paged_gb300 as rc
    import synth
    from synth import device as sdev
    from synth import workloads as W
    from tests import harness as H

    if name == "multi_turn_decode_unshared":
        w0 = W.multi_turn_decode()
        w = W.multi_turn_decode(shared=False, lengths=w0.notes["lengths"])
    elif name == "fork_extend_layer":
        fm = W.fork_mixed_step(layers=1)
        w = fm.workload
        w.phases = [W.Phase("cache", fm.programs), W.Phase("extend", fm.extend_seqs(0))]
    else:
        w = W.CONFIGS[name]()
    m = w.model
    stack_mode = {"auto": (True, 4), "off": (False, 4), "flat": (True, 1),
                  "always": ("always", 4), "always-flat": ("always", 1)}[stack]
    eng = H.make_engine(w, max_reqs=300, kv_chunk=kv_chunk, stack_extend=stack_mode[0],
                        stack_levels=stack_mode[1])
    for ph in w.phases[:-1]:
        if ph.kind == "cache":
            H.run_cache_phase(eng, m, ph.seqs, ph.keep_locked)
        else:
            H.run_extend_phase(eng, m, ph.seqs, keep_outputs=False)
    last = w.phases[-1]
    pk = peaks()
    if last.kind == "extend":
        b = eng.extend_begin(last.seqs)
        h = H.new_token_hashes(m, last.seqs, b.plan.prefix_len)
        q, k, v = H.dense_qkv(m, sdev.hashes_to_device(h), 0, b.num_tokens)
        o = torch.empty_like(q)
        run = lambda: eng.extend_layer(b, 0, q, k, v, o)
        Pl = b.plan.prefix_len.astype(np.int64)
        work = extend_flops(Pl, b.plan.lengths - Pl, m.n_q_heads, m.head_dim)
        unit, scale, bound = "TFLOP/s", 1e12, "tensor"
        peak, peak_src = pk["bf16_tflops"], pk["source"] + " bf16_tflops (burst)"
        kernel = "extend_attention"
        skipped = (int(Pl.sum()), int(b.plan.lengths.sum()))
        stacking = ("none" if b.stack is None else
                    {"groups_per_level": np.diff(b.stack[4]).tolist()})
        extra = {}
    else:
        seqs = last.seqs
        db = eng.decode_begin([s[:-1] for s in seqs])
        eng.decode_step(db)
        hh = np.array([synth.prefix_hashes(m.seed, s)[-1] for s in seqs], np.uint64)
        q, k, v = H.dense_qkv(m, sdev.hashes_to_device(hh), 0, len(seqs))
        o = torch.empty_like(q)
        mt = int(db.seq_len.sum())
        run = lambda: eng.decode_layer(db, 0, q, k, v, o, max_total_tokens=mt)
        per_request = decode_bytes(db.seq_len, m.n_kv_heads, m.head_dim)
        work = decode_unique_bytes(db.context_rows, db.context_len, db.seq_len, m.n_kv_heads,
                                   m.head_dim, 8 // m.group, kv_chunk or 512)
        unit, scale, bound = "GB/s", 1e9, "hbm"
        peak, peak_src = pk["hbm_gbs"], pk["source"] + " hbm_gbs"
        kernel = "decode_attention (plan + split-K main + merge)"
        skipped = (0, int(db.seq_len.sum()))
        stacking = {"shared_context_groups": int(db.num_groups)}
        extra = {"per_request_bytes": per_request, "unique_bytes": work}
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    launches0 = rc.launch_count()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for e0, e1 in evs:
        if flush:
            flush_buf.fill_(1.0)
        e0.record()
        run()
        e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert rc.device_status() == 0
    ms = float(np.mean([e0.elapsed_time(e1) for e0, e1 in evs]))
    val = work / (ms * 1e-3) / scale
    rec = {"value": round(val, 2), "unit": unit, "ms_per_step": round(ms, 4), "steps": steps,
           "warmup": warmup, "dtype": m.dtype,
           "config": {"workload": name, "mode": "kernel replay (same batch each step)",
                      "l2": ("flushed before every timed call (512 MB write)" if flush
                             else "not flushed between replays"),
                      "stack": stack, "stacking": stacking},
           "roofline": {"kernel": kernel, "bound": bound, "achieved": round(val, 2),
                        "peak": peak, "unit": unit, "frac": round(val / peak, 4),
                        "traffic": None, "peak_source": peak_src},
           "prefill_tokens_skipped": {"skipped": skipped[0], "prompt_tokens": skipped[1]},
           "clocks": clk, "gpu_launches": rc.launch_count() - launches0}
    if extra:
        rec["roofline"]["algorithmic_bytes"] = "unique: each shared context row once per group"
        rec["per_request_gbs"] = round(extra["per_request_bytes"] / (ms * 1e-3) / 1e9, 1)
        rec["per_request_note"] = ("every request's context rows counted (L x 4100 B); requests "
                                   "that share a prefix read it once, so this can exceed HBM")
    del flush_buf
    return rec


# the target configurations other than the fork step, each replayed on its own
CONFIG_REPLAYS = ("few_shot_extend", "two_level_extend", "multi_turn_decode",
                  "multi_turn_decode_unshared")


def bench_configs(args, local):
    """Replays of the other target configurations, appended to the fork step's line."""
    import gc
    import torch
    out = {}
    for name in CONFIG_REPLAYS:
        gc.collect()
        torch.cuda.empty_cache()
        out[name] = _replay(name, args.config_steps, 3, kv_chunk=args.kv_chunk, local=local)
    return out


def bench_replay(args, rank, world, local):
    """One kernel replay as the whole line (see _replay)."""
    rec = _replay(args.workload, args.steps, args.warmup, kv_chunk=args.kv_chunk,
                  stack=args.stack, local=local, flush=not args.no_flush)
    out = {"metric": METRIC, "value": rec["value"], "unit": rec["unit"], "n_gpus": world,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "data": "synthetic"}
    out.update(rec)
    return out


def _queue_batches(pq, policy, host_slots=0):
    """The batches the scheduler forms over the queue (host only; the engine's host cache makes
    the same decisions): [(request ids, matched lengths incl. tokens loaded from the host
    tier, tokens loaded)]."""
    from prefix_cached_paged_gb300.runtime import HostCache, WaitingQueue
    w = pq.workload
    hc = HostCache(w.pool_slots, w.max_ctx, w.pool_order, host_slots=host_slots)
    waiting = WaitingQueue(pq.seqs)
    out = []
    while len(waiting):
        idx = hc.schedule(waiting, pq.max_batch, pq.max_new_tokens, policy=policy)
        if not idx:
            raise RuntimeError("program queue: no request fits the pool")
        ids = [waiting.ids[i] for i in idx]
        p = hc.plan([pq.seqs[i] for i in ids])
        out.append((ids, p.prefix_len.copy(),
                    0 if p.host_len is None else int(p.host_len.sum())))
        hc.finish(p)
        waiting.remove(idx)
    return out


def _serve_queue(pq, policy, batches, inputs, overlap, host_slots=0, host_planes=None):
    """Serve the queue once through a fresh engine. overlap=False synchronises after every
    batch's kernels (host and GPU take turns); overlap=True never waits: the host schedules,
    plans and inserts batch k+1 while batch k's kernels run (stream order keeps the slots and
    slot-table rows that the host recycles safe). Returns host ms, tree ms, kernel ms (extend),
    wall ms, and the device time of the batches' begin work (slot table, host-tier copies)."""
    import torch
    from prefix_cached_paged_gb300.runtime import WaitingQueue
    from tests import harness as H
    m = pq.workload.model
    eng = H.make_engine(pq.workload, max_reqs=pq.max_batch + 8, host_tier_slots=host_slots,
                        host_planes=host_planes)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in batches]
    waiting = WaitingQueue(pq.seqs)
    host_s = 0.0
    torch.cuda.synchronize()
    tree0 = eng.host.host_seconds
    t_start = time.perf_counter()
    for k, (ids_ref, _, _) in enumerate(batches):
        t0 = time.perf_counter()
        idx = eng.host.schedule(waiting, pq.max_batch, pq.max_new_tokens, policy=policy)
        ids = [waiting.ids[i] for i in idx]
        assert ids == ids_ref
        evs[k][0].record()
        b = eng.extend_begin([pq.seqs[i] for i in ids])
        host_s += time.perf_counter() - t0
        q, kk, v, o = inputs[k]
        evs[k][1].record()
        for layer in range(m.layers):
            eng.extend_layer(b, layer, q, kk, v, o)
        evs[k][2].record()
        if not overlap:
            torch.cuda.synchronize()
        t0 = time.perf_counter()
        eng.extend_end(b)
        waiting.remove(idx)
        host_s += time.perf_counter() - t0
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_start
    gpu_ms = sum(e[1].elapsed_time(e[2]) for e in evs)
    begin_ms = sum(e[0].elapsed_time(e[1]) for e in evs)
    return host_s * 1e3, (eng.host.host_seconds - tree0) * 1e3, gpu_ms, wall * 1e3, begin_ms


def bench_queue(args, rank, world, local):
    """Cache-aware scheduling and host/GPU overlap on the program queue (32 attention layers):
    the whole queue served batch by batch through the engine (schedule -> plan + slot table ->
    extend kernels -> insert), one pass over the queue per step, a fresh engine each time.
      lspf / fcfs serial: longest-shared-prefix-first vs first-come-first-served, host and GPU
        taking turns (synchronised after every batch);
      lspf overlapped: the host runs ahead of the GPU (no synchronisation until the end);
      no_reuse overlapped: the same lengths with every prefix distinct, the tree's overhead
        when nothing is reused;
      fcfs_pool8k / fcfs_pool8k_host_tier: first-come-first-served behind an 8000-slot device
        pool (four prefixes), without and with a 50000-slot host tier in pinned host memory.
    Then the host tier's copy kernel alone: 16384 tokens x all layers spilled and loaded back.
    Timed: wall clock of the pass, the host calls (perf_counter; the tree and pool part
    separately) and each batch's kernels (CUDA events). The synthetic q / k / v of every batch
    are generated before the timed passes; every layer reads layer 0's values."""
    import torch
    import prefix_cached_paged_gb300 as rc
    from synth import device as sdev
    from synth import workloads as W
    from tests import harness as H

    L = args.layers
    HOST = 50_000
    cases = [("lspf", dict(), rc.RC_SCHED_LSPF, False, 0),
             ("fcfs", dict(), rc.RC_SCHED_FCFS, False, 0),
             ("lspf_overlapped", dict(), rc.RC_SCHED_LSPF, True, 0),
             ("no_reuse_overlapped", dict(shared=False), rc.RC_SCHED_LSPF, True, 0),
             ("fcfs_pool8k", dict(pool_slots=8_000), rc.RC_SCHED_FCFS, False, 0),
             ("fcfs_pool8k_host_tier", dict(pool_slots=8_000), rc.RC_SCHED_FCFS, False, HOST)]
    out = {}
    launches = 0
    m0 = W.program_queue(layers=L).workload.model
    dt = H.torch_dtype(m0.dtype)
    hshape = (L, HOST, m0.n_kv_heads, m0.head_dim)
    planes = (torch.empty(hshape, dtype=dt, pin_memory=True),
              torch.empty(hshape, dtype=dt, pin_memory=True))
    clocks = ClockSampler(local)
    clocks.start()
    for name, kw, policy, overlap, host_slots in cases:
        pq = W.program_queue(layers=L, **kw)
        m = pq.workload.model
        prompt = int(sum(len(s) for s in pq.seqs))
        batches = _queue_batches(pq, policy, host_slots)
        inputs, flops, computed = [], 0.0, 0
        loaded = sum(x[2] for x in batches)
        for ids, pl, _ in batches:
            seqs = [pq.seqs[i] for i in ids]
            h = H.new_token_hashes(m, seqs, pl)
            q, kk, v = H.dense_qkv(m, sdev.hashes_to_device(h), 0, len(h))
            inputs.append((q, kk, v, torch.empty_like(q)))
            Pl = pl.astype(np.int64)
            Ls = np.array([len(x) for x in seqs], np.int64)
            flops += extend_flops(Pl, Ls - Pl, m.n_q_heads, m.head_dim) * L
            computed += len(h)
        runs = []
        for rep in range(args.warmup + args.steps):
            l0 = rc.launch_count()
            r = _serve_queue(pq, policy, batches, inputs, overlap, host_slots,
                             planes if host_slots else None)
            assert rc.device_status() == 0
            if rep >= args.warmup:
                runs.append(r)
                launches += rc.launch_count() - l0
        host_ms, tree_ms, gpu_ms, wall_ms, begin_ms = (float(np.median([r[i] for r in runs]))
                                                       for i in range(5))
        out[name] = {"batches": len(batches), "computed_tokens": computed,
                     "hit_rate": round(1 - computed / prompt, 4),
                     "pool_slots": pq.workload.pool_slots, "host_tier_slots": host_slots,
                     "loaded_tokens": loaded, "begin_gpu_ms": round(begin_ms, 2),
                     "wall_ms": round(wall_ms, 2), "host_ms": round(host_ms, 2),
                     "tree_ms": round(tree_ms, 2), "kernel_ms": round(gpu_ms, 2),
                     "tree_frac_of_wall": round(tree_ms / wall_ms, 4),
                     "gpu_busy_frac": round(gpu_ms / wall_ms, 4),
                     "extend_tflops": round(flops / (gpu_ms * 1e-3) / 1e12, 1),
                     "prompt_tokens_per_s": round(prompt / (wall_ms * 1e-3), 1)}
        del inputs
        torch.cuda.empty_cache()
    # the host tier's copy kernel alone: spill 16384 tokens' rows of every layer to pinned host
    # memory, then load them back to other device slots
    n = 16_384
    dk = torch.empty((L, 20_000, m0.n_kv_heads, m0.head_dim), dtype=dt, device="cuda")
    dv = torch.empty_like(dk)
    g = np.random.default_rng(0)
    src = torch.from_numpy(g.choice(20_000, n, replace=False).astype(np.int32)).cuda()
    dst = torch.from_numpy(g.choice(20_000, n, replace=False).astype(np.int32)).cuda()
    hsl = torch.from_numpy(g.choice(HOST, n, replace=False).astype(np.int32)).cuda()
    nbytes = 2 * n * L * m0.n_kv_heads * m0.head_dim * dk.element_size()
    tier = {}
    for direction, args_ in (("spill_device_to_host", (dk, dv, src, planes[0], planes[1], hsl)),
                             ("load_host_to_device", (planes[0], planes[1], hsl, dk, dv, dst))):
        for _ in range(args.warmup):
            rc.kv_copy(*args_)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            rc.kv_copy(*args_)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        tier[direction] = {"gb_per_s": round(nbytes / (ms * 1e-3) / 1e9, 1),
                           "ms": round(ms, 3), "bytes": nbytes}
    # the link's own copy rate: one contiguous pinned <-> device copy of the same size
    # (cudaMemcpyAsync through torch), the roofline of the row copies above
    flat_h = planes[0].view(-1)[: nbytes // 2 // dk.element_size()]
    flat_d = dk.view(-1)[: flat_h.numel()]
    for direction, (dst_, src_) in (("spill_device_to_host", (flat_h, flat_d)),
                                    ("load_host_to_device", (flat_d, flat_h))):
        for _ in range(args.warmup):
            dst_.copy_(src_, non_blocking=True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            dst_.copy_(src_, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        link = flat_h.numel() * flat_h.element_size() / (ms * 1e-3) / 1e9
        tier[direction]["link_memcpy_gb_per_s"] = round(link, 1)
        tier[direction]["frac_of_link"] = round(tier[direction]["gb_per_s"] / link, 4)
    assert rc.device_status() == 0
    out["host_tier_copy"] = tier
    del dk, dv, planes
    clk = clocks.stop()
    pk = peaks()
    best = out["lspf_overlapped"]
    val = best["prompt_tokens_per_s"]
    pq = W.program_queue(layers=L)
    prompt = int(sum(len(s) for s in pq.seqs))
    return {"metric": METRIC, "value": val, "unit": "prompt tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": best["wall_ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": pq.workload.model.dtype, "data": "synthetic",
            "config": {"workload": "program_queue",
                       "queue": f"{int(pq.program.max()) + 1} programs x "
                                f"{len(pq.seqs) // (int(pq.program.max()) + 1)} questions, "
                                f"interleaved; {len(pq.seqs[0])} tokens each",
                       "pool_slots": pq.workload.pool_slots, "max_batch": pq.max_batch,
                       "max_new_tokens": pq.max_new_tokens, "layers": L,
                       "heads": "32x128 MHA",
                       "step": "the whole queue served once, fresh cache",
                       "value": "lspf_overlapped; ms_per_step its wall time",
                       "l2": "inputs larger than L2 (KV pool and per-batch q/k/v)"},
            "policies": out,
            "speedup_lspf_over_fcfs": round(out["lspf"]["prompt_tokens_per_s"]
                                            / out["fcfs"]["prompt_tokens_per_s"], 2),
            "roofline": {"kernel": "extend_attention (lspf batches)", "bound": "tensor",
                         "achieved": best["extend_tflops"], "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s",
                         "frac": round(best["extend_tflops"] / pk["bf16_tflops"], 4),
                         "traffic": None, "peak_source": pk["source"] + " bf16_tflops (burst)"},
            "prefill_tokens_skipped": {"skipped": prompt - best["computed_tokens"],
                                       "prompt_tokens": prompt},
            "clocks": clk, "gpu_launches": launches}


def bench_reference(args, rank, world):
    """The oracle timed on the host cores, same workload and metric, bounded sample per step."""
    if rank != 0:
        return None
    from synth import workloads as W
    fm = W.fork_mixed_step(layers=args.layers)
    ctx = {"m": fm.workload.model, "ext0": fm.extend_seqs(0)}
    vals = []
    per = max(2.0, args.ref_budget / max(args.steps + args.warmup, 1))
    t0 = time.perf_counter()
    for k in range(args.warmup + args.steps):
        r = cpu_baseline(ctx, args, budget_s=per)
        if k >= args.warmup:
            vals.append(r)
    total = time.perf_counter() - t0
    v = float(np.mean([r["value"] for r in vals]))
    return {"metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "impl": "reference",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * total / (args.warmup + args.steps), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "fork_mixed_step", "layers": args.layers},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "kind": "oracle",
                             "cores": vals[0]["cores"], "sample": vals[0]["sample"]},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--workload", default="fork_mixed_step",
                    choices=["fork_mixed_step", "tiny_extend", "few_shot_extend",
                             "two_level_extend", "multi_turn_decode",
                             "multi_turn_decode_unshared", "fork_extend_layer",
                             "program_queue", "tree_extend"],
                    help="fork_mixed_step = the full step; program_queue = the scheduler over a "
                         "request queue; the others replay one kernel")
    ap.add_argument("--kv-chunk", type=int, default=0)
    ap.add_argument("--stack", default="auto",
                    choices=["auto", "off", "flat", "always", "always-flat"],
                    help="extend prefix stacking in kernel replays: auto = the cost model over "
                         "up to 4 tree levels, flat = the cost model on the shallowest level "
                         "only, always = every group found")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the replays of the other target configurations after the fork "
                         "step")
    ap.add_argument("--config-steps", type=int, default=20,
                    help="timed calls per configuration replay")
    ap.add_argument("--no-flush", action="store_true",
                    help="kernel replays: do not flush L2 between timed calls")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=60.0)
    ap.add_argument("--write-traffic", metavar="NCU_CSV", default=None,
                    help="summarise an ncu capture of DRAM bytes into the traffic file and exit")
    ap.add_argument("--traffic-command", default="",
                    help="the command line the capture was taken with (recorded with it)")
    args = ap.parse_args()
    if args.write_traffic:
        write_traffic(args.write_traffic, args.traffic_command)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_init()
    if args.impl == "reference":
        out = bench_reference(args, rank, world)
    else:
        import __graft_entry__
        __graft_entry__.build()
        if args.workload == "fork_mixed_step":
            out = bench_ours(args, rank, world, local)
            if args.configs and world == 1:
                out["configs"] = bench_configs(args, local)
        elif args.workload == "program_queue":
            out = bench_queue(args, rank, world, local)
        else:
            out = bench_replay(args, rank, world, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
