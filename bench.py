#!/usr/bin/env python3
"""Benchmark of the speculative-decoding verify step on GB300.

One step = one verify round of the whole hot path over one batch of
synthetic logits: temperature softmax of the target and draft rows, the
accept/reject scan, the correction / bonus draw, tau, the outcome-prediction
keys (top-F of the draft rows and of the bonus draft row), the hit test and
the compaction of all rows' tokens.  On the default workload ("saguaro",
B=32, K=6, V=128256, bf16, T=0.7, fan-out 4,3,2,1,1,1,1) that is a single
fused sd_verify launch per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl reference]

Prints one JSON line (rank 0).  Timing: W untimed warm-up steps, then
exactly K steps between barrier + synchronize on both sides, CUDA events on
the launching stream, max over ranks.  The default run also measures every
config of the benchmark table (1 small, 2 peaked, 3 zipf, 4 saguaro, 5 mix)
into `per_config` (each with its own steps, clocks, roofline fraction, CPU
baseline sample and that sample's parity counts).  Inputs rotate over a pool of input
sets whose total exceeds 4x the L2 size, so no step reads logits a recent
step left in L2.  ``--impl reference`` times the CPU oracle on the host
cores instead (the reference arm).
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import sd_workloads as W  # noqa: E402

HEADLINE = "saguaro"
METRIC = "verify rounds/s"
UNIT = "rounds/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
KERNEL_DIR = os.path.join(ROOT, "speculative_decoding_verification_logits_gb300", "csrc")


def describe(name):
    s = W.WORKLOADS[name]
    d = f"{name}: B={s['B']} K={s['K']} V={s['V']} {s['dtype']} {s['kind']} T={s['temperature']}"
    if s.get("fanout"):
        d += f" fanout={','.join(map(str, s['fanout']))} + draft bonus row"
    if s.get("pack"):
        d += " + drafter pack of (1 + keys) blocks of K+1 tokens + KV rollback"
    return d


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.15)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4)
                          if r[i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "samples": len(rows),
                "reasons": reasons}


# ----------------------------------------------------------- helpers --------
def peaks():
    try:
        return json.load(open(PEAKS_FILE)), "measured"
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


TIMING_NOTE = ("CUDA events on the launching stream around exactly `steps` graph-replayed "
               "steps; barrier and device synchronisation before and after; one replay of "
               "untimed warm-up steps is queued right before the timed ones, so that they "
               "start on a busy GPU")

VERIFY_SOURCES = ("sd_device.cuh", "sd_split.cu", "sd_verify.cu")


def kernel_src_hash():
    """Hash of the code of the verify launches' CUDA sources (the profiled
    kernels), comments and blank space left out: a profile stays current
    while the code it measured does."""
    h = hashlib.sha256()
    for name in VERIFY_SOURCES:
        text = open(os.path.join(KERNEL_DIR, name), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch of the verify kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"sd_verify_kernel_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != kernel_src_hash():
        return None
    return float(m.group(1))


def launch_plan(call):
    """The launch plan the library took for `call` (run once, synchronised):
    with SDV_VERBOSE=1 it names it on stderr, read here at the descriptor
    level.  Returns the kernel launches of one verify round and the
    plan's name: 3 for the split launch (streaming grid, finish, packing), 2
    for the cluster kernel and the packing launch."""
    import tempfile
    old_env = os.environ.get("SDV_VERBOSE")
    os.environ["SDV_VERBOSE"] = "1"
    saved = os.dup(2)
    with tempfile.TemporaryFile(mode="w+b") as f:
        os.dup2(f.fileno(), 2)
        try:
            call()
            torch.cuda.synchronize()
        finally:
            os.dup2(saved, 2)
            os.close(saved)
            if old_env is None:
                del os.environ["SDV_VERBOSE"]
            else:
                os.environ["SDV_VERBOSE"] = old_env
        f.seek(0)
        text = f.read().decode(errors="replace")
    return (3, "split") if "sd_verify split:" in text else (2, "cluster")


def algorithmic_bytes(inp: W.Inputs) -> int:
    return W.logit_bytes(inp, algorithmic=True, with_bonus=inp.fanout is not None)


# ---------------------------------------------------------------- GPU arm ---
# the five benchmark workloads, in order (configs 1..5): the per-config object of the default run
CONFIGS = ["small", "peaked", "zipf", "saguaro", "mix"]


def l2_note(n_sets, set_bytes, l2):
    return (f"rotating {n_sets} input sets ({n_sets * set_bytes / 1e6:.0f} MB, "
            f"> 4x L2 {l2 / 1e6:.0f} MB)")


def pool_size(set_bytes, l2):
    """Input sets in the rotating pool: together more than 4x L2."""
    return max(2, int(np.ceil(4 * l2 / set_bytes)) + 1)


def config_of(name, ws_n, l2):
    """The `config` object of a workload's line (the same on both arms)."""
    s = W.WORKLOADS[name]
    B, K, V = s["B"], s["K"], s["V"]
    es = 2 if s["dtype"] == "bf16" else 4
    set_bytes = ((2 * K + 1) * V * B + (B * V if s.get("fanout") else 0)) * es
    n_sets = pool_size(set_bytes, l2)
    return {"workload": describe(name), "global_batch": B * ws_n, "seq_len": K + 1,
            "parallelism": f"replicas x{ws_n}" if ws_n > 1 else "single GPU",
            "l2": l2_note(n_sets, set_bytes, l2)}


def measure(name, steps, warmup, dev, rank, ws_n, e2e_steps=0):
    """Timed verify rounds of one workload on this GPU (graph-replayed, inputs
    rotating over a pool larger than 4x L2), and optionally the end-to-end
    rounds through host buffers.  Returns a dict; collective timing (max over
    ranks) when ws_n > 1."""
    import speculative_decoding_verification_logits_gb300 as sd
    spec = W.WORKLOADS[name]
    fan = spec.get("fanout")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    one = W.workload(name, round_idx=0, device=dev)
    set_bytes = W.logit_bytes(one, algorithmic=False, with_bonus=True)
    n_sets = pool_size(set_bytes, l2)
    pool = [one] + [W.workload(name, round_idx=i, device=dev) for i in range(1, n_sets)]
    B, K, V = one.B, one.K, one.V
    for p in pool:   # distinct uniforms per rank
        p.meta["row_base"] = rank * B
    outs = [sd.alloc_outputs(B, K, dev, hit=True, compact=True, n_keys=sum(fan) if fan else 0)
            for _ in range(n_sets)]
    stream = torch.cuda.Stream(dev)
    wss = sd.workspace(B, K, dev, stream)
    # The inputs and buffers above were made on the default stream; the
    # rounds run on `stream`.  Wait for all of it first: a conversion still
    # queued on the default stream could otherwise read a freed temporary
    # that the allocator has already handed out as an output buffer.
    torch.cuda.synchronize(dev)
    pack = "anchor" in one.meta   # the D3D workload also packs the drafter's next pass
    n_keys = sum(fan) if fan else 0
    packs = [(torch.empty((B, 1 + n_keys, K + 1), dtype=torch.int32, device=dev),
              torch.empty((B, 1 + n_keys, K + 1), dtype=torch.int32, device=dev),
              torch.empty((B, 1 + n_keys), dtype=torch.int32, device=dev))
             for _ in range(n_sets)] if pack else None
    rolls = [(torch.empty(B, dtype=torch.int32, device=dev),
              torch.empty(p_.meta["block_table"].numel(), dtype=torch.int32, device=dev),
              torch.empty(B + 1, dtype=torch.int32, device=dev))
             for p_ in pool] if pack else None

    def step(i):
        p = pool[i % n_sets]
        o = outs[i % n_sets]
        sd.verify(p.target, p.draft, p.tokens, p.temperature, p.seed + i // n_sets,
                  row_base=p.meta["row_base"], fanout=fan, draft_bonus=p.draft_bonus,
                  compact=True, out=o, ws=wss, stream=stream)
        if pack:
            sd.d3d_pack(o.keys, p.tokens, p.meta["anchor"], p.meta["anchor_pos"],
                        p.meta["mask_token"], out=packs[i % n_sets], stream=stream)
            # roll the target's KV cache back to the confirmed tokens (the
            # page table is reused from round to round: timing only)
            sd.kv_rollback(p.meta["block_table"], p.meta["kv_len"], o.tau, p.meta["page_size"],
                           K + 1, out=rolls[i % n_sets], stream=stream)

    with torch.cuda.stream(stream):
        n_launch, plan_name = launch_plan(lambda: step(0))
        n_launch += 2 if pack else 0
        for i in range(max(warmup, 3)):
            step(i)
    torch.cuda.synchronize(dev)

    # capture G steps per graph (launch-bound inner loop), replay to cover K
    G = min(steps, max(n_sets, (256 // n_sets) * n_sets))
    graphs = {}

    def graph_for(n):
        if n not in graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    step(i)
            graphs[n] = g
        return graphs[n]

    full, rem = divmod(steps, G)
    plan = [G] * full + ([rem] if rem else [])
    with torch.cuda.stream(stream):
        for n in set(plan):
            graph_for(n).replay()
    torch.cuda.synchronize(dev)

    def timed(fn, lead=None):
        if ws_n > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if lead is not None:   # untimed warm-up steps queued right ahead
            lead()
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1)
        if ws_n > 1:
            t = torch.tensor([ms], device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            ms = float(t.item())
        return ms

    def replay_all():
        with torch.cuda.stream(stream):   # replay on the stream the events are on
            for n in plan:
                graphs[n].replay()

    def lead_replay():
        # one more replay of untimed steps just before the timed ones, so
        # that these start on a busy GPU (as rounds do in a decode loop)
        # rather than after the idle gap of the synchronisation
        with torch.cuda.stream(stream):
            graphs[plan[0]].replay()

    with ClockSampler(dev.index) as clk:
        ms = timed(replay_all, lead_replay)
    clocks = clk.summary()

    # a verification pass on the last outputs of each set (cheap sanity)
    hit_rate = float(np.mean([o.hit.float().mean().item() for o in outs]))
    mean_tau = float(np.mean([o.tau.float().mean().item() for o in outs]))
    st = int(sum(o.status.item() for o in outs))

    # ---- end to end: inputs from pinned host memory, results back to host
    e2e = None
    if e2e_steps > 0:
        host = []
        for p in pool[:2]:
            hp = {}
            for k in ("target", "draft", "tokens", "temperature", "draft_bonus"):
                t = getattr(p, k)
                if t is not None:
                    hp[k] = t.cpu().pin_memory()
            if pack:
                hp["anchor"] = p.meta["anchor"].cpu().pin_memory()
                hp["anchor_pos"] = p.meta["anchor_pos"].cpu().pin_memory()
            host.append(hp)
        # two device copies of the inputs: step i's are copied on copy_stream
        # while step i - 1 verifies on `stream`
        dbufs = [{k: torch.empty_like(v, device=dev) for k, v in host[0].items()}
                 for _ in range(2)]
        copy_stream = torch.cuda.Stream(dev)
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        used = [torch.cuda.Event(), torch.cuda.Event()]
        torch.cuda.synchronize(dev)
        r_host = {"out_tokens": torch.empty((B, K + 1), dtype=torch.int32).pin_memory(),
                  "tau": torch.empty(B, dtype=torch.int32).pin_memory(),
                  "hit": torch.empty(B, dtype=torch.uint8).pin_memory(),
                  "offsets": torch.empty(B + 1, dtype=torch.int32).pin_memory(),
                  "packed": torch.empty(B * (K + 1), dtype=torch.int32).pin_memory()}
        h2d = sum(t.numel() * t.element_size() for t in host[0].values())
        d2h = sum(t.numel() * t.element_size() for t in r_host.values())
        out0 = outs[0]
        n_e2e = max(1, e2e_steps)

        # overlapped copies pay off once the link is the bound; for a few MB
        # per step the extra stream and event calls cost more host time
        overlap = h2d >= (8 << 20)

        def e2e_run():
            copy_stream.wait_stream(stream)
            for i in range(n_e2e):
                hp, dbuf = host[i % 2], dbufs[i % 2 if overlap else 0]
                if overlap:
                    with torch.cuda.stream(copy_stream):
                        if i >= 2:   # step i - 2 has finished reading this buffer
                            copy_stream.wait_event(used[i % 2])
                        for k, t in hp.items():
                            dbuf[k].copy_(t, non_blocking=True)
                        copied[i % 2].record(copy_stream)
                    stream.wait_event(copied[i % 2])
                else:
                    for k, t in hp.items():
                        dbuf[k].copy_(t, non_blocking=True)
                sd.verify(dbuf["target"], dbuf["draft"], dbuf["tokens"], dbuf["temperature"],
                          pool[0].seed + i, row_base=rank * B, fanout=fan,
                          draft_bonus=dbuf.get("draft_bonus"), compact=True, out=out0, ws=wss,
                          stream=stream)
                if pack:
                    sd.d3d_pack(out0.keys, dbuf["tokens"], dbuf["anchor"], dbuf["anchor_pos"],
                                pool[0].meta["mask_token"], out=packs[0], stream=stream)
                if overlap:
                    used[i % 2].record(stream)
                for k, t in r_host.items():
                    t.copy_(getattr(out0, k), non_blocking=True)
            stream.wait_stream(copy_stream)

        with torch.cuda.stream(stream):
            e2e_run()
            ms_e2e = timed(e2e_run)
        e2e = {"value": ws_n * n_e2e / (ms_e2e / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "copies": "overlapped with the previous step's verify" if overlap
                         else "in order with the verify"}

    # one round of set 0 with its first seed: the CPU baseline's oracle sample
    # runs on the same inputs, and its outputs are compared with these
    with torch.cuda.stream(stream):
        so = sd.verify(one.target, one.draft, one.tokens, one.temperature, one.seed,
                       row_base=one.meta["row_base"], fanout=fan, draft_bonus=one.draft_bonus,
                       compact=True, ws=wss, stream=stream)
    torch.cuda.synchronize(dev)
    sample = {k: getattr(so, k).cpu().numpy() for k in ("num_accepted", "out_tokens", "tau",
                                                        "hit") if getattr(so, k) is not None}
    if fan is not None:
        sample["keys"] = so.keys.cpu().numpy()
    alg = algorithmic_bytes(one)
    formula = W.logit_bytes(one, algorithmic=False, with_bonus=fan is not None)
    return dict(name=name, ms=ms, steps=steps, clocks=clocks, e2e=e2e, hit_rate=hit_rate,
                mean_tau=mean_tau, status=st, n_launch=n_launch, plan=plan_name, alg=alg,
                formula=formula, l2=l2, B=B, K=K, dtype=one.meta["dtype"], sample=sample)


def run_gpu(args):
    import speculative_decoding_verification_logits_gb300 as sd

    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    sd.lib()
    name = args.workload
    m = measure(name, args.steps, args.warmup, dev, rank, ws_n,
                e2e_steps=0 if args.no_e2e else min(args.steps, args.e2e_steps))
    # every benchmark workload measured in the same run (the default run only)
    per = {}
    if name == HEADLINE and not args.no_per_config:
        for c in CONFIGS:
            per[c] = m if c == name else measure(c, max(args.steps, args.config_steps),
                                                 args.warmup, dev, rank, ws_n)
    if ws_n > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return None

    pk, pk_kind = peaks()

    def roofline(mx):
        per_launch_ms = mx["ms"] / mx["steps"]
        achieved = mx["alg"] / (per_launch_ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "peak_source": pk_kind,
                "kernel": "verify step: all launches of one round (duration = step time)",
                "algorithmic_bytes_per_launch": mx["alg"],
                "formula_bytes_per_launch": mx["formula"]}

    rl = roofline(m)
    rl["traffic"] = profiled_traffic(name)
    line = {
        "metric": METRIC, "value": ws_n * m["steps"] / (m["ms"] / 1e3), "unit": UNIT,
        "n_gpus": ws_n, "steps": m["steps"], "warmup": args.warmup,
        "ms_per_step": m["ms"] / m["steps"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": m["dtype"],
        "data": "synthetic (seeded logits shaped like the workload; draft tokens drawn from q)",
        "config": config_of(name, ws_n, m["l2"]),
        "roofline": rl,
        # per step: the streaming grid, the finish and the packing launch
        # (split launch), or the cluster kernel and the packing launch
        "gpu_launches": m["n_launch"] * m["steps"],
        "clocks": m["clocks"],
        "e2e": m["e2e"],
        "hit_rate": m["hit_rate"], "mean_tau": m["mean_tau"], "status_bits": m["status"],
        "launch_plan": m["plan"],
        "timing": TIMING_NOTE,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"], line["parity_sample"] = cpu_baseline(name, args.cpu_seconds,
                                                                   m["sample"])
    if per:
        pc = {}
        for i, c in enumerate(CONFIGS):
            mc = per[c]
            r = roofline(mc)
            e = {"config": i + 1, "workload": describe(c),
                 "rounds_per_s": ws_n * mc["steps"] / (mc["ms"] / 1e3),
                 "ms_per_step": mc["ms"] / mc["steps"], "steps": mc["steps"],
                 "algorithmic_gbs": r["achieved"], "frac": r["frac"],
                 "algorithmic_bytes_per_step": mc["alg"], "launch_plan": mc["plan"],
                 "gpu_launches_per_step": mc["n_launch"], "clocks": mc["clocks"],
                 "mean_tau": mc["mean_tau"], "hit_rate": mc["hit_rate"],
                 "status_bits": mc["status"]}
            if not args.no_cpu_baseline:
                if c == name:
                    cb, ps = line["cpu_baseline"], line["parity_sample"]
                else:
                    cb, ps = cpu_baseline(c, args.config_cpu_seconds, mc["sample"])
                e["cpu_baseline"], e["parity_sample"] = cb, ps
            pc[c] = e
        line["per_config"] = pc
    return line


# ------------------------------------------------ n-gram drafting workload ---
def run_ngram(args):
    """Prompt-lookup drafting rounds (one sd_ngram_draft launch per round)
    over seeded histories; same timing rules as the verify workloads."""
    import speculative_decoding_verification_logits_gb300 as sd
    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    sd.lib()
    h0, lens, s = W.ngram_inputs(0, device=dev)
    B, L, K, V = s["B"], s["L"], s["K"], s["V"]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    set_bytes = h0.numel() * 4
    n_sets = max(2, int(np.ceil(4 * l2 / set_bytes)) + 1)
    pool = [h0] + [((h0.to(torch.int64) + 7919 * r) % V).to(torch.int32) for r in range(1, n_sets)]
    e = lambda *sh: torch.empty(sh, dtype=torch.int32, device=dev)
    outs = [(e(B, K), e(B), e(B), e(B)) for _ in range(n_sets)]
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)   # the pool is made on the default stream

    def step(i):
        sd.ngram_draft(pool[i % n_sets], lens, K, s["n_max"], s["n_min"], out=outs[i % n_sets],
                       stream=stream)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    torch.cuda.synchronize(dev)
    G = min(args.steps, max(n_sets, (256 // n_sets) * n_sets))
    graphs = {}
    full, rem = divmod(args.steps, G)
    plan = [G] * full + ([rem] if rem else [])
    for n in set(plan):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step(i)
        graphs[n] = g
    with torch.cuda.stream(stream):
        for n in set(plan):
            graphs[n].replay()
    torch.cuda.synchronize(dev)

    def timed(fn, lead=None):
        if ws_n > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if lead is not None:   # untimed warm-up steps queued right ahead
            lead()
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1)
        if ws_n > 1:
            t = torch.tensor([ms], device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            ms = float(t.item())
        return ms

    def replay_all():
        with torch.cuda.stream(stream):
            for n in plan:
                graphs[n].replay()

    def lead_replay():   # untimed steps right before the timed ones (see measure)
        with torch.cuda.stream(stream):
            graphs[plan[0]].replay()

    with ClockSampler(local) as clk:
        ms = timed(replay_all, lead_replay)
    clocks = clk.summary()
    # history bytes the backward scan must read: from each row's end back to
    # its match, or the whole row when nothing matches
    mp = outs[0][2].cpu().numpy()
    ln = lens.cpu().numpy()
    alg = int(4 * np.where(mp >= 0, ln - mp, ln).sum())
    e2e = None
    if not args.no_e2e:
        hh = [pool[0].cpu().pin_memory(), pool[1].cpu().pin_memory()]
        dh = torch.empty_like(pool[0])
        rh = [torch.empty((B, K), dtype=torch.int32).pin_memory(),
              torch.empty(B, dtype=torch.int32).pin_memory()]
        n_e2e = max(1, min(args.steps, args.e2e_steps))

        def e2e_steps():
            for i in range(n_e2e):
                dh.copy_(hh[i % 2], non_blocking=True)
                sd.ngram_draft(dh, lens, K, s["n_max"], s["n_min"], out=outs[0], stream=stream)
                rh[0].copy_(outs[0][0], non_blocking=True)
                rh[1].copy_(outs[0][1], non_blocking=True)

        with torch.cuda.stream(stream):
            e2e_steps()
            ms_e2e = timed(e2e_steps)
        e2e = {"value": ws_n * n_e2e / (ms_e2e / 1e3), "unit": UNIT, "steps": n_e2e,
               "h2d_bytes_per_step": hh[0].numel() * 4, "d2h_bytes_per_step": B * (K + 1) * 4}
    if ws_n > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return None
    pk, pk_kind = peaks()
    achieved = alg / (ms / args.steps / 1e3) / 1e9
    return {
        "metric": "n-gram drafting rounds/s", "value": ws_n * args.steps / (ms / 1e3),
        "unit": UNIT, "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32",
        "data": "synthetic (seeded phrase-book token histories)",
        "config": {"workload": f"ngram: B={B} L={L} (lengths {L // 4}..{L}) K={K} "
                               f"n={s['n_max']}..{s['n_min']}", "global_batch": B * ws_n,
                   "parallelism": f"replicas x{ws_n}" if ws_n > 1 else "single GPU",
                   "l2": f"rotating {n_sets} history sets ({n_sets * set_bytes / 1e6:.0f} MB, "
                         f"> 4x L2 {l2 / 1e6:.0f} MB)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"], "traffic": None, "peak_source": pk_kind,
                     "kernel": "sd_ngram_kernel (duration = step time)",
                     "algorithmic_bytes_per_launch": alg},
        "gpu_launches": args.steps, "clocks": clocks, "e2e": e2e, "timing": TIMING_NOTE,
        "match_rate": float((mp >= 0).mean()),
    }


# ------------------------------------------------------------- oracle arm ---
def _oracle_round(inp: W.Inputs, rows, threads):
    """The oracle on the given rows of one round: outcome prediction, verify
    (one row per call, in parallel threads), then compaction of the rows."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor

    t = W.to_numpy_logits(inp.target)
    d = W.to_numpy_logits(inp.draft)
    bonus = W.to_numpy_logits(inp.draft_bonus) if inp.draft_bonus is not None else None
    tok = inp.tokens.cpu().numpy()
    temps = inp.temperature.cpu().numpy()
    fan = inp.fanout

    def one(b):
        keys = None
        if fan is not None:
            keys = oracle.outcome_predict(d[b:b + 1], tok[b:b + 1], fan,
                                          None if bonus is None else bonus[b:b + 1])
        return oracle.verify(t[b:b + 1], d[b:b + 1], tok[b:b + 1], temps[b:b + 1], inp.seed,
                             row_base=int(b), keys=keys), keys

    with ThreadPoolExecutor(threads) as ex:
        pairs = list(ex.map(one, rows))
    res = [r for r, _ in pairs]
    keys = [k for _, k in pairs]
    out = np.concatenate([r["out_tokens"] for r in res])
    tau = np.concatenate([r["tau"] for r in res])
    oracle.compact(out, tau)
    if "anchor" in inp.meta:   # the D3D workload also packs the drafter's next pass
        idx = np.asarray(rows)
        oracle.d3d_pack(np.concatenate([k for _, k in pairs]), tok[idx],
                        inp.meta["anchor"].cpu().numpy()[idx],
                        inp.meta["anchor_pos"].cpu().numpy()[idx], inp.meta["mask_token"])
        oracle.kv_rollback(inp.meta["block_table"].cpu().numpy()[idx],
                           inp.meta["kv_len"].cpu().numpy()[idx], tau,
                           inp.meta["page_size"], inp.K + 1)
    return res, keys


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or ''."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "hardware")):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return ""


def _parity(res, keys, inp, gpu):
    """Row-by-row comparison of the oracle's results (rows 0..B-1 of the
    round, in order) with the GPU's for the same inputs: exact outside the
    guard band; guarded rows counted."""
    B, K = inp.B, inp.K
    temps = inp.temperature.cpu().numpy()
    c = dict(rows=B, positions=B * max(K, 1), sampled=0, guarded=0, guarded_mismatch=0,
             mismatch_outside_guard=0, keys_mismatch=0)
    for b in range(B):
        o = res[b]
        same = (int(o["tau"][0]) == int(gpu["tau"][b])
                and int(o["num_accepted"][0]) == int(gpu["num_accepted"][b])
                and np.array_equal(o["out_tokens"][0], gpu["out_tokens"][b]))
        if "hit" in gpu and inp.fanout is not None:
            same = same and int(o["hit"][0]) == int(gpu["hit"][b])
        sampled = temps[b] > 0
        c["sampled"] += int(sampled)
        guarded = sampled and int(o["guard_pos"][0]) >= 0
        c["guarded"] += int(guarded)
        if not same:
            c["guarded_mismatch" if guarded else "mismatch_outside_guard"] += 1
        if keys[b] is not None and "keys" in gpu:
            c["keys_mismatch"] += int(not np.array_equal(keys[b][0], gpu["keys"][b]))
    return c


def cpu_baseline(name, seconds, gpu_sample=None):
    """The oracle on a bounded sample of round 0 of the workload, on this
    host's cores (the reported CPU baseline).  The first pass runs every row
    of the round once, and its results are compared with the GPU's for the
    same inputs (`gpu_sample`), giving the parity counts."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    # the GPU's inputs (drawn on the device: its generator differs from the
    # host's), copied to the host by the oracle's marshalling
    dev = torch.device("cuda", torch.cuda.current_device()) if gpu_sample is not None else "cpu"
    inp = W.workload(name, round_idx=0, device=dev)
    B = inp.B
    # calibrate on one row (single thread), then size the sample to about
    # `seconds` of wall time on all cores, at least one pass over the round
    t0 = time.perf_counter()
    _oracle_round(inp, [0], 1)
    per_row = time.perf_counter() - t0
    n_rows = int(max(B, min(B * 50, seconds * cores / max(per_row, 1e-6))))
    rows = [i % B for i in range(n_rows)]
    t0 = time.perf_counter()
    res, keys = _oracle_round(inp, rows, cores)
    dt = time.perf_counter() - t0
    cb = {"value": (n_rows / B) / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
          "cpu": cpu_model(), "single_thread_ms_per_round": per_row * B * 1e3,
          "sample": f"{n_rows} rows ({n_rows / B:.2f} rounds) of {name}, one row per oracle "
                    f"call, {cores} threads; single-thread {per_row * 1e3:.1f} ms/row"}
    ps = _parity(res[:B], keys[:B], inp, gpu_sample) if gpu_sample is not None else None
    return cb, ps


def _l2_bytes():
    """L2 size of GPU 0 when one is visible (it names the rotation in
    `config`), else 0."""
    try:
        if torch.cuda.is_available():
            return torch.cuda.get_device_properties(0).L2_cache_size
    except Exception:
        pass
    return 0


def run_reference(args):
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    name = args.workload
    sharded = name == "vshard"   # the oracle computes the unsharded verify
    if sharded:
        name = HEADLINE
    cores = os.cpu_count() or 1
    if name == "ngram":   # the oracle's drafter over whole rounds, one thread
        h, lens, s = W.ngram_inputs(0)
        hn, ln = h.numpy(), lens.numpy()
        for _ in range(args.warmup):
            oracle.ngram_draft(hn, ln, s["K"], s["n_max"], s["n_min"])
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle.ngram_draft(hn, ln, s["K"], s["n_max"], s["n_min"])
        dt = time.perf_counter() - t0
        v = args.steps / dt
        return {"impl": "reference", "metric": "n-gram drafting rounds/s", "value": v,
                "unit": UNIT, "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
                "config": {"workload": "ngram", "global_batch": s["B"]},
                "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                                 "sample": "whole rounds, one thread"},
                "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
    inp = W.workload(name, round_idx=0, device="cpu")
    B = inp.B
    t0 = time.perf_counter()
    _oracle_round(inp, [0], 1)
    per_row = time.perf_counter() - t0
    # rows per step so that warm-up + steps end within ~3 minutes
    budget_rows = 180.0 * cores / max(per_row, 1e-6)
    rows_per_step = int(max(1, min(B, budget_rows / max(1, args.steps + args.warmup))))
    for i in range(args.warmup):
        _oracle_round(inp, [(i * rows_per_step + r) % B for r in range(rows_per_step)], cores)
    t0 = time.perf_counter()
    for i in range(args.steps):
        _oracle_round(inp, [(i * rows_per_step + r) % B for r in range(rows_per_step)], cores)
    dt = time.perf_counter() - t0
    rounds = args.steps * rows_per_step / B
    v = rounds / dt
    sample = (f"each step {rows_per_step} of {B} rows of {name} (one row per oracle call, "
              f"{cores} threads), scaled to rounds")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws_n,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": (vshard_config(args.shards, ws_n, _l2_bytes()) if sharded
                       else config_of(name, ws_n, _l2_bytes())),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "cpu": cpu_model(), "sample": sample,
                             "single_thread_ms_per_round": per_row * B * 1e3},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def vshard_config(S, ws_n, l2):
    """The `config` object of the sharded workload's line (both arms)."""
    c = config_of(HEADLINE, ws_n, l2)
    c["workload"] += f"; logits cut into {S} vocabulary shards, all on one GPU"
    c["shards"] = S
    return c


def run_vshard(args):
    """The vocabulary-sharded verify with every shard on this GPU: the
    headline workload's logits cut into S column blocks, each round the S
    shards' statistics, mass and pick launches in turn, the exchanges being
    the shards' blocks laid side by side.  Same timing rules as the other
    workloads; the oracle sample checks the outputs of one round."""
    import speculative_decoding_verification_logits_gb300 as sd
    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    sd.lib()
    name, S = HEADLINE, args.shards
    fan = W.WORKLOADS[name].get("fanout")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    one = W.workload(name, round_idx=0, device=dev)
    set_bytes = W.logit_bytes(one, algorithmic=False, with_bonus=True)
    n_sets = pool_size(set_bytes, l2)
    bounds = sd.vshard_bounds(one.V, S)

    def shards(x):
        return [x[..., a:a + n].contiguous() for a, n in bounds] if x is not None else None

    pool = []
    for i in range(n_sets):
        p = one if i == 0 else W.workload(name, round_idx=i, device=dev)
        pool.append((shards(p.target), shards(p.draft), p.tokens, p.temperature, p.seed,
                     shards(p.draft_bonus)))
    B, K, V = one.B, one.K, one.V
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)   # the pool is made on the default stream
    outs = [None] * n_sets

    def step(i):
        t, d, tok, temp, seed, bon = pool[i % n_sets]
        outs[i % n_sets] = sd.verify_vsharded(t, d, tok, temp, seed + i // n_sets, V=V,
                                              fanout=fan, draft_bonus=bon,
                                              row_base=rank * B, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    torch.cuda.synchronize(dev)
    G = min(args.steps, max(n_sets, (64 // n_sets) * n_sets))
    graphs = {}
    full, rem = divmod(args.steps, G)
    plan = [G] * full + ([rem] if rem else [])
    for n in set(plan):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step(i)
        graphs[n] = g
    with torch.cuda.stream(stream):
        for n in set(plan):
            graphs[n].replay()
    torch.cuda.synchronize(dev)

    def timed(fn, lead=None):
        if ws_n > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if lead is not None:   # untimed warm-up steps queued right ahead
            lead()
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1)
        if ws_n > 1:
            t = torch.tensor([ms], device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            ms = float(t.item())
        return ms

    def replay_all():
        with torch.cuda.stream(stream):
            for n in plan:
                graphs[n].replay()

    def lead_replay():   # untimed steps right before the timed ones (see measure)
        with torch.cuda.stream(stream):
            graphs[plan[0]].replay()

    with ClockSampler(local) as clk:
        ms = timed(replay_all, lead_replay)
    clocks = clk.summary()
    # one round of set 0 with its first seed, for the oracle's comparison
    t, d, tok, temp, seed, bon = pool[0]
    with torch.cuda.stream(stream):
        so = sd.verify_vsharded(t, d, tok, temp, seed, V=V, fanout=fan, draft_bonus=bon,
                                row_base=one.meta.get("row_base", 0), stream=stream)
    torch.cuda.synchronize(dev)
    sample = {k: getattr(so, k).cpu().numpy() for k in ("num_accepted", "out_tokens", "tau",
                                                        "hit", "keys")}
    status = int(so.status.item()) if so.status is not None else None
    if ws_n > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return None
    pk, pk_kind = peaks()
    alg = algorithmic_bytes(one)
    achieved = alg / (ms / args.steps / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": ws_n * args.steps / (ms / 1e3), "unit": UNIT,
        "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": one.meta["dtype"],
        "data": "synthetic (seeded logits shaped like the workload; draft tokens drawn from q)",
        "config": vshard_config(S, ws_n, l2),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": None,
                     "peak_source": pk_kind,
                     "kernel": "sharded verify step: all launches of one round "
                               "(duration = step time)",
                     "algorithmic_bytes_per_launch": alg},
        # per step: S statistics, S mass and S pick launches of this library
        "gpu_launches": 3 * S * args.steps, "clocks": clocks,
        "e2e": None, "status_bits": status,
        "launch_plan": f"sharded x{S} (stats, mass, pick per shard)",
        "timing": TIMING_NOTE,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"], line["parity_sample"] = cpu_baseline(name, args.cpu_seconds, sample)
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=HEADLINE, choices=W.ORDER + ["ngram", "vshard"])
    ap.add_argument("--shards", type=int, default=4,
                    help="vocabulary shards of the vshard workload (the headline's logits)")
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=400)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure the headline workload only (no per_config object)")
    ap.add_argument("--config-steps", type=int, default=500,
                    help="timed steps of each config in per_config (at least --steps)")
    ap.add_argument("--config-cpu-seconds", type=float, default=4.0,
                    help="oracle sample time of each config in per_config")
    args = ap.parse_args()
    if args.impl == "reference":
        line = run_reference(args)
    elif args.workload == "ngram":
        line = run_ngram(args)
    elif args.workload == "vshard":
        line = run_vshard(args)
    else:
        line = run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
