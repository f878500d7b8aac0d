"""Benchmark of the paged KV-cache hot path on GB300.

One step = one decode layer step of the GQA 8B-shape workload (bf16, 32 q /
8 kv heads, head_dim 128, block_size 128, batch 64, lognormal KV lengths):
slot mapping of the new token, its cache write, and paged decode attention
with split-KV and the merge.  Inputs stay resident in HBM; the K/V read per
step (~0.6 GB) is larger than L2, so no flush is needed between steps.

Printed: one JSON line (metric = achieved HBM GB/s of algorithmic bytes, plus
decode tokens/s, the roofline of the dominant kernel, the CPU oracle as a
reported baseline, and an end-to-end figure through the public API with host
buffers).  ``--impl reference`` times the CPU oracle on the same workload.

Multi-GPU (torchrun): every rank runs an independent replica of the
workload (the path shards by sequence with no exchange), timing is the max
over ranks, value is the sum of all ranks' work.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

# The oracle baseline is reported per core: keep NumPy's BLAS single-threaded.
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from synth import CONFIGS, decode_case, make_config  # noqa: E402

WORKLOAD = "gqa8b_decode"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    """(HBM GB/s, kind): the measured copy bandwidth, else the fallback figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """(dense bf16 TFLOP/s burst, kind) for a kernel timed on its own."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def decode_bytes(seq_lens, Hq, Hkv, D, bs, elt=2):
    """Algorithmic bytes of one paged decode: K/V rows attended, Q, O, table, lengths."""
    toks = int(sum(int(x) for x in seq_lens))
    blocks = sum(-(-int(x) // bs) for x in seq_lens)
    B = len(seq_lens)
    return toks * Hkv * D * 2 * elt + 2 * B * Hq * D * elt + 4 * blocks + 4 * B


def write_bytes(B, Hkv, D, elt=2):
    """New K/V rows read + written into the cache, plus slot ints written and read."""
    return 2 * (2 * B * Hkv * D * elt) + 3 * 4 * B


DECODE_METRIC = "paged decode achieved HBM GB/s (algorithmic bytes) and decode tokens/s"


def decode_workload(name, case, ws):
    """(config dict, decode bytes, step bytes) of a decode workload; both arms print this config."""
    m = case.meta
    B = case.q.shape[0]
    lens = case.seq_lens.tolist()
    d_bytes = decode_bytes(lens, m["num_q_heads"], m["num_kv_heads"], m["head_dim"],
                           case.block_size)
    step_bytes = d_bytes + write_bytes(B, m["num_kv_heads"], m["head_dim"])
    config = {
        "workload": CONFIGS[name]["about"],
        "batch": B, "num_q_heads": m["num_q_heads"], "num_kv_heads": m["num_kv_heads"],
        "head_dim": m["head_dim"], "block_size": case.block_size,
        "kv_tokens": int(sum(lens)), "step": "slot mapping + cache write + paged decode "
        "(split-KV, fused merge) in one launch (kvc_paged_decode_append); consecutive steps "
        "replayed from one CUDA graph", "algorithmic_bytes_per_step": step_bytes,
        "l2": "no flush: each step reads %.0f MB of K/V, more than the 129 MB L2" % (d_bytes / 1e6),
        "parallelism": f"replicas x{ws}",
    }
    return config, d_bytes, step_bytes


def kernel_source_digest():
    h = hashlib.sha256()
    for name in ("paged_decode.cu", "kvc_device.cuh", "api.cu"):  # api.cu: tensor-map encoding
        with open(os.path.join(ROOT, "paged_kv_cache_135_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


TRAFFIC_RECORD = "traffic.json"


def recorded_traffic(key, digest):
    """DRAM bytes per launch recorded by ncu (profiles/traffic.json, entry `key`), if the
    record was taken on this kernel source (same digest); else None."""
    try:
        with open(os.path.join(ROOT, "profiles", TRAFFIC_RECORD)) as f:
            rec = json.load(f).get(key)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("kernel_source_digest") != digest:
        return None
    return float(rec["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


class DecodeStep:
    """Device-resident decode-layer step through the public API."""

    def __init__(self, kvc, case, device):
        self.kvc = kvc
        self.case = case
        dv = device
        self.q = case.q.to(dv)
        self.kc = case.key_cache.to(dv)
        self.vc = case.value_cache.to(dv)
        self.bt = case.block_table.to(dv)
        self.sl = case.seq_lens.to(dv)
        self.nk = case.new_key.to(dv)
        self.nv = case.new_value.to(dv)
        self.wp = case.write_pos.to(dv)
        self.out = torch.empty_like(self.q)
        self.slots = torch.empty(self.q.shape[0], dtype=torch.int32, device=dv)
        m = case.meta
        self.Hq, self.Hkv, self.D = m["num_q_heads"], m["num_kv_heads"], m["head_dim"]
        n = kvc.decode_workspace_size(self.Hq, self.Hkv, self.D)
        self.ws = torch.zeros(max(n, 16), dtype=torch.uint8, device=dv)
        self.nb = self.kc.shape[0]

    def write(self):
        k = self.kvc
        k.build_slot_mapping(self.bt, self.case.block_size, self.wp, self.nb, out=self.slots)
        k.reshape_and_cache(self.nk, self.nv, self.kc, self.vc, self.slots)

    def decode(self):
        self.kvc.paged_decode(self.q, self.kc, self.vc, self.bt, self.sl, self.case.scale,
                              out=self.out, workspace=self.ws)

    def step(self):
        """The whole step in one launch: slot mapping, new-token write, decode."""
        self.kvc.paged_decode_append(self.q, self.nk, self.nv, self.kc, self.vc, self.bt,
                                     self.sl, self.case.scale, out=self.out,
                                     slot_mapping=self.slots, workspace=self.ws)

    LAUNCHES = 1  # kvc_paged_decode_append: slot mapping, cache write, decode, split merge


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, device):
    """The largest x over all ranks of the job (x itself on one rank): every timing
    is the slowest replica's."""
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_oracle_rate(case, budget_s=10.0):
    """Time the oracle on the workload's sequences, in order and wrapping around, until
    about budget_s of oracle time has elapsed."""
    from oracle import kvc_oracle as O
    m = case.meta
    bs = case.block_size
    done_bytes, t_total, n_seq = 0, 0.0, 0
    B = case.q.shape[0]
    for i in range(1000 * B):
        b = i % B
        L = int(case.seq_lens[b])
        nblk = max(1, -(-L // bs))
        ids = case.block_table[b, :nblk].long()
        k = case.key_cache[ids.to(case.key_cache.device)].double().cpu().numpy()
        v = case.value_cache[ids.to(case.value_cache.device)].double().cpu().numpy()
        q = case.q[b:b + 1].double().cpu().numpy()
        table = np.arange(nblk)[None]
        t0 = time.perf_counter()
        O.paged_decode(q, k, v, table, [L], case.scale)
        t_total += time.perf_counter() - t0
        done_bytes += decode_bytes([L], m["num_q_heads"], m["num_kv_heads"], m["head_dim"], bs)
        n_seq += 1
        if t_total > budget_s:
            break
    return done_bytes / t_total / 1e9, n_seq, B, t_total


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def cpu_oracle_rate_all_cores(case, budget_s=10.0):
    """The oracle on every host core: one spawned worker process per core (single-threaded
    BLAS each) evaluating whole sequences, inputs memory-mapped; passes over the workload's
    sequences until about budget_s of wall time.  Returns (GB/s, evaluations, workers, s)."""
    from oracle.pool import OraclePool
    m = case.meta
    bs, B = case.block_size, case.q.shape[0]
    kb, vb, lens = [], [], []
    for b in range(B):
        L = int(case.seq_lens[b])
        nblk = max(1, -(-L // bs))
        ids = case.block_table[b, :nblk].long()
        kb.append(case.key_cache[ids.to(case.key_cache.device)].view(torch.int16).cpu().numpy())
        vb.append(case.value_cache[ids.to(case.value_cache.device)].view(torch.int16).cpu().numpy())
        lens.append(L)
    workers = os.cpu_count() or 1
    pool = OraclePool(kb, vb, case.q.view(torch.int16).cpu().numpy(), lens, case.dtype, workers)
    try:
        pool.run(range(min(B, workers)), case.scale)          # workers up, pages mapped
        per = [decode_bytes([L], m["num_q_heads"], m["num_kv_heads"], m["head_dim"], bs)
               for L in lens]
        done, t, passes = 0, 0.0, 0
        while t < budget_s and passes < 1000:
            t += pool.run(range(B), case.scale)
            done += sum(per)
            passes += 1
    finally:
        pool.close()
    return done / t / 1e9, passes * B, workers, t


def cpu_baseline(case):
    """The oracle timed on this host: all cores (the reported value) and one core, plus one
    core on the tiny and Llama-7B-shape decode workloads (a bounded sample of each)."""
    gbs1, n1, B, t1 = cpu_oracle_rate(case)
    gbs, n, workers, t = cpu_oracle_rate_all_cores(case)
    others = {}
    for name, budget in (("tiny_decode", 1.0), ("llama7b_mha_decode", 4.0)):
        g, k, _, tt = cpu_oracle_rate(make_config(name, seed=0), budget_s=budget)
        others[name] = {"value": g, "unit": "GB/s", "cores": 1,
                        "sample": f"{k} sequence evaluations, {tt:.1f} s"}
    return {"value": gbs, "unit": "GB/s", "cores": workers, "kind": "oracle",
            "sample": f"{n} sequence evaluations ({n // B} passes over the {B} sequences) "
                      f"spread over {workers} spawned single-threaded worker processes, fp64 "
                      f"NumPy oracle, {t:.1f} s wall",
            "single_core": {"value": gbs1, "unit": "GB/s", "cores": 1,
                            "sample": f"{n1} sequence evaluations, {t1:.1f} s"},
            "single_core_other_workloads": others,
            "cpu_count": os.cpu_count(), "cpu_model": cpu_model(), "blas_threads_per_worker": 1}


def run_reference(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    case = make_config(WORKLOAD, seed=0)
    # About 90 s of oracle time over the whole run, so it ends within a few minutes
    # at any --steps/--warmup; a step evaluates at least one sequence.
    budget = max(0.05, min(20.0, 90.0 / max(1, args.steps + args.warmup)))
    vals = []
    for i in range(args.warmup + args.steps):
        gbs, n_seq, B, t = cpu_oracle_rate(case, budget_s=budget)
        if i >= args.warmup:
            vals.append((gbs, n_seq, t))
    value = statistics.median(v[0] for v in vals)
    n_seq = vals[0][1]
    print(json.dumps({
        "impl": "reference", "metric": DECODE_METRIC,
        "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(v[2] for v in vals),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": decode_workload(WORKLOAD, case, ws)[0],
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n_seq} sequence evaluations per step, the workload's "
                                   f"{B} sequences in order, wrapping (fp64 NumPy oracle)"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def time_graphs(graphs, steps):
    """Replay each graph in turn `steps` times; events around each replay.

    Returns (total ms, {name: mean ms per replay})."""
    stream = torch.cuda.current_stream()
    evs = {n: [] for n, _ in graphs}
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(steps):
        for n, g in graphs:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            evs[n].append((a, b))
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1), {n: statistics.mean(a.elapsed_time(b) for a, b in v)
                                 for n, v in evs.items()}


def capture(fn):
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            fn()
    torch.cuda.current_stream().wait_stream(cap)
    return g


def steps_per_graph(steps, cap=10):
    """Steps captured per CUDA graph replay: the largest divisor of `steps` up to `cap`,
    so the timed region is exactly `steps` steps."""
    return max(d for d in range(1, cap + 1) if steps % d == 0)


def prefill_flops(lens, ctx, Hq, D):
    """Causal attention FLOPs: 4 * Hq * D per (query, visible key) pair."""
    pairs = sum(c * n + n * (n + 1) // 2 for n, c in zip(lens, ctx))
    return 4 * Hq * D * pairs


def _roofline(name, ms, work, unit, peak, peak_kind, clocks, **extra):
    """A secondary figure: the kernel's mean time per launch and its roofline fraction."""
    achieved = work / (ms * 1e-3) / (1e9 if unit == "GB/s" else 1e12)
    d = {"kernel": name, "avg_launch_ms": ms, "achieved": achieved, "unit": unit,
         "peak": peak, "peak_kind": peak_kind, "frac": achieved / peak,
         ("algorithmic_bytes" if unit == "GB/s" else "algorithmic_flops"): work,
         "clocks": clocks}
    d.update(extra)
    return d


def measure_mixed(kvc, dev, rank, steps, warmup):
    """Mixed packed batch (one stream): packed slot mapping + prefill, then the 128-sequence
    decode step.  Returns (prefill figure, decode figure, ms per whole step)."""
    pre, dec = make_config("mixed_packed", seed=rank, value_device=str(dev))
    m = pre.meta
    Hq, Hkv, D, bs = m["num_q_heads"], m["num_kv_heads"], m["head_dim"], pre.block_size
    P = {k: getattr(pre, k).to(dev) for k in ("q", "key", "value", "cu_seqlens", "context_lens",
                                               "block_table")}
    kc, vc = pre.key_cache, pre.value_cache          # one pool shared by both halves
    T = pre.q.shape[0]
    pslots = torch.empty(T, dtype=torch.int32, device=dev)
    pout = torch.empty_like(P["q"])
    dec.key_cache, dec.value_cache = kc, vc
    step = DecodeStep(kvc, dec, dev)

    def prefill():
        kvc.build_slot_mapping(P["block_table"], bs, P["context_lens"], kc.shape[0],
                               cu_seqlens=P["cu_seqlens"], num_tokens=T, out=pslots)
        # the 16 prompts have no cached context: context_lens None (write fused into attention)
        kvc.varlen_prefill_paged(P["q"], P["key"], P["value"], P["cu_seqlens"], pslots,
                                 P["block_table"], kc, vc, pre.scale, pre.max_seqlen_q,
                                 context_lens=None, out=pout)

    for _ in range(warmup):
        prefill()
        step.step()
    torch.cuda.synchronize()
    graphs = [("prefill", capture(prefill)), ("decode", capture(step.step))]
    for _ in range(warmup):
        for _, g in graphs:
            g.replay()
    with ClockSampler(dev.index or 0) as clk:
        total_ms, per = time_graphs(graphs, steps)
    lens = pre.meta["lens"]
    flops = prefill_flops(lens, [0] * len(lens), Hq, D)
    d_lens = dec.seq_lens.tolist()
    d_bytes = decode_bytes(d_lens, Hq, Hkv, D, bs) + write_bytes(len(d_lens), Hkv, D)
    tp, tkind = tensor_peak()
    hp, hkind = peaks()
    clocks = clk.summary()
    pf = _roofline("prefill_tc2_kernel (kvc_varlen_prefill_paged: packed slot mapping, then the "
                   "cache write fused into the causal attention)", per["prefill"], flops, "TFLOP/s",
                   tp, tkind, clocks,
                   tokens=T, bound="tensor")
    dc = _roofline("paged_decode_kernel (kvc_paged_decode_append, 128 sequences on the shared "
                   "pool)", per["decode"], d_bytes, "GB/s", hp, hkind, clocks, bound="hbm")
    del P, kc, vc, pre, dec, step, graphs
    return pf, dc, total_ms / steps


def measure_mla(kvc, dev, rank, steps, warmup):
    """MLA decode step: latent write of the new token, then MLA decode."""
    c = make_config("mla_decode", seed=rank, value_device=str(dev))
    d = {k: getattr(c, k).to(dev) for k in ("q_nope", "q_rope", "cache_nope", "cache_rope",
                                             "block_table", "seq_lens", "new_nope", "new_rope",
                                             "write_pos")}
    B = c.q_nope.shape[0]
    slots = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty_like(d["q_nope"])
    ws = torch.zeros(max(kvc.mla_workspace_size(), 16), dtype=torch.uint8, device=dev)

    def step():  # latent write of the new token and MLA decode, one call
        kvc.mla_paged_decode_append(d["q_nope"], d["q_rope"], d["new_nope"], d["new_rope"],
                                    d["cache_nope"], d["cache_rope"], d["block_table"],
                                    d["seq_lens"], c.scale, out=out, slot_mapping=slots,
                                    workspace=ws)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    graphs = [("decode", capture(step))]
    for _ in range(warmup):
        for _, g in graphs:
            g.replay()
    with ClockSampler(dev.index or 0) as clk:
        total_ms, per = time_graphs(graphs, steps)
    lens = c.seq_lens.tolist()
    toks = sum(lens)
    by = toks * 576 * 2 + B * 128 * (576 + 512) * 2 + \
        4 * sum(-(-x // c.block_size) for x in lens) + 4 * B
    flops = toks * 128 * (2 * 576 + 2 * 512)
    hp, hkind = peaks()
    tp, tkind = tensor_peak()
    by += B * 576 * 2 * 2 + 4 * B          # the new latent rows read and written, slots
    fig = _roofline("mla_decode_kernel + mla_merge_kernel (kvc_mla_paged_decode_append: latent "
                    "write of the new token and MLA decode in one call)", per["decode"],
                    by, "GB/s", hp, hkind, clk.summary(), bound="hbm",
                    tflops=flops / (per["decode"] * 1e-3) / 1e12, tensor_peak=tp,
                    tensor_frac=flops / (per["decode"] * 1e-3) / 1e12 / tp,
                    ms_per_step=total_ms / steps, tokens_per_s=B / (total_ms / steps * 1e-3))
    del d, out, ws, c, graphs
    return fig


def measure_decode(kvc, dev, rank, name, steps, warmup):
    """A decode workload's one-launch step (kvc_paged_decode_append), graph-replayed."""
    case = make_config(name, seed=rank, value_device=str(dev))
    m = case.meta
    step = DecodeStep(kvc, case, dev)
    for _ in range(warmup):
        step.step()
    torch.cuda.synchronize()
    graphs = [("step", capture(step.step))]
    for _ in range(warmup):
        graphs[0][1].replay()
    with ClockSampler(dev.index or 0) as clk:
        _, per = time_graphs(graphs, steps)
    lens = case.seq_lens.tolist()
    by = decode_bytes(lens, m["num_q_heads"], m["num_kv_heads"], m["head_dim"],
                      case.block_size) + write_bytes(len(lens), m["num_kv_heads"], m["head_dim"])
    hp, hkind = peaks()
    fig = _roofline("paged_decode_kernel (kvc_paged_decode_append)", per["step"], by, "GB/s", hp,
                    hkind, clk.summary(), bound="hbm", workload=CONFIGS[name]["about"])
    del step, case, graphs
    return fig


def launch_percentiles(ms):
    """p10, median and p90 of per-launch times (each replay's mean over its launches)."""
    q = np.percentile(np.asarray(ms, dtype=np.float64), [10, 50, 90])
    return [float(x) for x in q]


def measure_block_sizes(kvc, dev, rank, steps, warmup, sizes=(16, 64, 128)):
    """The GQA 8B-shape decode step at block sizes 16, 64 and 128: the same lengths (drawn
    first from the same seed), the same pool of 524,288 token slots, a block table per size."""
    c = CONFIGS[WORKLOAD]
    slots = c["num_blocks"] * c["block_size"]
    max_tokens = c["max_blocks_per_seq"] * c["block_size"]
    out = {}
    for bs in sizes:
        case = decode_case(rank, c["batch"], c["lens"], c["num_q_heads"], c["num_kv_heads"],
                           c["head_dim"], bs, slots // bs, max_tokens // bs, c["dtype"],
                           c["scale"], value_device=str(dev))
        step = DecodeStep(kvc, case, dev)
        for _ in range(warmup):
            step.step()
        torch.cuda.synchronize()
        graphs = [("step", capture(step.step))]
        for _ in range(warmup):
            graphs[0][1].replay()
        with ClockSampler(dev.index or 0) as clk:
            _, per = time_graphs(graphs, steps)
        lens = case.seq_lens.tolist()
        by = decode_bytes(lens, c["num_q_heads"], c["num_kv_heads"], c["head_dim"], bs) + \
            write_bytes(len(lens), c["num_kv_heads"], c["head_dim"])
        hp, hkind = peaks()
        out[f"block_size_{bs}"] = _roofline("paged_decode_kernel (kvc_paged_decode_append)",
                                            per["step"], by, "GB/s", hp, hkind, clk.summary(),
                                            bound="hbm")
        del step, case, graphs
        torch.cuda.empty_cache()
    return out


def int8_decode_bytes(seq_lens, Hq, Hkv, D, bs):
    """Algorithmic bytes of one INT8-cache decode: codes and fp32 scales of the K/V rows
    attended, Q and O (16-bit), table entries, lengths."""
    toks = int(sum(int(x) for x in seq_lens))
    blocks = sum(-(-int(x) // bs) for x in seq_lens)
    B = len(seq_lens)
    return toks * Hkv * (D + 4) * 2 + 2 * B * Hq * D * 2 + 4 * blocks + 4 * B


def int8_write_bytes(B, Hkv, D):
    """The INT8 step's write: new 16-bit K/V rows read, their codes and fp32 scales written,
    slot ints written."""
    return 2 * B * Hkv * D * 2 + 2 * B * Hkv * (D + 4) + 4 * B


def measure_int8(kvc, dev, rank, steps, warmup):
    """The GQA 8B-shape decode step over an INT8 cache (codes + one fp32 scale per row): the
    new token's rows quantised into the cache and the decode, one kvc_paged_decode_int8_append
    launch."""
    case = make_config(WORKLOAD, seed=rank, value_device=str(dev))
    m = case.meta
    Hq, Hkv, D, bs = m["num_q_heads"], m["num_kv_heads"], m["head_dim"], case.block_size
    NB = case.key_cache.shape[0]
    codes = [torch.empty(NB, bs, Hkv, D, dtype=torch.int8, device=dev) for _ in range(2)]
    scales = [torch.empty(NB, Hkv, bs, dtype=torch.float32, device=dev) for _ in range(2)]
    # quantise the whole pool once with the library's own write (every slot in order)
    allslots = torch.arange(NB * bs, dtype=torch.int32, device=dev)
    kvc.reshape_and_cache_int8(case.key_cache.view(NB * bs, Hkv, D),
                               case.value_cache.view(NB * bs, Hkv, D), codes[0], codes[1],
                               scales[0], scales[1], allslots)
    del case.key_cache, case.value_cache
    q, bt, sl = case.q.to(dev), case.block_table.to(dev), case.seq_lens.to(dev)
    nk, nv = case.new_key.to(dev), case.new_value.to(dev)
    out = torch.empty_like(q)
    slots = torch.empty(q.shape[0], dtype=torch.int32, device=dev)
    ws = torch.zeros(max(kvc.decode_workspace_size(Hq, Hkv, D), 16), dtype=torch.uint8,
                     device=dev)

    def decode():
        kvc.paged_decode_int8_append(q, nk, nv, codes[0], codes[1], scales[0], scales[1], bt, sl,
                                     case.scale, out=out, slot_mapping=slots, workspace=ws)

    for _ in range(warmup):
        decode()
    torch.cuda.synchronize()
    graphs = [("decode", capture(decode))]
    for _ in range(warmup):
        graphs[0][1].replay()
    with ClockSampler(dev.index or 0) as clk:
        _, per = time_graphs(graphs, steps)
    lens = case.seq_lens.tolist()
    B = len(lens)
    by = int8_decode_bytes(lens, Hq, Hkv, D, bs) + int8_write_bytes(B, Hkv, D)
    hp, hkind = peaks()
    fig = _roofline("paged_decode_kernel, INT8 cache (kvc_paged_decode_int8_append: quantising "
                    "write of the new token, decode and split-KV merge in one launch)",
                    per["decode"], by, "GB/s", hp, hkind, clk.summary(), bound="hbm",
                    bytes_vs_16bit=by / (decode_bytes(lens, Hq, Hkv, D, bs) +
                                         write_bytes(B, Hkv, D)),
                    traffic=recorded_traffic("paged_decode_kernel_int8/" + WORKLOAD,
                                             kernel_source_digest()))
    del codes, scales, q, bt, sl, nk, nv, out, slots, ws, graphs
    return fig


def measure_serving_loop(kvc, dev, rank, steps):
    """A decode loop driven by the host block manager on the GQA 8B-shape workload, timed
    end to end on the host clock: per step BlockManager.step (slots, copy pairs, table,
    lengths for 64 sequences), their copy to the device, kvc_paged_decode_append, and a
    synchronisation."""
    case = make_config(WORKLOAD, seed=rank, value_device=str(dev))
    m = case.meta
    bs, NB = case.block_size, case.key_cache.shape[0]
    lens = case.seq_lens.tolist()
    maxb = case.block_table.shape[1] + 1 + (steps + 3) // bs   # room for the steps' tokens
    bm = kvc.BlockManager(NB, bs, maxb)
    for b, L in enumerate(lens):          # prompts already cached: L - 1 tokens
        bm.add(b, L - 1)
    ids = torch.arange(len(lens), dtype=torch.int64)
    buf = bm.step_buffer(len(lens), pin_memory=True)
    step = DecodeStep(kvc, case, dev)
    dtab = torch.empty(len(lens), maxb, dtype=torch.int32, device=dev)
    dlen = torch.empty(len(lens), dtype=torch.int32, device=dev)
    step.bt, step.sl = dtab, dlen

    def one():
        _, cs, cd, table, ln = bm.step(ids, out=buf)
        dtab.copy_(table, non_blocking=True)
        dlen.copy_(ln, non_blocking=True)
        step.step()
        torch.cuda.synchronize()

    for _ in range(3):
        one()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    wall = (time.perf_counter() - t0) / steps
    by = decode_bytes([L + 3 + steps for L in lens], m["num_q_heads"], m["num_kv_heads"],
                      m["head_dim"], bs)
    res = {"ms_per_step": wall * 1e3, "tokens_per_s": len(lens) / wall,
           "approx_gbs": by / wall / 1e9, "steps": steps,
           "step": "BlockManager.step (host) + H2D of block table and lengths + "
                   "kvc_paged_decode_append + synchronize, host clock"}
    del step, case, bm
    return res


def measure_fused_write(kvc, dev, rank, steps, warmup):
    """The MLA decode step's fused latent write: 64 rows [compressed kv 512 | key rope 64],
    RMSNorm of the first part into cache_nope and RoPE (at seq_lens - 1) of the second into
    cache_rope, on the MLA workload's caches."""
    c = make_config("mla_decode", seed=rank, value_device=str(dev))
    B, bs = c.q_nope.shape[0], c.block_size
    g = torch.Generator(device=dev).manual_seed(rank + 7)
    kv = torch.randn(B, 1, 576, generator=g, device=dev).to(c.q_nope.dtype)
    gamma = torch.ones(512, dtype=c.q_nope.dtype, device=dev)
    table = kvc.rope_cos_sin_table(8192, 64, 10000.0, device=dev)
    slots = kvc.build_slot_mapping(c.block_table.to(dev), bs, c.write_pos.to(dev),
                                   c.cache_nope.shape[0])
    pos = c.write_pos.to(dev)

    def write():
        kvc.rmsnorm_rope_cache(kv, gamma, 1e-6, table, pos, slots, c.cache_nope, c.cache_rope)

    for _ in range(warmup):
        write()
    torch.cuda.synchronize()
    graphs = [("write", capture(write))]
    with ClockSampler(dev.index or 0) as clk:
        _, per = time_graphs(graphs, steps)
    by = B * 576 * 2 * 2 + B * 64 * 4 + 2 * B * 4 + 512 * 2
    hp, hkind = peaks()
    fig = _roofline("rmsnorm_rope_cache_kernel (kvc_rmsnorm_rope_cache, 64 latent rows)",
                    per["write"], by, "GB/s", hp, hkind, clk.summary(), bound="launch",
                    rows=B)
    del c, kv, table, graphs
    return fig


def run_mixed(args, kvc, dev, rank):
    pf, dc, ms = measure_mixed(kvc, dev, rank, max(3, args.steps // 4), args.warmup)
    print(json.dumps({"workload": CONFIGS["mixed_packed"]["about"], "ms_per_step": ms,
                      "prefill": pf, "decode": dc}), flush=True)


def run_mla(args, kvc, dev, rank):
    print(json.dumps(dict(workload=CONFIGS["mla_decode"]["about"],
                          **measure_mla(kvc, dev, rank, args.steps, args.warmup))), flush=True)


MEASURES = {
    "mla_decode": measure_mla,
    "mixed": lambda kvc, dev, rank, steps, warmup: measure_mixed(kvc, dev, rank, steps, warmup),
    "llama7b_mha_decode": lambda kvc, dev, rank, steps, warmup: measure_decode(
        kvc, dev, rank, "llama7b_mha_decode", steps, warmup),
    "gqa8b_decode_int8": measure_int8,
    "serving_loop": lambda kvc, dev, rank, steps, warmup: measure_serving_loop(kvc, dev, rank,
                                                                               steps),
    "mla_fused_write": measure_fused_write,
    "gqa8b_block_size_sweep": measure_block_sizes,
}


def secondary(kvc, dev, rank, steps, warmup):
    """Builder-timed figures of the other kernels, each against its own roofline."""
    out = {}
    out["mla_decode"] = measure_mla(kvc, dev, rank, steps, warmup)
    torch.cuda.empty_cache()
    out["mixed_prefill"], out["mixed_decode"], _ = measure_mixed(kvc, dev, rank, steps, warmup)
    torch.cuda.empty_cache()
    out["llama7b_mha_decode"] = measure_decode(kvc, dev, rank, "llama7b_mha_decode", steps,
                                               warmup)
    torch.cuda.empty_cache()
    out["gqa8b_decode_int8"] = measure_int8(kvc, dev, rank, steps, warmup)
    torch.cuda.empty_cache()
    out["serving_loop"] = measure_serving_loop(kvc, dev, rank, steps)
    torch.cuda.empty_cache()
    out["mla_fused_write"] = measure_fused_write(kvc, dev, rank, steps, warmup)
    torch.cuda.empty_cache()
    out["gqa8b_block_size_sweep"] = measure_block_sizes(kvc, dev, rank, min(steps, 50), warmup)
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="kvc", choices=["kvc", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the builder-timed figures of the other kernels")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--profile", action="store_true",
                    help="short run for ncu: no CPU baseline, few e2e steps")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(CONFIGS),
                    help="the timed workload (default: the headline GQA 8B-shape decode)")
    ap.add_argument("--measure", choices=sorted(MEASURES),
                    help="print one of the secondary figures alone (a short run for ncu)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        args.no_cpu_baseline = True
        args.no_secondary = True
        args.e2e_steps = 1

    ws, rank, local = dist_info()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import paged_kv_cache_135_gb300 as kvc
    kvc.build()
    kvc.lib()

    if args.measure:
        print(json.dumps({args.measure: MEASURES[args.measure](kvc, dev, rank, args.steps,
                                                              args.warmup)}), flush=True)
        return
    if CONFIGS[args.workload]["kind"] == "mixed":
        return run_mixed(args, kvc, dev, rank)
    if CONFIGS[args.workload]["kind"] == "mla":
        return run_mla(args, kvc, dev, rank)
    case = make_config(args.workload, seed=rank, value_device=str(dev))
    m = case.meta
    step = DecodeStep(kvc, case, dev)
    B = case.q.shape[0]
    lens = case.seq_lens.tolist()
    d_bytes = decode_bytes(lens, m["num_q_heads"], m["num_kv_heads"], m["head_dim"],
                           case.block_size)
    w_bytes = write_bytes(B, m["num_kv_heads"], m["head_dim"])
    step_bytes = d_bytes + w_bytes

    for _ in range(args.warmup):
        step.step()
    torch.cuda.synchronize()

    # Consecutive steps are captured into one CUDA graph, as a serving loop
    # captures its decode iterations: `per_graph` whole steps (each one full
    # launch over the whole cache) per replay, so no host or graph-launch gap
    # sits between steps.  The K/V read per step (far above L2) is the same
    # whatever the grouping.
    per_graph = steps_per_graph(args.steps)
    g_dec = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g_dec, stream=cap):
            for _ in range(per_graph):
                step.step()
    torch.cuda.current_stream().wait_stream(cap)
    for _ in range(max(1, -(-args.warmup // per_graph))):
        g_dec.replay()
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    n_replay = args.steps // per_graph
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_replay)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize()
        t_start.record(stream)
        for i in range(n_replay):
            ev[i][0].record(stream)
            g_dec.replay()
            ev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier()
    total_ms = t_start.elapsed_time(t_end)
    dec_ms = [a.elapsed_time(b) / per_graph for a, b in ev]  # per launch

    # Diagnostic: the same step launched eagerly through the Python binding.
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(20):
        step.step()
    e1.record(stream)
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1) / 20
    total_ms = max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / args.steps
    value = ws * step_bytes / (ms_per_step * 1e-3) / 1e9
    tokens_per_s = ws * B / (ms_per_step * 1e-3)

    # End to end through the public API: per step, the step's inputs (staged
    # in one pinned host buffer, as a serving loop would) -> device in one
    # copy, the step, device -> pinned host output, and the host waits for
    # that output.  Serial: each step synchronised before the next.
    # Pipelined: two buffer sets; step i+1's inputs copy (copy stream) while
    # step i runs (compute stream) and step i-1's output copies back (a third
    # stream); the host waits for step i's output before it stages step i+2.
    names = ("q", "new_key", "new_value", "block_table", "seq_lens")
    src = {k: getattr(case, k).cpu().contiguous() for k in names}
    offs, total = {}, 0
    for k in names:
        offs[k] = total
        total += (src[k].numel() * src[k].element_size() + 255) // 256 * 256
    h_pack = torch.empty(total, dtype=torch.uint8).pin_memory()
    d_packs = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    outs = [step.out, torch.empty_like(step.out)]

    def view(buf, k):
        n = src[k].numel() * src[k].element_size()
        return buf[offs[k]:offs[k] + n].view(src[k].dtype).view(src[k].shape)

    sets = [tuple(view(d_packs[j], k) for k in names) for j in range(2)]

    def use(i):  # point the step at buffer set i % 2
        step.q, step.nk, step.nv, step.bt, step.sl = sets[i % 2]
        step.out = outs[i % 2]

    for k in names:
        view(h_pack, k).copy_(src[k])
    h_outs = [torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory() for _ in range(2)]
    h2d = total
    d2h = h_outs[0].numel() * h_outs[0].element_size()
    for i in range(3 + args.e2e_steps):
        if i == 3:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
        use(0)
        d_packs[0].copy_(h_pack, non_blocking=True)
        step.step()
        h_outs[0].copy_(step.out, non_blocking=True)
        torch.cuda.synchronize()
    e2e_serial_s = (time.perf_counter() - t0) / max(1, args.e2e_steps)

    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    n_pipe = 3 + args.e2e_steps
    ev_in = [torch.cuda.Event() for _ in range(n_pipe)]
    ev_done = [torch.cuda.Event() for _ in range(n_pipe)]
    ev_out = [torch.cuda.Event() for _ in range(n_pipe)]
    torch.cuda.synchronize()
    for i in range(n_pipe):
        if i == 3:
            ev_out[2].synchronize()
            t0 = time.perf_counter()
        if i >= 2:
            ev_out[i - 2].synchronize()    # step i-2's result is on the host
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_done[i - 2])  # its input buffer is free again
            d_packs[i % 2].copy_(h_pack, non_blocking=True)
            ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        use(i)
        step.step()
        ev_done[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[i])
            h_outs[i % 2].copy_(outs[i % 2], non_blocking=True)
            ev_out[i].record(s_out)
    ev_out[n_pipe - 1].synchronize()
    e2e_s = (time.perf_counter() - t0) / max(1, args.e2e_steps)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(e2e_s, dev)
    e2e_serial_s = max_over_ranks(e2e_serial_s, dev)

    peak, peak_kind = peaks()
    dec_avg_ms = statistics.mean(dec_ms)
    achieved = step_bytes / (dec_avg_ms * 1e-3) / 1e9
    digest = kernel_source_digest()
    traffic = (recorded_traffic("paged_decode_kernel/" + WORKLOAD, digest)
               if args.workload == WORKLOAD else None)

    if rank == 0:
        res = {
            "metric": DECODE_METRIC,
            "value": value,
            "unit": "GB/s",
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms_per_step,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": case.dtype,
            "data": "synthetic",
            "config": dict(decode_workload(args.workload, case, ws)[0],
                           steps_per_graph=per_graph),
            "decode_tokens_per_s": tokens_per_s,
            "pct_of_nominal_8tbps": 100.0 * value / NOMINAL_HBM_GBS,
            "roofline": {
                "kernel": "paged_decode_kernel (one kvc_paged_decode_append call: new-token "
                          "write, decode and split-KV merge fused)",
                "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_kind": peak_kind, "traffic": traffic,
                "algorithmic_bytes_per_launch": step_bytes, "avg_launch_ms": dec_avg_ms,
                "launch_ms_p10_p50_p90": launch_percentiles(dec_ms),
                "eager_launch_ms": eager_ms,
                "frac_of_nominal_8tbps": achieved / NOMINAL_HBM_GBS,
            },
            "e2e": {"value": ws * step_bytes / e2e_s / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_s * 1e3, "tokens_per_s": ws * B / e2e_s,
                    "pipelined": "2 buffer sets: step i+1's H2D and step i-1's D2H overlap "
                                 "step i; the host waits for each step's output",
                    "serial": {"value": ws * step_bytes / e2e_serial_s / 1e9,
                               "ms_per_step": e2e_serial_s * 1e3}},
            "gpu_launches": DecodeStep.LAUNCHES * args.steps,
            "clocks": clk.summary(),
        }
        if not args.no_secondary:
            del step, g_dec, d_packs, outs, h_pack, h_outs
            torch.cuda.empty_cache()
            res["secondary"] = secondary(kvc, dev, rank, min(args.steps, 100), args.warmup)
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(case)
        print(json.dumps(res), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
