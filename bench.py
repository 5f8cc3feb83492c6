#!/usr/bin/env python
"""Benchmark of the KV-cache scoring -> pruning -> compaction path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c2] [--impl kvs|reference]

One step = one pass of the whole path over one batch of synthetic input (all layers):
  c3 (default; the largest single-GPU workload, Qwen3-8B-shaped chunked KVzip+):
      vnorm -> 16 x (lse -> score_max) -> threshold at each layer's 25th score percentile
      (selected on the GPU in every step) with w=128 -> compaction
  c1: lse -> score_max -> top-k 25% + w=16 -> compaction
  c2: (Qwen2.5-1.5B-shaped KVzip+) vnorm -> lse -> score_max -> top-k at
      r = 0.3 / 0.5 / 0.7 -> paged compaction of each
  c4: lse (causal) -> future mass (w=128) -> top-k 25% / 12.5% + window -> compaction
      (--attn-forward: pass 1 is the attention forward, output + LSE, instead)
  c2 --refit: adds the closed-form value refit (Select+Fit) of the r=0.3 budget's kept keys
  c5: surrogate (+ fused threshold tau=-5, w=128) -> compaction
  c6: MLP surrogate 4096 -> 512 -> 8 (+ threshold tau=-4, w=128) -> compaction
  c7: decode step of 64 sequences: surrogate score of the arriving tokens -> window-boundary
      threshold + append to the paged cache (metric: tokens decided per second per layer)
Metric: context KV tokens scored+pruned per second per layer (all heads) = T * L / step time.

Timing: inputs resident in HBM; W warm-up steps; K timed steps, each bracketed by CUDA
events on the launching stream, with a 512 MB buffer written between steps (outside the
events) to flush L2; barrier + synchronize on both sides; max over ranks.  SM clocks and
throttle reasons are sampled with nvidia-smi during the timed steps.  Each library entry
point is then timed on its own (same rules) for the roofline of the dominant kernel.
`e2e` repeats the step through the same public calls with the inputs in pinned host
memory: host->device copies of every input and a device->host read of the results are
inside the timed region.  `cpu_baseline` times the fp64 CPU oracle on a bounded sample.

The step is replayed from a CUDA graph captured once (``--no-graph`` launches every
call from Python instead); each entry point's timing also replays its own graph.

`--impl reference` times the CPU oracle itself (the only reference implementation: the
pages ship no code) on the host's CPU cores, each step a bounded sample of the workload:
its `steps` and `ms_per_step` are the samples it ran and their measured wall time, and
the line's `extrapolation` states how a sample's time converts to a layer's.
Under torchrun (N > 1) every rank runs its own replica of the workload (weak scaling; the
path shards by independent problems and needs no data exchange).
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

METRIC = "context KV tokens scored+pruned/s per layer (all heads); % of tensor/HBM roofline"
UNIT = "tokens/s/layer"
# a contraction timed over at least this much back-to-back replay runs under the power cap
LONG_RUN_MS = 1000.0
L2_FLUSH_BYTES = 512 << 20


def read_traffic(workload, stage):
    """DRAM bytes per launch of `stage` on `workload` from profiles/traffic.txt (an ncu
    capture of the same kernel), or None when no capture of the current kernel exists."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        f = line.split()
        if len(f) >= 3 and not f[0].startswith("#") and f[0] == workload and f[1] == stage:
            return int(f[2])
    return None


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="c3", choices=["c1", "c2", "c3", "c4", "c5", "c6", "c7"])
    ap.add_argument("--impl", default="kvs", choices=["kvs", "reference"])
    ap.add_argument("--attn-forward", action="store_true",
                    help="c4: pass 1 is the attention forward (output + LSE) instead of the "
                         "LSE-only pass")
    ap.add_argument("--refit", action="store_true",
                    help="c1/c2: add the closed-form value refit on the first budget's kept keys")
    ap.add_argument("--e2e-groups", type=int, default=12,
                    help="layer groups of the end-to-end run: copies of one group overlap the "
                         "kernels of the previous one (1: copy everything, then compute)")
    ap.add_argument("--e2e-copy-streams", type=int, default=1,
                    help="streams the host-to-device copies of a layer group are spread over")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stage-reps", type=int, default=None)
    ap.add_argument("--layers", type=int, default=None,
                    help="run only the first N layers (profiling on a smaller case)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every call from Python instead of replaying a CUDA graph")
    return ap.parse_args()


DEFAULT_STEPS = {"c1": 200, "c2": 200, "c3": 10, "c4": 10, "c5": 20, "c6": 10, "c7": 200}


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


# ----------------------------------------------------------------------------- work model

def algorithmic_work(wl, p):
    """Algorithmic flops / bytes of one call of each library entry point of a step,
    summed over the step: 2 d flops per query-key element that the method defines (the
    visible pairs of the causal rule, every context key for the maximum, the band
    j >= i + w for the future mass), the Gram form of the value norms, and the bytes an
    HBM-bound kernel must move at least once."""
    d, L = wl.d, p.L
    out = {}
    if wl.kind in ("kvzip", "kvzip_plus", "kvzip_plus_chunked"):
        chunks = wl.n_chunks if wl.kind == "kvzip_plus_chunked" else 1
        nq = wl.n_rep
        el1 = 0
        for c in range(chunks):
            nk = wl.T + wl.tail_len(c)
            off = nk - nq
            el1 += L * wl.H_q * (nq * off + nq * (nq + 1) // 2)
        el2 = L * wl.H_q * nq * wl.T * chunks
        out["kvs_lse"] = ("tensor", 2 * d * el1, "flop")
        out["kvs_score_max"] = ("tensor", 2 * d * el2, "flop")
        if wl.kind != "kvzip":
            out["kvs_vnorm"] = ("tensor", 2 * L * wl.H_q * d * d * (wl.D_h + wl.T), "flop")
        if getattr(p, "refit", False):
            # forward over the context (S and P V), S and softmax over the kept keys, the
            # symmetric Gram, the right-hand side, Cholesky and the two triangular solves
            k, n, B = p.k_fit, wl.g * nq, L * wl.H_kv
            out["kvs_value_refit"] = ("tensor", B * (4 * d * n * wl.T + 2 * d * n * k
                                                     + n * k * (k + 1) + 2 * n * k * d
                                                     + k ** 3 // 3 + 2 * k * k * d), "flop")
    if wl.kind == "future":
        n, w = wl.T, wl.w
        el1 = L * wl.H_q * n * (n + 1) // 2
        m = max(0, n - w)
        el2 = L * wl.H_q * m * (m + 1) // 2
        out["kvs_lse"] = ("tensor", 2 * d * el1, "flop")
        out["kvs_attn_fwd"] = ("tensor", 4 * d * el1, "flop")  # S = Q K^T and O = P V
        out["kvs_score_future_sum"] = ("tensor", 2 * d * el2, "flop")
    if wl.kind == "kvzap":
        rows = L * wl.H_kv
        out["kvs_surrogate"] = ("hbm", L * wl.T * wl.D_h * 2 + L * wl.D_h * wl.H_kv * 2
                                + rows * wl.T * (4 + 1), "byte")
    if wl.kind == "decode":
        B, H = wl.batch, wl.H_kv
        out["kvs_surrogate"] = ("hbm", L * B * wl.D_h * 2 + L * wl.D_h * H * 2 + L * H * B * 4,
                                "byte")
        # per row: the arriving K/V read and written into the ring, the leaving K/V read,
        # the appended fraction written to a page, plus the scalars
        rows = L * H * B
        steps = max(1, int(p.pos[0].item()) - wl.w)
        frac = float(p.seq_lens.sum().item()) / (rows * steps)
        out["kvs_decode_step"] = ("hbm", int(rows * (4 * wl.d * (3 + frac) + 16)), "byte")
    if wl.kind == "kvzap_mlp":
        # two linear layers per token: 2 D_h D_mid + 2 D_mid H = (D_h / 4)(D_h + H)
        out["kvs_surrogate_mlp"] = ("tensor", L * wl.T * (2 * wl.D_h * wl.D_mid
                                                          + 2 * wl.D_mid * wl.H_kv), "flop")
    return out


def units_per_step(wl, p):
    """Context tokens a step scores and prunes in each layer (decode: one arriving token
    per sequence), times the layers."""
    return (wl.batch if wl.kind == "decode" else wl.T) * p.L


def compaction_bytes(p, wl):
    pages = p.pages if isinstance(p.pages, list) else [p.pages]
    rows = p.L * wl.H_kv
    kept = sum(int(pg.seq_lens.sum().item()) for pg in pages)
    pad = sum(int(((-pg.seq_lens) % wl.page_size).sum().item()) for pg in pages)
    return (kept * wl.d * 2 * 2 * 2 + pad * wl.d * 2 * 2
            + len(pages) * rows * (wl.T + pages[0].max_pages * 4))


def prune_bytes(p, wl):
    n = len(p.masks) if hasattr(p, "masks") else 1
    return n * p.L * wl.H_kv * wl.T * (4 + 1)


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(value, world, device="cpu"):
    """Maximum of a per-rank timing over all ranks (the slowest rank sets the step)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank, world, ms_step):
    """Units processed by all ranks per second, timed by the slowest rank."""
    return world * units_per_rank / (ms_step / 1e3)


def run_config(wl, args, world, layers):
    """The workload description that both arms print, with the same keys and values, so
    that their lines name the same configuration."""
    return {"workload": f"{wl.name}: {wl.title}", "layers": layers, "T": wl.T, "H_q": wl.H_q,
            "H_kv": wl.H_kv, "d": wl.d, "D_h": wl.D_h, "parallelism": f"replicas x{world}",
            "pass1": "attention forward (output + LSE)" if args.attn_forward else "LSE-only pass",
            "value_refit": bool(args.refit),
            "l2": f"GPU arm: a {L2_FLUSH_BYTES >> 20} MB buffer is written between timed steps"}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.error = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu_id)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception as e:  # no nvidia-smi
            self.error = str(e)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        if self.error or not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": self.error or "no samples"}
        rows = [l.split(", ") for t, l in self.lines if t0 - 0.15 <= t <= t1 + 0.15]
        if not rows:
            rows = [self.lines[-1][1].split(", ")]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if len(r) > 5 + i and r[5 + i].strip().lower() == "active"})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ----------------------------------------------------------------------------- GPU arm

def build_pipeline(wl, device, attn_forward=False, refit=False):
    from kv_cache_eviction_lse_gb300 import pipeline, workloads as W
    x = W.generate(wl, device=device)
    kw = {}
    if attn_forward:
        kw["attn_forward"] = True
    if refit:
        kw["refit"] = True
    p = pipeline.make_pipeline(wl, x, **kw)
    return x, p


def run_gpu(args, rank, world, local):
    import torch
    import torch.distributed as dist
    from kv_cache_eviction_lse_gb300 import build as B
    B.build()
    from kv_cache_eviction_lse_gb300 import capi as C
    from kv_cache_eviction_lse_gb300 import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    wl = W.WORKLOADS[args.workload]
    if args.layers:
        wl = wl.scaled(L=min(args.layers, wl.L))
    K = args.steps or DEFAULT_STEPS[args.workload]
    Wm = max(3, args.warmup)
    x, p = build_pipeline(wl, dev, attn_forward=args.attn_forward, refit=args.refit)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    for _ in range(Wm):
        p.step()
    torch.cuda.synchronize()
    n_before = C.kvs_launch_count()
    p.step()
    torch.cuda.synchronize()
    launches = C.kvs_launch_count() - n_before
    step_fn = p.step if args.no_graph else capture(p.step)
    for _ in range(Wm):
        step_fn()
    torch.cuda.synchronize()

    # ---------------------------------------------------------------- timed steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    props = torch.cuda.get_device_properties(dev)
    gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else local
    with ClockSampler(gpu_id) as clk:
        barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        for i in range(K):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            step_fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
        barrier()
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), world, dev)
    ms_step = ms / K
    value = whole_job_value(units_per_step(wl, p), world, ms_step)

    # ---------------------------------------------------------------- per entry point
    reps = args.stage_reps or max(3, min(50, K))
    work = algorithmic_work(wl, p)
    stage_ms = {}
    for name, fn in p.stages():
        run = fn if args.no_graph else capture(fn)
        run()
        e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(reps)]
        for i in range(reps):
            flush.fill_(float(i))
            e[i][0].record(stream)
            run()
            e[i][1].record(stream)
        torch.cuda.synchronize()
        stage_ms[name] = sum(a.elapsed_time(b) for a, b in e) / reps
    step_fn()  # leave consistent outputs
    torch.cuda.synchronize()
    for name in stage_ms:
        if name.startswith("kvs_compact_paged"):
            work[name] = ("hbm", compaction_bytes(p, wl), "byte")
        if name.startswith("kvs_prune"):
            work[name] = ("hbm", prune_bytes(p, wl), "byte")

    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
        src = "measured"
    except Exception:
        src = "fallback"
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    tc_peak = peaks.get("bf16_tflops", 1900.0)
    tc_sus = peaks.get("bf16_tflops_sustained", 1700.0)
    kernels = {}
    for name, t in stage_ms.items():
        bound, amount, unit = work.get(name, ("hbm", None, "byte"))
        k = {"ms": round(t, 5), "share": None}
        if amount is not None:
            if unit == "flop":
                ach = amount / (t / 1e3) / 1e12
                # a contraction whose timed replays run back to back for a second or more
                # is held to the power-capped (sustained) tensor peak, a shorter one to
                # the burst peak; both fractions are reported
                sustained = reps * t >= LONG_RUN_MS
                pk = tc_sus if sustained else tc_peak
                k.update(bound="tensor", achieved=round(ach, 2), unit="TFLOP/s",
                         peak=pk, frac=round(ach / pk, 4),
                         peak_kind="sustained" if sustained else "burst",
                         frac_burst=round(ach / tc_peak, 4),
                         frac_sustained=round(ach / tc_sus, 4))
            else:
                ach = amount / (t / 1e3) / 1e9
                k.update(bound="hbm", achieved=round(ach, 1), unit="GB/s",
                         peak=hbm_peak, frac=round(ach / hbm_peak, 4))
        kernels[name] = k
    # each stage is replayed on its own; its share is of the graph-replayed step, so the
    # shares need not add up to one (a stage alone pays its own graph launch and tail)
    for k in kernels.values():
        k["share"] = round(k["ms"] / ms_step, 4)
    dom = max(kernels, key=lambda n: kernels[n]["ms"])
    dk = kernels[dom]
    roofline = {"kernel": dom, "bound": dk.get("bound"), "achieved": dk.get("achieved"),
                "peak": dk.get("peak"), "unit": dk.get("unit"), "frac": dk.get("frac"),
                "traffic": None}
    if dk.get("bound") == "tensor":
        kind = dk["peak_kind"]
        key = "bf16_tflops_sustained" if kind == "sustained" else "bf16_tflops"
        roofline["peak_source"] = (
            f"{src} (MEASURED_PEAKS.json {key}: the stage's {reps} timed replays ran "
            f"{reps * stage_ms[dom] / 1e3:.2f} s back to back"
            + (", so the power-capped peak applies)" if kind == "sustained" else ")")
            if src == "measured" else "fallback")
        roofline.update(peak_burst=tc_peak, frac_burst=dk.get("frac_burst"),
                        peak_sustained=tc_sus, frac_sustained=dk.get("frac_sustained"))
    else:
        roofline["peak_source"] = (f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured"
                                   else "fallback")
    roofline["traffic"] = read_traffic(wl.name, dom)

    # ---------------------------------------------------------------- end to end
    e2e = None
    if not args.no_e2e:
        from kv_cache_eviction_lse_gb300 import pipeline as PL
        kw = {"attn_forward": True} if args.attn_forward else {}
        if args.refit:
            kw["refit"] = True

        def make_group(xg, l0, l1):
            return PL.make_pipeline(wl, xg, **kw)
        groups = 1 if wl.kind == "decode" else min(args.e2e_groups, p.L)
        e2e = run_e2e(wl, x, p, dev, K=min(K, 20), units=world * units_per_step(wl, p), world=world,
                      flush=flush, graph=not args.no_graph, groups=groups, make_group=make_group,
                      copy_streams=args.e2e_copy_streams)

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": run_config(wl, args, world, p.L),
        "launch": "python calls" if args.no_graph else "CUDA graph of the step",
        "roofline": roofline,
        "kernels": kernels,
        "kernels_share_basis": (f"stage time (each stage replayed alone) / step time "
                                f"{ms_step:.4f} ms; the stages sum to "
                                f"{sum(stage_ms.values()):.4f} ms"),
        "gpu_launches": launches,
        "clocks": clk.summary(t0, t1),
        "e2e": e2e,
    }
    return result, wl, p


def capture(fn):
    """Record the library calls `fn` enqueues into a CUDA graph; returns its replay.
    The graph holds exactly the kernels (and memsets) that `fn` launches."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    capture.graphs.append(g)
    return g.replay


capture.graphs = []


def _layer_slice(x, l0, l1):
    """The inputs of layers [l0, l1) as views of x (every tensor is layer-major)."""
    return {k: ([t[l0:l1] for t in v] if isinstance(v, list) else v[l0:l1]) for k, v in x.items()}


def _step_outputs(p):
    """The results a step hands back to the host: scores plus the pages' block tables and
    lengths (decode: the fill levels)."""
    outs = [p.score]
    if hasattr(p, "pages"):
        pages = p.pages if isinstance(p.pages, list) else [p.pages]
        for pg in pages:
            outs += [pg.seq_lens, pg.block_table]
    else:
        outs += [p.seq_lens]
    return outs


def run_e2e(wl, x, p, dev, K, units, world, flush, graph=True, groups=1, make_group=None,
            copy_streams=1):
    """Same step through the same calls, inputs from pinned host memory: the H2D copies
    of every input and the D2H read of the results are inside the timed region.

    With groups > 1 the layers are split into that many groups, each with its own
    pipeline over views of the same device tensors: the host->device copies of group
    g+1 run on a copy stream while group g computes, and each group's results are read
    back as soon as it finishes.  Every byte still crosses the link inside the timed
    region; only their overlap with the kernels changes."""
    import torch

    L = p.L
    groups = max(1, min(groups, L))
    bounds = [(L * g // groups, L * (g + 1) // groups) for g in range(groups)]
    host = {}
    for k, v in x.items():
        ts = v if isinstance(v, list) else [v]
        hs = []
        for t in ts:
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t.cpu())
            hs.append(h)
        host[k] = hs if isinstance(v, list) else hs[0]
    parts = []  # per group: (copy pairs, step function, outputs, pinned outputs)
    keep = []   # the group pipelines: their buffers must outlive the captured graphs
    for l0, l1 in bounds:
        pg = p if groups == 1 else make_group(_layer_slice(x, l0, l1), l0, l1)
        xs, hs = _layer_slice(x, l0, l1), _layer_slice(host, l0, l1)
        pairs = []
        for k in xs:
            dv, hv = xs[k], hs[k]
            for d, h in (zip(dv, hv) if isinstance(dv, list) else [(dv, hv)]):
                pairs.append((h, d))
        outs = _step_outputs(pg)
        outs_h = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
        keep.append(pg)
        parts.append((pairs, capture(pg.step) if graph else pg.step, outs, outs_h))
    bi = sum(h.numel() * h.element_size() for pr in parts for h, _ in pr[0])
    bo = sum(o.numel() * o.element_size() for pr in parts for o in pr[2])
    stream = torch.cuda.current_stream()
    nstreams = max(1, copy_streams) if groups > 1 else 1
    copy_ss = [torch.cuda.Stream() for _ in range(nstreams)] if groups > 1 else [stream]
    tot = 0.0
    for i in range(K + 2):
        flush.fill_(float(i))
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for cs in copy_ss:
            cs.wait_event(a)
        ready = []
        for pairs, _, _, _ in parts:
            evs = []
            for j, cs in enumerate(copy_ss):  # a group's tensors, spread over the copy streams
                with torch.cuda.stream(cs):
                    for h, d in pairs[j::len(copy_ss)]:
                        d.copy_(h, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cs)
                evs.append(ev)
            ready.append(evs)
        for (pairs, step_fn, outs, outs_h), evs in zip(parts, ready):
            for ev in evs:
                stream.wait_event(ev)
            step_fn()
            for o, oh in zip(outs, outs_h):
                oh.copy_(o, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        if i >= 2:
            tot += a.elapsed_time(b)
    ms = tot / K
    del keep
    out = {"value": round(units / (ms / 1e3), 1), "unit": UNIT, "ms_per_step": round(ms, 4),
           "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo}
    if groups > 1:
        out["overlap"] = (f"layers in {groups} groups: the H2D copies of group g+1 (on "
                          f"{len(copy_ss)} copy streams) overlap the kernels of group g")
    return out


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample(wl, x, frac=1.0):
    """Time the CPU oracle on a bounded sample of the workload (layer 0).

    kvzip kinds: KV-head group 0 (its g query heads), the first max(1, frac*n_q) scoring
    queries of the block (tail keys trimmed so the causal offset is unchanged), all T
    context keys; vnorm of those heads, LSE, score, then top-k/threshold + compaction of
    the group's score row.  The query-proportional parts are scaled by n_q / n_sub (and
    the chunks), and everything by the number of groups.  future: the first frac*T tokens
    of group 0 (cost ~ n^2, scaled by (T/n)^2 and the groups).  kvzap: the first frac*T
    tokens of layer 0 (all heads), scaled by T/n; kvzap_mlp likewise.
    Returns (seconds per layer, tokens per layer, description)."""
    import numpy as np
    import torch

    import oracle as O

    def f64(t):
        return O.bf16_bits_to_f64(t.contiguous().view(torch.int16).numpy().view(np.uint16))

    def i16(t):
        return t.contiguous().view(torch.int16).numpy()

    tick = time.perf_counter
    if wl.kind in ("kvzip", "kvzip_plus", "kvzip_plus_chunked"):
        g, d = wl.g, wl.d
        chunked = wl.kind == "kvzip_plus_chunked"
        q_all = x["q"][0] if chunked else x["q"]
        kt_all = x["k_tail"][0] if chunked else x["k_tail"]
        h_all = (x["h"][0] if chunked else x["h"]) if "h" in x else None
        n_q = q_all.shape[2]
        n_sub = max(1, min(n_q, int(round(frac * n_q))))
        trim = n_q - n_sub
        q = f64(q_all[:, 0:g, :n_sub])
        kt = f64(kt_all[:, 0:1, : kt_all.shape[2] - trim])
        kc = f64(x["k_ctx"][:, 0:1])
        t0 = tick()
        vn = O.value_norm(f64(x["v_ctx"][:, 0:1]), f64(x["w_o"][:, :, 0:g * d]), g) \
            if "w_o" in x else None
        t1 = tick()
        lse = O.lse(q, kc, kt)
        s = O.kvzip_score(q, kc, kt, lse_=lse, vnorm=vn,
                          h=f64(h_all[:, :n_sub]) if h_all is not None else None)
        t2 = tick()
        if wl.keep_ratios:
            for r in wl.keep_ratios:
                m, _ = O.prune_topk(s, wl.topk_budget(r), wl.w)
                O.compact_paged(i16(x["k_ctx"][:, 0:1]), i16(x["v_ctx"][:, 0:1]), m, wl.page_size)
        else:
            m, _, _ = O.prune_quantile(s, wl.tau_quantile, wl.w)
            O.compact_paged(i16(x["k_ctx"][:, 0:1]), i16(x["v_ctx"][:, 0:1]), m, wl.page_size)
        t3 = tick()
        chunks = wl.n_chunks if chunked else 1
        dt = wl.H_kv * ((t1 - t0) + (t2 - t1) * (n_q / n_sub) * chunks + (t3 - t2))
        desc = (f"layer 0, KV-head group 0 ({g} query heads), {n_sub} of {n_q} scoring queries"
                f"{' of chunk 0' if chunked else ''}: vnorm, LSE, score, "
                f"{'top-k' if wl.keep_ratios else 'threshold'} + compaction; query-proportional "
                f"time scaled x{n_q / n_sub * chunks:g}, all x{wl.H_kv} groups")
        return dt, wl.T, desc
    if wl.kind == "future":
        g = wl.g
        n = max(256, min(wl.T, int(round(frac * wl.T))))
        t0 = tick()
        q = f64(x["q"][:, 0:g, :n]); k = f64(x["k"][:, 0:1, :n])
        f = O.future_attention_mass(q, k, wl.w)
        for r in wl.keep_ratios:
            m, _ = O.prune_topk(f, int(r * n + 0.5), wl.w)
            O.compact_paged(i16(x["k"][:, 0:1, :n]), i16(x["v"][:, 0:1, :n]), m, wl.page_size)
        dt = (tick() - t0) * wl.H_kv * (wl.T / n) ** 2
        return dt, wl.T, (f"layer 0, KV-head group 0, first {n} of {wl.T} tokens: LSE, future mass, "
                          f"top-k + compaction; scaled x{wl.H_kv}*(T/{n})^2")
    if wl.kind == "kvzap":
        n = max(1024, min(wl.T, int(round(frac * wl.T))))
        t0 = tick()
        z = O.linear_surrogate(f64(x["h"][:, :n]), f64(x["W"]), x["b"].double().numpy())
        m, _ = O.prune_threshold(z, wl.tau, wl.w)
        O.compact_paged(i16(x["k"][:, :, :n]), i16(x["v"][:, :, :n]), m, wl.page_size)
        dt = (tick() - t0) * (wl.T / n)
        return dt, wl.T, (f"layer 0, first {n} of {wl.T} tokens (all heads): surrogate, threshold, "
                          f"compaction; scaled x(T/{n})")
    if wl.kind == "decode":
        steps = 2 * wl.w
        t0 = tick()
        # the same surrogate on every step's arriving tokens (the inputs repeat), then
        # the window-boundary decisions of every (head, sequence) row over `steps` steps
        z = None
        for _ in range(steps):
            z = O.linear_surrogate(f64(x["h"]), f64(x["W"]), x["b"].double().numpy())
        rows = np.repeat(z.reshape(-1, 1), steps, axis=1)
        O.decode_prune(rows, wl.tau, wl.w)
        dt = tick() - t0
        return dt / steps, wl.batch, (f"layer 0, {wl.batch} sequences x {wl.H_kv} KV heads, "
                                      f"{steps} decode steps: surrogate of the arriving tokens "
                                      f"and window-boundary decisions; per step")
    if wl.kind == "kvzap_mlp":
        n = max(1024, min(wl.T, int(round(frac * wl.T))))
        t0 = tick()
        z = O.mlp_surrogate(f64(x["h"][:, :n]), f64(x["W1"]), x["b1"].double().numpy(),
                            f64(x["W2"]), x["b2"].double().numpy())
        m, _ = O.prune_threshold(z, wl.tau, wl.w)
        O.compact_paged(i16(x["k"][:, :, :n]), i16(x["v"][:, :, :n]), m, wl.page_size)
        dt = (tick() - t0) * (wl.T / n)
        return dt, wl.T, (f"layer 0, first {n} of {wl.T} tokens (all heads): MLP surrogate, "
                          f"threshold, compaction; scaled x(T/{n})")
    raise ValueError(wl.kind)


def host_layer0(wl):
    from kv_cache_eviction_lse_gb300 import workloads as W
    return W.generate(wl, layers=[0], device="cpu")


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


CPU_BASELINE_FRAC = {"c1": 1.0, "c2": 1.0, "c3": 1 / 8, "c4": 1 / 4, "c5": 1 / 8, "c6": 1 / 16,
                     "c7": 1.0}


def run_cpu_baseline(wl):
    x = host_layer0(wl)
    dt, tokens, desc = oracle_sample(wl, x, CPU_BASELINE_FRAC[wl.name])
    return {"value": round(tokens / dt, 2), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": desc + f"; {dt:.2f} s per layer; numpy fp64 (BLAS threads = host cores, "
                             "elementwise single-threaded)"}


REFERENCE_BUDGET_S = 120.0


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, timed on the host cores.

    Each step is one bounded sample of the workload (oracle_sample), sized so that the
    warm-up and timed samples take about REFERENCE_BUDGET_S seconds.  `steps` is the
    number of samples timed and `ms_per_step` their measured mean wall time, so that
    steps x ms_per_step is the timed region.  `value` converts a sample's time to the
    time of one whole layer (the rule is in the line's `extrapolation`) and divides the
    layer's context tokens by it."""
    if rank != 0:
        return None
    from kv_cache_eviction_lse_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    if args.layers:
        wl = wl.scaled(L=min(args.layers, wl.L))
    K = args.steps or 3
    Wm = max(3, args.warmup)
    x = host_layer0(wl)
    frac = CPU_BASELINE_FRAC[wl.name]
    t = time.perf_counter()
    oracle_sample(wl, x, frac / 8)
    probe = time.perf_counter() - t
    per_step = REFERENCE_BUDGET_S / (K + Wm)
    frac = max(frac / 64, min(frac, frac / 8 * per_step / max(probe, 1e-6)))
    for _ in range(Wm):
        oracle_sample(wl, x, frac)
    layer_s, wall, desc, tokens = [], [], "", wl.T
    for _ in range(K):
        t = time.perf_counter()
        dt, tokens, desc = oracle_sample(wl, x, frac)
        wall.append(time.perf_counter() - t)
        layer_s.append(dt)
    ms_sample = 1e3 * statistics.mean(wall)
    ms_layer = 1e3 * statistics.mean(layer_s)
    value = tokens / (ms_layer / 1e3)
    cb = {"value": round(value, 2), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
          "sample": desc + f"; {ms_sample / 1e3:.2f} s of CPU work per step"}
    return {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
            "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": round(ms_sample, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": run_config(wl, args, world, wl.L),
            "extrapolation": {
                "measured_ms_per_step": round(ms_sample, 3),
                "layer_equivalent_ms": round(ms_layer, 3),
                "tokens_per_layer": tokens,
                "rule": ("value = tokens_per_layer / layer_equivalent_ms; each step times one "
                         "sample and scales its parts to a whole layer: " + desc)},
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    res, wl, p = run_gpu(args, rank, world, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = run_cpu_baseline(wl)
        else:
            res["cpu_baseline"] = None
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
