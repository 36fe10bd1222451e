"""Benchmark of the CSA decode step on GB300.

One step = the whole hot path (plan, indexer score, Top-K, gather + split
softmax attention + LSE merge + inverse RoPE) over one batch of the long
ragged workload (B=64, S=1, L_b ~ U{1024..65536}, H=64, D=576, K=512,
WIN=128, bf16) through the C ABI.  Prints one JSON line; its "workloads"
object carries the same measurements (throughput, roofline, oracle on all
host cores and on one) for every other named workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

Inputs are resident in HBM.  Every step reads a different one of several
device copies of the batch, so each step's reads (about 190 MB) come from
HBM, not from a warm L2.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 126 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="long_ragged_b64")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--copies", type=int, default=3, help="device copies of the inputs, rotated per step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--workloads", default="all",
                    help="other named workloads measured after the headline one: all, none, or a comma list")
    ap.add_argument("--other-steps", type=int, default=300, help="timed steps of each other workload")
    ap.add_argument("--cpu-seconds", type=float, default=6.0, help="wall time of each oracle baseline")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_seed(base_seed: int, rank: int) -> int:
    """Weak scaling: every rank decodes its own batch, drawn from its own seed."""
    return base_seed + 7919 * rank


def reduce_max(value: float, dist, device) -> float:
    """Max over ranks (the slowest rank defines the step time); identity at N=1."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(queries_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job queries/s: every rank's queries over the slowest rank's step time."""
    return queries_per_rank * world / (ms_per_step * 1e-3)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        hbm = d.get("hbm_gbs")
        if hbm:
            return float(hbm), "measured", d
    except Exception:
        pass
    return FALLBACK_HBM_GBS, "fallback", {}


# ---------------------------------------------------------------------------
# algorithmic bytes (what the step must move; the score scratch is not counted)

def step_bytes(cfg, lens, S, topk_idx=None):
    """Per-step algorithmic bytes and per-kernel shares for one batch.

    Per query: q (H*D*e), output (H*V*e); per request, counted once: the
    window rows and selected compressed rows it reads (union over its
    queries), the indexer keys it scores and q_idx/w of scored queries, and
    the heavy-compression rows (FP8 keys: Di bytes + a 4-byte scale per row).
    topk_idx [B*S, K] (numpy) gives the selected
    rows; without it every query is assumed to read min(vis, K) rows.
    """
    e = cfg.esize
    fp8 = getattr(cfg, "idx_dtype", "same") == "fp8"
    key_row = cfg.Di + 4 if fp8 else cfg.Di * e  # FP8 keys: one byte per dim + the row scale
    tot_q = tot_rows = idx_b = 0
    for b, L in enumerate(lens):
        win_rows, sel, hca_rows, krows = set(), set(), 0, 0
        for s in range(S):
            pos = L - S + s
            vis = (pos + 1) // cfg.ratio
            nwin = min(cfg.win, pos + 1)
            win_rows.update(range(pos - nwin + 1, pos + 1))
            if topk_idx is not None:
                row = topk_idx[b * S + s]
                sel.update(int(x) for x in row[row >= 0])
            else:
                sel.update(range(min(vis, cfg.topk)))
            if vis > cfg.topk:
                krows = max(krows, vis)
                idx_b += cfg.Hi * cfg.Di * e + 4 * cfg.Hi
            if cfg.hca_ratio:
                hca_rows = max(hca_rows, (pos + 1) // cfg.hca_ratio)
        idx_b += krows * key_row
        tot_rows += len(win_rows) + len(sel) + hca_rows
        tot_q += S
    attn_b = tot_q * (cfg.H * cfg.D * e + cfg.H * cfg.V * e) + tot_rows * cfg.D * e
    return {"total": attn_b + idx_b, "indexer": idx_b, "attention": attn_b}


# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
def cpu_baseline(wl, hb, budget_s=6.0, threads=None):
    """The oracle as it stands, on the host cores, over a bounded sample of
    queries: the first max(16, threads) queries of the batch (one oracle
    thread per query, so every thread has a query), repeated for about
    budget_s seconds.  threads=None uses every host core."""
    import numpy as np
    import oracle
    oracle.build()
    cores = threads or os.cpu_count() or 1
    T = hb["B"] * hb["S"]
    nq = min(T, max(16, cores))
    used = min(cores, nq)
    qids = np.arange(nq, dtype=np.int32)
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.decode(wl.cfg, hb, qids=qids, nthreads=used)
        done += qids.size
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": done / el, "unit": "queries/s", "cores": used, "kind": "oracle",
            "sample": f"{nq} queries of {wl.name} (the first {nq} of the batch, their full context), "
                      f"repeated {done // nq}x, fp64 C oracle, {used} thread(s), {el:.1f} s wall"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from compressed_sparse_attention_indexer_gb300.workloads import WORKLOADS, make_batch
    import numpy as np
    import oracle
    oracle.build()
    wl = WORKLOADS[args.workload]
    hb = make_batch(wl)
    cores = os.cpu_count() or 1
    T = hb["B"] * hb["S"]
    nq = min(T, max(cores, 8))
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        oracle.decode(wl.cfg, hb, qids=rng.choice(T, nq, replace=False).astype(np.int32), nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode(wl.cfg, hb, qids=rng.choice(T, nq, replace=False).astype(np.int32), nthreads=cores)
    el = time.perf_counter() - t0
    value = nq * args.steps / el
    line = {"impl": "reference", "metric": "csa_decode_queries_per_s", "value": value,
            "unit": "queries/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "B": hb["B"], "S": hb["S"],
                       "description": wl.description},
            "cpu_baseline": {"value": value, "unit": "queries/s", "cores": min(cores, nq), "kind": "oracle",
                             "sample": f"{nq} random queries of {wl.name} per step (full context each)"},
            "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def src_sha(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


# sources of the kernels each stage runs by default (a recorded traffic figure
# is dropped once any of them changes)
_C = "compressed_sparse_attention_indexer_gb300/csrc/"
KERNEL_SOURCES = {
    "indexer": [_C + "indexer_tc5.cu", _C + "tc5.cuh", _C + "ptx.cuh", _C + "csa_internal.cuh"],
    "attention": [_C + "attention_tc5.cu", _C + "tc5.cuh", _C + "ptx.cuh", _C + "csa_internal.cuh"],
    "topk": [_C + "topk.cu", _C + "ptx.cuh", _C + "csa_internal.cuh"],
    "plan": [_C + "plan.cu", _C + "csa_internal.cuh"],
}


def load_traffic(kernel: str, workload: str):
    """ncu-measured DRAM bytes per launch, if recorded for the current kernel source."""
    p = os.path.join(ROOT, "profiles", f"traffic_{kernel}_{workload}.json")
    try:
        d = json.load(open(p))
    except Exception:
        return None
    if d.get("source_sha") != src_sha(KERNEL_SOURCES.get(kernel, d.get("sources", []))):
        return None
    return d.get("dram_bytes_per_launch")


def e2e_group_sizes(n: int, G: int) -> list:
    """The end-to-end loop's groups for n steps: one step, then groups of G,
    the rest, and one step (exactly n steps; no group empty or above G)."""
    if n <= 2:
        return [1] * n
    mid, sizes = n - 2, [1]
    sizes += [G] * (mid // G) + ([mid % G] if mid % G else [])
    return sizes + [1]


def run_e2e(args, csa, dec, hb, copies, lens_host, out, idx, cnt, stream, dev, T, ws, dist):
    """The same step through the public API with host buffers, as a serving
    loop runs it: every step copies its activations (q, q_idx, w, lengths,
    pool offsets) from pinned host memory in one packed H2D copy and reads its
    output back D2H.  The copies run on their own streams, so step i+1's
    upload and step i-1's download overlap step i's kernels; the KV and
    indexer caches are resident state and are not copied."""
    import torch
    keys = ("q", "q_idx", "w", "ctx_len", "raw_off", "cmp_off", "idx_off")
    offs, tot, h2d = {}, 0, 0
    for k in keys:
        nb = hb[k].numel() * hb[k].element_size()
        offs[k] = (tot, nb)
        tot += (nb + 255) // 256 * 256
        h2d += nb
    host_buf = torch.empty(tot, dtype=torch.uint8, pin_memory=True)
    for k in keys:
        o, nb = offs[k]
        host_buf[o:o + nb].copy_(hb[k].contiguous().view(-1).view(torch.uint8))
    # Steps go in groups of up to G: a group's uploads are issued while the
    # previous group runs, and the compute stream meets the copy streams only
    # between groups (one wait before a group, one event after it), so the
    # kernels of a group's consecutive steps stay chained by programmatic
    # dependent launch.  The first and the last group hold one step, so that
    # only one step's upload precedes the first kernels and only one step's
    # read-back follows the last.  Every step still uploads its own inputs and
    # reads back its own output.
    G = 4
    nbuf = 2 * G
    dev_bufs = [torch.empty(tot, dtype=torch.uint8, device=dev) for _ in range(nbuf)]

    def view(buf, k):
        o, nb = offs[k]
        return buf[o:o + nb].view(hb[k].dtype).view(hb[k].shape)

    structs = []
    for j in range(nbuf):
        c = dict(copies[j % len(copies)])
        for k in keys:
            c[k] = view(dev_bufs[j], k)
        structs.append(csa.make_batch_struct(c, lens_host))
    outs = [torch.empty_like(out) for _ in range(nbuf)]
    out_host = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(nbuf)]
    d2h = out_host[0].numel() * out_host[0].element_size()
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]   # per group parity
    x_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]

    def upload(g, size):  # group g's inputs into buffers (g % 2) * G ...
        p = g % 2
        if g >= 2:
            up.wait_event(x_done[p])          # group g - 2 has run on these buffers
        with torch.cuda.stream(up):
            for t in range(size):
                dev_bufs[p * G + t].copy_(host_buf, non_blocking=True)
        h2d_done[p].record(up)

    def run_group(g, size):
        p = g % 2
        stream.wait_event(h2d_done[p])
        if g >= 2:
            stream.wait_event(d2h_done[p])    # group g - 2's outputs have been read back
        for t in range(size):
            dec.decode_step(structs[p * G + t], outs[p * G + t], None, idx, cnt, stream)
        x_done[p].record(stream)
        down.wait_event(x_done[p])
        with torch.cuda.stream(down):
            for t in range(size):
                out_host[p * G + t].copy_(outs[p * G + t], non_blocking=True)
        d2h_done[p].record(down)
        return out_host[p * G + size - 1]

    def run_steps(n):
        sizes = e2e_group_sizes(n, G)
        upload(0, sizes[0])
        last = None
        for g, size in enumerate(sizes):
            if g + 1 < len(sizes):
                upload(g + 1, sizes[g + 1])
            last = run_group(g, size)
        return last

    run_steps(max(args.warmup, 2 * G))
    torch.cuda.synchronize()
    nsteps = max(args.steps, 1)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    last = run_steps(nsteps)
    e1.record(down)
    torch.cuda.synchronize()
    ems = reduce_max(e0.elapsed_time(e1) / nsteps, dist, dev)
    # the pipelined step computes what the device-resident step computes
    if not torch.equal(last, out.cpu()):
        raise RuntimeError("end-to-end output differs from the device-resident step")
    return {"value": job_throughput(T, ws, ems), "unit": "queries/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ems,
            "note": "per step: activations (q, q_idx, w, lengths, pool offsets) in one packed H2D "
                    "copy from pinned memory, the output D2H; copies on their own streams overlap "
                    "the neighbouring steps' kernels; KV/indexer caches stay resident"}


def measure(args, name, steps, warmup, dev, ws, rank, dist, with_e2e, with_cpu):
    """One workload: K timed steps through csa_decode_step (inputs resident in
    HBM, rotated over device copies), per-stage times, roofline of the
    dominant stage, optionally the end-to-end leg and the oracle baseline."""
    import torch

    from compressed_sparse_attention_indexer_gb300 import csa
    from compressed_sparse_attention_indexer_gb300.workloads import WORKLOADS, make_batch, to_device

    wl = WORKLOADS[name]
    cfg = wl.cfg
    # weak scaling: every rank decodes its own batch (different seed per rank)
    hb = make_batch(wl, seed=rank_seed(wl.seed, rank))
    B, S = hb["B"], hb["S"]
    T = B * S
    lens = [int(x) for x in hb["ctx_len"]]
    max_ctx = 65536 if name.startswith("long_ragged") else max(lens)
    copies = [to_device(hb, dev)]
    for _ in range(args.copies - 1):
        copies.append({k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in copies[0].items()})
    lens_host = hb["ctx_len"].clone()
    structs = [csa.make_batch_struct(c, lens_host) for c in copies]
    dec = csa.Decoder(cfg, B, S, max_ctx)
    out = torch.empty(B, S, cfg.H, cfg.V, dtype=cfg.torch_dtype, device=dev)
    idx = torch.empty(B, S, cfg.topk, dtype=torch.int32, device=dev)
    cnt = torch.empty(B, S, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        dec.decode_step(structs[i % len(structs)], out, None, idx, cnt, stream)

    # a first step gives the status, the launch count and the selection the
    # algorithmic bytes are counted from
    step(0)
    torch.cuda.synchronize()
    st = dec.status()
    if st != csa.CSA_OK:
        raise RuntimeError(f"{name}: device status {st}: {csa.last_error()}")
    launches_per_step = dec.last_launch_count()
    sel = idx.cpu().numpy().reshape(T, cfg.topk)
    bytes_ = step_bytes(cfg, lens, S, sel)

    # ---- W warm-up steps right before the timed region (the clock sampler is
    # started first: its start-up, and the host work above, leave the GPU idle,
    # which a timed region that follows directly would pay for), then K steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        for i in range(max(warmup, 3)):
            step(i)
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = reduce_max(ev0.elapsed_time(ev1) / steps, dist if ws > 1 else None, dev)
    st = dec.status()
    if st != csa.CSA_OK:
        raise RuntimeError(f"{name}: device status {st} after the timed steps: {csa.last_error()}")
    if ws > 1:
        dist.barrier()

    # ---- per-kernel times (events around each launch, same stream), separate pass
    dec.profile(True)
    for i in range(steps):
        step(i)
    torch.cuda.synchronize()
    prof = dec.profile_read()
    dec.profile(False)
    per_kernel_ms = {k: (v[0] / v[1] if v[1] else 0.0) for k, v in prof.items()}
    dom = max(("indexer", "attention", "topk"), key=lambda k: prof[k][0])
    peak, peak_kind, _ = measured_peaks()
    alg = bytes_[dom] if dom in bytes_ else None
    achieved = alg / (per_kernel_ms[dom] * 1e-3) / 1e9 if (alg and per_kernel_ms[dom] > 0) else None
    roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": (achieved / peak) if achieved else None, "peak_source": peak_kind,
            "algorithmic_bytes_per_launch": alg,
            "traffic": load_traffic(dom, name),
            "per_kernel_us": {k: round(v * 1e3, 3) for k, v in per_kernel_ms.items()},
            "time_share": {k: round(v[0] / max(sum(x[0] for x in prof.values()), 1e-9), 4)
                           for k, v in prof.items()},
            "step_achieved_gbs": bytes_["total"] / (ms * 1e-3) / 1e9,
            "step_frac": bytes_["total"] / (ms * 1e-3) / 1e9 / peak}

    # ---- end to end through the public API with host buffers
    e2e = None
    if with_e2e:
        e2e = run_e2e(args, csa, dec, hb, copies, lens_host, out, idx, cnt, stream, dev, T, ws,
                      dist if ws > 1 else None)
    cpu = cpu1 = None
    if with_cpu:
        cpu = cpu_baseline(wl, hb, budget_s=args.cpu_seconds)
        cpu1 = cpu_baseline(wl, hb, budget_s=max(2.0, args.cpu_seconds / 3), threads=1)
    foot = sum(v.numel() * v.element_size() for v in copies[0].values() if isinstance(v, torch.Tensor))
    res = {
        "value": job_throughput(T, ws, ms), "unit": "queries/s", "ms_per_step": ms, "steps": steps,
        "dtype": cfg.dtype,
        "config": {"workload": wl.name, "B": B, "S": S, "H": cfg.H, "D": cfg.D, "K": cfg.topk,
                   "WIN": cfg.win, "L_range": list(wl.L_range) if wl.L_range else wl.L,
                   "sum_L": int(sum(lens)), "parallelism": f"replicas{ws}",
                   "l2": f"inputs rotate over {len(copies)} device copies ({foot / 1e9:.2f} GB each); "
                         f"each step reads ~{bytes_['total'] / 1e6:.1f} MB (L2 {L2_BYTES / 1e6:.0f} MB)",
                   "algorithmic_bytes_per_step": bytes_["total"]},
        "achieved_hbm_gbs": bytes_["total"] / (ms * 1e-3) / 1e9,
        "roofline": roof, "cpu_baseline": cpu, "cpu_baseline_1core": cpu1, "e2e": e2e,
        "clocks": clk.summary(), "gpu_launches": launches_per_step * steps,
        "launches_per_step": launches_per_step,
    }
    dec.close()
    del copies, structs
    torch.cuda.empty_cache()
    return res


# the other named workloads, measured after the headline one (their shapes are
# the pages' decode shapes, the Top-K-active and multi-token variants, the
# prefill chunk and the FP8-key cache)
OTHER_WORKLOADS = ("tiny_f32", "bypass_b16_l256", "topk_b16_l8192", "multitoken_hca_b16_s8",
                   "prefill_b2_t512", "long_ragged_b64_fp8idx")


def run_ours(args):
    import torch

    from compressed_sparse_attention_indexer_gb300 import build as csa_build

    ws, rank, local = dist_env()
    dist = None
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    csa_build.build()
    head = measure(args, args.workload, args.steps, args.warmup, dev, ws, rank, dist,
                   with_e2e=not args.no_e2e, with_cpu=(ws == 1 and rank == 0 and not args.no_cpu_baseline))
    others = {}
    names = [] if args.workloads == "none" else (
        [n for n in OTHER_WORKLOADS if n != args.workload] if args.workloads == "all" else args.workloads.split(","))
    for n in names:
        r = measure(args, n, min(args.steps, args.other_steps), args.warmup, dev, ws, rank, dist,
                    with_e2e=False, with_cpu=(ws == 1 and rank == 0 and not args.no_cpu_baseline))
        others[n] = {k: r[k] for k in ("value", "unit", "ms_per_step", "steps", "dtype", "achieved_hbm_gbs",
                                       "roofline", "cpu_baseline", "cpu_baseline_1core", "launches_per_step")}
        others[n]["config"] = r["config"]
    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    line = {
        "metric": "csa_decode_queries_per_s", "value": head["value"], "unit": "queries/s",
        "n_gpus": ws, "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
        "data": "synthetic (seeded normal / uniform draws, shapes of the workload)",
        "config": head["config"],
        "achieved_hbm_gbs": head["achieved_hbm_gbs"],
        "roofline": head["roofline"], "cpu_baseline": head["cpu_baseline"],
        "cpu_baseline_1core": head["cpu_baseline_1core"], "e2e": head["e2e"],
        "clocks": head["clocks"], "gpu_launches": head["gpu_launches"],
        "launches_per_step": head["launches_per_step"],
        "workloads": others,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
