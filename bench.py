#!/usr/bin/env python
"""Decode-step benchmark of the LOCKS sparse decode path on one GB300.

A step is one layer's decode step for the whole batch: score every full page
from its summary, select the GQA-shared page set, attend over the selected
pages.  Summaries are built once before timing (the build is reported
separately).  Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W]
                    [--impl locks|reference] [--workload NAME] [--batch B]
                    [--quick [--ablation]] [--ctx T]

Under torchrun every rank runs its own replica of the workload (the path
shards by sequence with no exchange step), so `value` is the sum over ranks
and scaling is weak.  `--impl reference` times the float64 oracle on the
host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# The float64 oracle (CPU baseline and reference arm) runs its BLAS on every
# core this process may use; set before numpy is first imported.
try:
    _CORES = len(os.sched_getaffinity(0))
except AttributeError:
    _CORES = os.cpu_count() or 1
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

METRIC = ("decode tokens/s per layer (score+select+sparse attn) @128K; "
          "% HBM roofline")
RECORD_PAYLOAD = 818          # algorithmic bytes of one page summary
KV_PAGE_HEAD = 2 * 16 * 128 * 2  # K + V bytes of one full page-head (bf16)
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="locks", choices=["locks", "reference"])
    p.add_argument("--workload", default="llama8b_128k")
    p.add_argument("--batch", type=int, default=0,
                   help="override the workload's batch (profiling cases)")
    p.add_argument("--ctx", type=int, default=0,
                   help="override the workload's context length in tokens "
                        "(profiling cases: the decode work is batch x h_kv x "
                        "k pages whatever the context)")
    p.add_argument("--quick", action="store_true",
                   help="skip e2e, dense context, build timing and CPU "
                        "baseline (profiling runs)")
    p.add_argument("--ablation", action="store_true",
                   help="with --quick: run the rank / precision ablation "
                        "as well (profiling the variant kernels)")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(x: float) -> float:
    """Max of a scalar over ranks (the slowest rank sets the job time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_spec(spec, rank: int, batch: int = 0, ctx: int = 0):
    """Each rank runs its own replica: same shape, its own seed."""
    kw = {"seed": spec.seed + 7919 * rank}
    if batch:
        kw["batch"] = batch
    if ctx:
        kw["ctx"] = ctx
    return dataclasses.replace(spec, **kw)


# ---------------------------------------------------------------------------
# measurement helpers
# ---------------------------------------------------------------------------
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}",
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"),
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def _sha256(path):
    import hashlib
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def step_traffic(units, group):
    """DRAM bytes of one decode step from the committed small-case ncu
    captures (profiles/step_traffic.json): for each kernel of the step,
    dram__bytes_read.sum + dram__bytes_write.sum per unit of work (record,
    score entry, selected page-head) times the units of this step.  Returns
    (total, {kernel: bytes}) or (None, reason) when a kernel's source
    changed since its capture or the group size selects another form of a
    kernel than the captured one."""
    try:
        with open(os.path.join(ROOT, "profiles", "step_traffic.json")) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None, "no capture"
    if d.get("group_size") != group:
        return None, f"captured at group size {d.get('group_size')}"
    out = {}
    for name, k in d["kernels"].items():
        for f in k["sources"]:
            src = os.path.join(ROOT, "sparse_paged_kv_locks_gb300", "csrc", f)
            try:
                if _sha256(src) != k["source_sha256"][f]:
                    return None, f"{f} changed since the {name} capture"
            except OSError:
                return None, f"{f} missing"
        out[name] = round(float(k["dram_bytes_per_unit"]) *
                          units[k["unit"]])
    return sum(out.values()), out


def build_issue(n_page_heads, build_ms, sm_mhz):
    """Fraction of the instruction-issue floor the summary build reaches:
    warp instructions per page-head from the committed ncu capture
    (profiles/build_kernel_instructions.json), one warp instruction per
    scheduler per cycle on every SM (4 schedulers per SM) at the sampled SM
    clock.  None when csrc/build.cu changed since the capture."""
    import hashlib

    import torch
    try:
        with open(os.path.join(ROOT, "profiles",
                               "build_kernel_instructions.json")) as f:
            d = json.load(f)
        src = os.path.join(ROOT, "sparse_paged_kv_locks_gb300", "csrc",
                           "build.cu")
        with open(src, "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
    except (OSError, ValueError):
        return None
    if d.get("build_cu_sha256") != digest or not sm_mhz:
        return None
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    per = float(d["warp_instructions_per_page_head"])
    floor_ms = n_page_heads * per / (n_sm * 4 * sm_mhz * 1e6) * 1e3
    return {"bound": "issue", "warp_instructions_per_page_head": per,
            "floor_ms": round(floor_ms, 3),
            "frac": round(floor_ms / build_ms, 4),
            "peak": f"{n_sm} SMs x 4 schedulers x {sm_mhz:.0f} MHz"}


def small_configs(B, W, dev, n_steps=200):
    """The two small workloads (tiny_4k: 1 x 4K, 8q/2kv, k = 16;
    llama8b_32k: 8 x 32K, 32q/8kv, k = 64), which fit largely in the
    129 MB L2: the same decode step (score + select + sparse attention),
    timed warm (steps launched back to back from the host), with the L2
    flushed before every step (a 2 x L2 buffer written between steps,
    outside the timed events), and warm as one CUDA graph replay per step
    (these steps are launch-bound without it)."""
    import torch
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    out = {}
    for name in ("tiny_4k", "llama8b_32k"):
        spec = W.SPECS[name]
        wl = W.generate(spec, dev)
        lens = [int(x) for x in wl.seq_lens]
        batch, max_pages = wl.page_table.shape
        seq = torch.tensor([b for b in range(batch)
                            for _ in range(lens[b] // 16)],
                           dtype=torch.int32, device=dev)
        pgs = torch.tensor([p for b in range(batch)
                            for p in range(lens[b] // 16)],
                           dtype=torch.int32, device=dev)
        store = B.new_summary_store(batch, spec.h_kv, max_pages, dev)
        B.locks_build_summaries(wl.k_cache, wl.page_table, seq, pgs, store)
        ws = B.new_workspace(batch, spec.h_q, spec.h_kv, max_pages, spec.k,
                             dev)
        idx = torch.empty(batch, spec.h_kv, spec.k, dtype=torch.int32,
                          device=dev)
        o = torch.empty(batch, spec.h_q, 128, dtype=torch.bfloat16,
                        device=dev)
        lse = torch.empty(batch, spec.h_q, dtype=torch.float32, device=dev)
        qs = wl.queries

        def step(i):
            q = qs[i % qs.shape[0]]
            B.locks_score_select(q, store, wl.seq_lens, spec.k, idx, ws)
            B.locks_sparse_decode(q, wl.k_cache, wl.v_cache, wl.page_table,
                                  wl.seq_lens, idx, spec.k, o, lse, ws)

        for i in range(5):
            step(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(
            enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for i in range(n_steps):
            step(i)
        e1.record()
        torch.cuda.synchronize()
        warm = e0.elapsed_time(e1) / n_steps
        cold = []
        for i in range(min(n_steps, 50)):
            flush.fill_(float(i))
            e0.record()
            step(i)
            e1.record()
            torch.cuda.synchronize()
            cold.append(e0.elapsed_time(e1))
        assert B.locks_read_status(ws) == 0
        cold_ms = statistics.mean(cold)
        # the same step replayed as one CUDA graph (no host launch per
        # kernel), query already on the device
        dec = B.LocksDecoder(wl.k_cache, wl.v_cache, wl.page_table, store,
                             spec.h_q, spec.k, graph=True,
                             seq_lens=wl.seq_lens)
        dec.q_dev.copy_(qs[0])
        for _ in range(5):
            dec.step(dec.q_dev)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(n_steps):
            dec.step(dec.q_dev)
        e1.record()
        torch.cuda.synchronize()
        graph_ms = e0.elapsed_time(e1) / n_steps
        assert dec.status() == 0
        out[name] = {"batch": batch, "context": spec.ctx, "k": spec.k,
                     "warm": {"ms_per_step": round(warm, 4),
                              "tokens_per_s": round(batch / (warm / 1e3))},
                     "l2_flushed": {"ms_per_step": round(cold_ms, 4),
                                    "tokens_per_s":
                                        round(batch / (cold_ms / 1e3))},
                     "graph_warm": {"ms_per_step": round(graph_ms, 4),
                                    "tokens_per_s":
                                        round(batch / (graph_ms / 1e3))}}
        del wl, store, ws, dec
        torch.cuda.empty_cache()
    return out


def ragged_config(B, W, dev, peak_gbs, n_steps=50):
    """The ragged serving batch (ragged_64: 64 sequences with lengths
    U{4096..131072}, most ending in a partial page, 32q/8kv) over the
    budget sweep k = 16..256 pages: the decode step (score + select +
    sparse attention) timed back to back on the device; the summaries
    (about 1.8 GB) are larger than L2 at every k.  Algorithmic bytes per
    step as on the main workload: summaries of every full page, the
    selected pages' valid K/V tokens, q and o."""
    import torch
    spec = W.SPECS["ragged_64"]
    wl = W.generate(spec, dev)
    lens = [int(x) for x in wl.seq_lens]
    batch, max_pages = wl.page_table.shape
    seq = torch.tensor([b for b in range(batch)
                        for _ in range(lens[b] // 16)],
                       dtype=torch.int32, device=dev)
    pgs = torch.tensor([p for b in range(batch)
                        for p in range(lens[b] // 16)],
                       dtype=torch.int32, device=dev)
    store = B.new_summary_store(batch, spec.h_kv, max_pages, dev)
    B.locks_build_summaries(wl.k_cache, wl.page_table, seq, pgs, store)
    k_max = max(spec.k_sweep)
    ws = B.new_workspace(batch, spec.h_q, spec.h_kv, max_pages, k_max, dev)
    o = torch.empty(batch, spec.h_q, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(batch, spec.h_q, dtype=torch.float32, device=dev)
    qs = wl.queries
    n_full = sum(L // 16 for L in lens)
    score_bytes = n_full * spec.h_kv * RECORD_PAYLOAD
    q_bytes = batch * spec.h_q * 128 * 2
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(
        enable_timing=True)
    sweep = []
    for k in spec.k_sweep:
        idx = torch.empty(batch, spec.h_kv, k, dtype=torch.int32, device=dev)

        def step(i):
            q = qs[i % qs.shape[0]]
            B.locks_score_select(q, store, wl.seq_lens, k, idx, ws)
            B.locks_sparse_decode(q, wl.k_cache, wl.v_cache, wl.page_table,
                                  wl.seq_lens, idx, k, o, lse, ws)

        for i in range(5):
            step(i)
        torch.cuda.synchronize()
        e0.record()
        for i in range(n_steps):
            step(i)
        e1.record()
        torch.cuda.synchronize()
        assert B.locks_read_status(ws) == 0
        ms = e0.elapsed_time(e1) / n_steps
        # K/V bytes of the last step's selection (valid tokens only)
        idx_h = idx.cpu().numpy()
        kv_bytes = 0
        for b in range(batch):
            for h in range(spec.h_kv):
                for p in idx_h[b, h]:
                    if p >= 0:
                        kv_bytes += min(16, lens[b] - 16 * int(p)) * 2 * 128 * 2
        step_bytes = score_bytes + kv_bytes + 2 * q_bytes
        gbs = step_bytes / (ms / 1e3) / 1e9
        sweep.append({"k": k, "ms_per_step": round(ms, 4),
                      "tokens_per_s": round(batch / (ms / 1e3)),
                      "algorithmic_bytes": step_bytes,
                      "gbs": round(gbs, 1),
                      "frac_of_copy_peak": round(gbs / peak_gbs, 4)})
    out = {"batch": batch, "h_q": spec.h_q, "h_kv": spec.h_kv,
           "context_min": min(lens), "context_max": max(lens),
           "context_mean": round(statistics.mean(lens)),
           "partial_last_pages": sum(1 for L in lens if L % 16),
           "steps": n_steps, "sweep": sweep}
    del wl, store, ws
    torch.cuda.empty_cache()
    return out


def append_config(B, W, dev, sm_mhz, n_steps=64):
    """The append workload (llama70b_128k_append: 8 x 131072 tokens,
    64q/8kv, k = 128): the summary build of the whole cache at the
    prefill/decode boundary (524,288 page-heads, timed on its own, warm), then
    steps that each append one token per sequence (writing K and V and
    building the summary of a page the append fills, once every 16 steps
    here) and run the decode step; the incremental build is part of the
    step.  CUDA events around the build, the append (launched alone) and
    the whole step (replayed as one CUDA graph)."""
    import torch
    spec = W.SPECS["llama70b_128k_append"]
    wl = W.generate(spec, dev)
    lens0 = [int(x) for x in wl.seq_lens]
    batch, max_pages = wl.page_table.shape
    seq = torch.tensor([b for b in range(batch)
                        for _ in range(lens0[b] // 16)],
                       dtype=torch.int32, device=dev)
    pgs = torch.tensor([p for b in range(batch)
                        for p in range(lens0[b] // 16)],
                       dtype=torch.int32, device=dev)
    store = B.new_summary_store(batch, spec.h_kv, max_pages, dev)
    B.locks_build_summaries(wl.k_cache, wl.page_table, seq, pgs, store)
    b0, b1 = torch.cuda.Event(True), torch.cuda.Event(True)
    torch.cuda.synchronize()
    b0.record()
    B.locks_build_summaries(wl.k_cache, wl.page_table, seq, pgs, store)
    b1.record()
    torch.cuda.synchronize()
    build_ms = b0.elapsed_time(b1)
    n_build = int(seq.numel()) * spec.h_kv
    ws = B.new_workspace(batch, spec.h_q, spec.h_kv, max_pages, spec.k, dev)
    idx = torch.empty(batch, spec.h_kv, spec.k, dtype=torch.int32,
                      device=dev)
    o = torch.empty(batch, spec.h_q, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(batch, spec.h_q, dtype=torch.float32, device=dev)
    lens = wl.seq_lens.clone()
    n_eager = 32
    n_steps = min(n_steps, spec.append_steps - n_eager)
    # the append alone, launched eagerly with events around it (a plain
    # append and one that fills a page and builds its summary)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
          for _ in range(n_eager)]
    torch.cuda.synchronize()
    for s in range(n_eager):
        q = wl.queries[s % wl.queries.shape[0]]
        ev[s][0].record()
        B.locks_append_kv(wl.k_append[s], wl.v_append[s], wl.k_cache,
                          wl.v_cache, wl.page_table, lens, store)
        ev[s][1].record()
        B.locks_score_select(q, store, lens, spec.k, idx, ws)
        B.locks_sparse_decode(q, wl.k_cache, wl.v_cache, wl.page_table, lens,
                              idx, spec.k, o, lse, ws)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == 0
    fills = [s for s in range(n_eager) if (lens0[0] + s + 1) % 16 == 0]
    plain = [s for s in range(n_eager) if s not in fills and s >= 2]
    app = [ev[s][0].elapsed_time(ev[s][1]) for s in range(n_eager)]
    # the whole step -- append (with the page build when a page fills),
    # score, select, sparse attention -- replayed as one CUDA graph; the
    # step's inputs are staged in the decoder's buffers before the events
    dec = B.LocksDecoder(wl.k_cache, wl.v_cache, wl.page_table, store,
                         spec.h_q, spec.k, graph=True, seq_lens=lens,
                         append=True)
    evg = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
           for _ in range(n_steps)]
    for i in range(n_steps):
        s = n_eager + i
        dec.q_dev.copy_(wl.queries[s % wl.queries.shape[0]])
        dec.k_new.copy_(wl.k_append[s])
        dec.v_new.copy_(wl.v_append[s])
        evg[i][0].record()
        dec.step(dec.q_dev, k_new=dec.k_new, v_new=dec.v_new)
        evg[i][1].record()
    torch.cuda.synchronize()
    assert dec.status() == 0
    step = [evg[i][0].elapsed_time(evg[i][1]) for i in range(2, n_steps)]
    res = {"batch": batch, "context": spec.ctx, "h_q": spec.h_q,
           "h_kv": spec.h_kv, "k": spec.k, "steps": n_steps,
           "append_us": round(1e3 * statistics.median(
               [app[s] for s in plain]), 2),
           "append_filling_a_page_us": round(1e3 * statistics.median(
               [app[s] for s in fills]), 2) if fills else None,
           "step_ms": round(statistics.mean(step), 4),
           "step": "append + score + select + sparse attention replayed as "
                   "one CUDA graph (LocksDecoder(graph=True, append=True)); "
                   "mean over steps, one in 16 of which fills a page",
           "tokens_per_s": round(batch / (statistics.mean(step) / 1e3)),
           "boundary_build": {
               "page_heads": n_build, "ms": round(build_ms, 3),
               "page_heads_per_s": round(n_build / (build_ms / 1e3)),
               "roofline": build_issue(n_build, build_ms, sm_mhz)}}
    del wl, store, ws, dec
    torch.cuda.empty_cache()
    return res


def selection_quality(B, wl, store, scores, ws, lens, k, h_q, n_records,
                      n_steps=4):
    """Selection quality on the planted needles, GPU only.  The pages
    holding a needle token (carrier pages) kept by the LOCKS selection and
    by the exact-mass selection (exact page LSE from every key, the
    selector the LOCKS notes compare against in §6 Fig. 1(b)), over a budget
    sweep; the page-score error of the quantised summaries against the
    exact page LSE (the measured counterpart of eta, Eq.(6)); and the exact
    scorer's time and bandwidth (it reads every full page's keys)."""
    import torch
    dev = scores.device
    batch, h_kv, G, max_pages = scores.shape
    ex = torch.empty_like(scores)
    status = ws[:4].view(torch.int32)
    sweep = [kk for kk in (16, 32, 64, 128) if kk <= k] or [k]
    needles = wl.needle_pages.to(dev)                     # [b][h_kv][nn]
    hit_l = {kk: 0 for kk in sweep}
    hit_e = {kk: 0 for kk in sweep}
    n_car = 0
    err_max, err_sum, err_cnt, p99 = 0.0, 0.0, 0, []
    times = []
    rules = ("share_average", "group_max", "group_mass", "per_head")
    # per-head selection treats every query head as its own group
    ws_ph = B.new_workspace(batch, h_q, h_q, max_pages, k, dev)
    coverage = {r: [] for r in rules}
    e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
    n_steps = min(n_steps, wl.queries.shape[0])
    for i in range(n_steps):
        q = wl.queries[i]
        B.locks_score_pages(q, store, wl.seq_lens, scores, status)
        e0.record()
        B.locks_exact_page_scores(q, wl.k_cache, wl.page_table, wl.seq_lens,
                                  ex, status)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
        for b in range(batch):
            nf = lens[b] // 16
            d = (scores[b, :, :, :nf] - ex[b, :, :, :nf]).abs().flatten()
            err_max = max(err_max, float(d.max()))
            err_sum += float(d.double().sum())
            err_cnt += d.numel()
            p99.append(float(torch.kthvalue(
                d.cpu(), max(1, int(0.99 * d.numel()))).values))
        n_car += int((needles >= 0).sum())
        # exact mass fractions of every full page, per head
        mass = torch.zeros_like(ex)
        for b in range(batch):
            nf = lens[b] // 16
            if nf:
                mass[b, :, :, :nf] = torch.softmax(ex[b, :, :, :nf].double(),
                                                   -1).float()
        for rule in rules:
            idx = torch.empty(batch, h_kv, k, dtype=torch.int32, device=dev)
            if rule == "per_head":
                idx = torch.empty(batch, h_q, k, dtype=torch.int32,
                                  device=dev)
                B.locks_select_pages(scores.view(batch, h_q, 1, max_pages),
                                     wl.seq_lens, h_q, k, idx, ws_ph)
                idx = idx.view(batch, h_kv, G, k)
            else:
                B.locks_select_pages_merge(scores, wl.seq_lens, h_q, k, rule,
                                           idx, ws)
                idx = idx[:, :, None, :].expand(batch, h_kv, G, k)
            valid = idx >= 0
            cov = torch.gather(mass, 3, idx.clamp(min=0).long())
            coverage[rule].append((cov * valid).sum(-1))     # [b][h][G]
        for kk in sweep:
            for src, hits in ((scores, hit_l), (ex, hit_e)):
                idx = torch.empty(batch, h_kv, kk, dtype=torch.int32,
                                  device=dev)
                B.locks_select_pages(src, wl.seq_lens, h_q, kk, idx, ws)
                kept = (idx[:, :, None, :] == needles[:, :, :, None]).any(-1)
                hits[kk] += int((kept & (needles >= 0)).sum())
    assert B.locks_read_status(ws) == 0, "quality pass reported an error"
    assert B.locks_read_status(ws_ph) == 0, "quality pass reported an error"
    ms = statistics.mean(times)
    merge = {}
    for r in rules:
        c = torch.stack(coverage[r])                        # [steps][b][h][G]
        flat = c.flatten().double()
        merge[r] = {"mean": round(float(flat.mean()), 4),
                    "worst_head": round(float(c.min(-1).values.mean()), 4),
                    "p5": round(float(torch.quantile(flat, 0.05)), 4)}
    return {
        "budget_pages": sweep,
        "carrier_retention": {
            "locks": [round(hit_l[kk] / max(1, n_car), 4) for kk in sweep],
            "exact_mass": [round(hit_e[kk] / max(1, n_car), 4)
                           for kk in sweep]},
        "carrier_pages": n_car // n_steps, "steps": n_steps,
        "gqa_merge_coverage": {"budget_pages": k, "rules": merge,
                               "note": "exact attention mass kept per "
                                       "query head, selections from the "
                                       "summaries' scores"},
        "score_error_vs_exact": {"max": round(err_max, 4),
                                 "mean": round(err_sum / max(1, err_cnt), 5),
                                 "p99_per_sequence_max": round(max(p99), 4)},
        "exact_scorer": {"ms": round(ms, 4),
                         "gbs": round(n_records * 4096 / (ms / 1e3) / 1e9,
                                      1)}}


def rank_precision_ablation(B, wl, lens, k, h_q, peak_gbs, n_seqs=4,
                            n_steps=2):
    """The notes' rank / basis-precision ablation (§6) on the first n_seqs
    sequences of the workload: for every variant, carrier retention on the
    planted needles, exact coverage and page-score error against the exact
    LSE at budget k, with the variant's record bytes (the scoring stream's
    bytes per page-head) and its build and scoring times (scoring: mean of
    10 calls after warm-up, each after an L2 flush); the scoring stream's
    rate against the measured copy peak."""
    import torch
    dev = wl.k_cache.device
    batch = min(n_seqs, wl.page_table.shape[0])
    pt = wl.page_table[:batch].contiguous()
    sl = wl.seq_lens[:batch].contiguous()
    max_pages = pt.shape[1]
    h_kv = wl.k_cache.shape[1]
    G = h_q // h_kv
    seq = torch.tensor([b for b in range(batch) for _ in range(lens[b] // 16)],
                       dtype=torch.int32, device=dev)
    pgs = torch.tensor([p for b in range(batch) for p in range(lens[b] // 16)],
                       dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = B.new_workspace(batch, h_q, h_kv, max_pages, k, dev)
    sc = torch.zeros(batch, h_kv, G, max_pages, device=dev)
    ex = torch.zeros_like(sc)
    idx = torch.empty(batch, h_kv, k, dtype=torch.int32, device=dev)
    needles = wl.needle_pages[:batch].to(dev)
    e0, e1, e2 = (torch.cuda.Event(True) for _ in range(3))
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    n_time = 10

    def time_scoring(call):
        # warm launches, then n_time calls each after an L2 flush (the
        # smaller variant stores fit in L2)
        for _ in range(3):
            call()
        ms = []
        for i in range(n_time):
            flush.fill_(float(i))
            e1.record()
            call()
            e2.record()
            torch.cuda.synchronize()
            ms.append(e1.elapsed_time(e2))
        return statistics.mean(ms)

    # the shipped record and scorer on the same sequences, the reference
    # point of the variants' time per record
    shipped = B.new_summary_store(batch, h_kv, max_pages, dev)
    B.locks_build_summaries(wl.k_cache, pt, seq, pgs, shipped, status=status)
    q0 = wl.queries[0, :batch].contiguous()
    shipped_ms = time_scoring(lambda: B.locks_score_pages(
        q0, shipped, sl, sc, status))
    n_rec = int(seq.numel()) * h_kv
    shipped_ns = shipped_ms * 1e6 / n_rec
    del shipped
    out = []
    for rank in (4, 8, 12, 15):
        for vbits in (2, 4, 8):
            rec = B.new_variant_store(batch, h_kv, max_pages, rank, vbits, dev)
            e0.record()
            B.locks_build_variant(wl.k_cache, pt, seq, pgs, rec, rank, vbits,
                                  status=status)
            e1.record()
            torch.cuda.synchronize()
            build_ms = e0.elapsed_time(e1)
            hit = tot = 0
            cov, err = [], []
            for i in range(n_steps):
                q = wl.queries[i, :batch].contiguous()
                B.locks_exact_page_scores(q, wl.k_cache, pt, sl, ex, status)
                B.locks_score_variant(q, rec, rank, vbits, sl, sc, status)
                B.locks_select_pages(sc, sl, h_q, k, idx, ws)
                kept = (idx[:, :, None, :] == needles[:, :, :, None]).any(-1)
                hit += int((kept & (needles >= 0)).sum())
                tot += int((needles >= 0).sum())
                for b in range(batch):
                    nf = lens[b] // 16
                    mass = torch.softmax(ex[b, :, :, :nf].double(), -1)
                    sel = idx[b][:, None, :].expand(h_kv, G, k)
                    valid = (sel >= 0) & (sel < nf)
                    c = torch.gather(mass, 2, sel.clamp(0, nf - 1).long())
                    cov.append(float((c * valid).sum(-1).mean()))
                    err.append((sc[b, :, :, :nf] - ex[b, :, :, :nf]).abs()
                               .flatten())
            s_ms = time_scoring(lambda: B.locks_score_variant(
                q0, rec, rank, vbits, sl, sc, status))
            assert int(status.item()) == 0 and B.locks_read_status(ws) == 0
            e = torch.cat(err).double()
            rb = B.locks_variant_record_bytes(rank, vbits)
            out.append({
                "rank": rank, "basis_bits": vbits,
                "record_bytes": rb,
                "payload_bytes": 16 * rank * vbits + 16 * rank + 128 +
                                 2 * rank + 34,
                "carrier_retention": round(hit / max(1, tot), 4),
                "coverage_mean": round(statistics.mean(cov), 5),
                "score_error_mean": round(float(e.mean()), 5),
                "score_error_p99": round(float(torch.quantile(
                    e[torch.randperm(e.numel(), device=e.device)[:1 << 20]],
                    0.99)), 5),
                "build_ms": round(build_ms, 3),
                "score_ms": round(s_ms, 4),
                "score_gbs": round(rb * n_rec / (s_ms / 1e3) / 1e9, 1),
                "score_frac_of_copy_peak": round(
                    rb * n_rec / (s_ms / 1e3) / 1e9 / peak_gbs, 3),
                "score_ns_per_record": round(s_ms * 1e6 / n_rec, 4),
                "vs_shipped_time_per_record": round(
                    s_ms * 1e6 / n_rec / shipped_ns, 3),
                "page_heads": n_rec})
            del rec
    return {"sequences": batch, "budget_pages": k, "steps": n_steps,
            "score_timing": f"mean of {n_time} calls, L2 flushed before "
                            "each", "variants": out,
            "shipped_scorer": {
                "score_ms": round(shipped_ms, 4),
                "score_ns_per_record": round(shipped_ns, 4),
                "score_frac_of_copy_peak": round(
                    832 * n_rec / (shipped_ms / 1e3) / 1e9 / peak_gbs, 3)},
            "note": "variant records (fragment-ordered; the (8, 4) record "
                    "is the shipped record byte for byte) scored by the "
                    "variant kernel: the shipped scorer's persistent bulk-"
                    "copy stream and tensor-core products, templated on "
                    "rank and basis width; record_bytes is the stride, "
                    "payload_bytes the codes and scales alone"}


def host_cores():
    return _CORES


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True,
                             timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def blas_threads():
    return int(os.environ.get("OPENBLAS_NUM_THREADS", _CORES))


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_step(O, recs, keys, vals, q, seq_len, k, heads):
    """One oracle decode step of one sequence for the listed KV heads:
    score every summarised page, select, attend.  recs [h][n][832]."""
    import numpy as np
    G = q.shape[0] // keys.shape[1]
    for h in heads:
        mu, V, C = O.dequantize(O.decode_records(recs[h]))
        s_hat = O.score_from_summaries(q[h * G:(h + 1) * G], mu, V, C)
        sel = O.select_one(s_hat, seq_len, k)
        toks_k, toks_v = [], []
        for p in sel:
            nt = min(16, seq_len - 16 * p)
            toks_k.append(keys[p, h, :nt])
            toks_v.append(vals[p, h, :nt])
        O.attend(q[h * G:(h + 1) * G], np.concatenate(toks_k),
                 np.concatenate(toks_v))


def oracle_records(O, keys, seq_len):
    """Oracle summaries [h][n_full][832] of one sequence's full pages."""
    nf = seq_len // 16
    q8, _ = O.build_page(keys[:nf])                    # [n][h][...]
    rec = O.encode_records(q8)                          # [n][h][832]
    return rec.transpose(1, 0, 2).copy()


def cpu_baseline(O, keys, vals, queries, seq_len, k, steps=4):
    """Time `steps` oracle decode steps of one sequence (all KV heads)."""
    import numpy as np
    recs = oracle_records(O, keys, seq_len)
    h_kv = keys.shape[1]
    t0 = time.perf_counter()
    for s in range(steps):
        oracle_step(O, recs, keys, vals, queries[s % len(queries)].astype(
            np.float64), seq_len, k, range(h_kv))
    dt = time.perf_counter() - t0
    return steps / dt, dt


# ---------------------------------------------------------------------------
# the LOCKS arm
# ---------------------------------------------------------------------------
def run_locks(args):
    import numpy as np
    import torch

    from sparse_paged_kv_locks_gb300 import binding as B
    from sparse_paged_kv_locks_gb300 import workload as W

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist_init(world, "nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec = rank_spec(W.SPECS[args.workload], rank, args.batch, args.ctx)
    B.lib()

    wl = W.generate(spec, dev)
    lens = [int(x) for x in wl.seq_lens]
    batch, max_pages = wl.page_table.shape
    h_kv, G, k = spec.h_kv, spec.group, spec.k
    seq = torch.tensor([b for b in range(batch) for _ in range(lens[b] // 16)],
                       dtype=torch.int32, device=dev)
    pgs = torch.tensor([p for b in range(batch) for p in range(lens[b] // 16)],
                       dtype=torch.int32, device=dev)
    n_records = int(seq.numel()) * h_kv
    store = B.new_summary_store(batch, h_kv, max_pages, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(
        enable_timing=True)
    e0.record()
    B.locks_build_summaries(wl.k_cache, wl.page_table, seq, pgs, store,
                            status=status)
    e1.record()
    torch.cuda.synchronize()
    build_ms = e0.elapsed_time(e1)
    if not args.quick:   # rebuild once warm for a steady number
        e0.record()
        B.locks_build_summaries(wl.k_cache, wl.page_table, seq, pgs, store,
                                status=status)
        e1.record()
        torch.cuda.synchronize()
        build_ms = e0.elapsed_time(e1)
    assert int(status.item()) == 0, "build reported a device error"

    ws = B.new_workspace(batch, spec.h_q, h_kv, max_pages, max_pages, dev)
    scores = ws[256:256 + 4 * batch * h_kv * G * max_pages].view(
        torch.float32).view(batch, h_kv, G, max_pages)
    idx = torch.empty(batch, h_kv, k, dtype=torch.int32, device=dev)
    o = torch.empty(batch, spec.h_q, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(batch, spec.h_q, dtype=torch.float32, device=dev)
    qs = wl.queries
    n_q = qs.shape[0]

    # the kernels locks_score_select launches, called one by one so that
    # events can sit between them
    def step(i, evs=None):
        q = qs[i % n_q]
        if evs:
            evs[0].record()
        B.locks_score_pages(q, store, wl.seq_lens, scores, ws[:4].view(
            torch.int32))
        if evs:
            evs[1].record()
        B.locks_select_pages(scores, wl.seq_lens, spec.h_q, k, idx, ws)
        if evs:
            evs[2].record()
        B.locks_sparse_decode(q, wl.k_cache, wl.v_cache, wl.page_table,
                              wl.seq_lens, idx, k, o, lse, ws)
        if evs:
            evs[3].record()

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert B.locks_read_status(ws) == 0, "decode reported a device error"
    # per-kernel events on every sixteenth timed step: an event between two
    # kernels stops the second from launching early (programmatic
    # dependent launch), so the other steps run with none, as a step does
    # in production
    EV_EVERY = 16
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
           if i % EV_EVERY == 0 else None for i in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(
        enable_timing=True)
    launches0 = B.locks_kernel_launches()
    t_start.record()
    for i in range(args.steps):
        step(args.warmup + i, evs[i])
    t_end.record()
    timed_launches = B.locks_kernel_launches() - launches0
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    evs = [e for e in evs if e]
    score_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    select_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    decode_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    job_ms = reduce_max(total_ms)
    value = world * batch * args.steps / (job_ms / 1e3)

    # algorithmic bytes: summaries of every full page + selected K/V (valid
    # tokens) + q + o
    idx_h = idx.cpu().numpy()
    kv_bytes = 0
    for b in range(batch):
        for h in range(h_kv):
            for p in idx_h[b, h]:
                if p >= 0:
                    kv_bytes += min(16, lens[b] - 16 * int(p)) * 2 * 128 * 2
    q_bytes = batch * spec.h_q * 128 * 2
    score_bytes = n_records * RECORD_PAYLOAD
    step_bytes = score_bytes + kv_bytes + 2 * q_bytes
    peak, peak_src = measured_peaks()
    score_gbs = score_bytes / (score_ms / 1e3) / 1e9
    step_gbs = step_bytes / (total_ms / args.steps / 1e3) / 1e9
    decode_gbs = kv_bytes / (decode_ms / 1e3) / 1e9
    traffic, per_kernel = step_traffic(
        {"record": n_records,
         "score_entry": batch * h_kv * G * max_pages,
         "page_head": int((idx_h >= 0).sum())}, G)
    step_ms = total_ms / args.steps
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": job_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "precision": "bf16 K/V and queries, int4/int8 summaries with fp16 "
                     "scales, fp16/bf16 tensor-core operands, fp32 "
                     "accumulation",
        "data": "synthetic (seeded generator, no datasets or weights)",
        "config": {
            "workload": f"{spec.name}: batch {batch} x {spec.ctx} tokens, "
                        f"{spec.h_q} query / {h_kv} KV heads, d=128, page 16, "
                        f"rank 8, budget k={k} pages",
            "batch": batch, "context": spec.ctx, "h_q": spec.h_q,
            "h_kv": h_kv, "k": k,
            "l2": "inputs larger than L2: every step streams "
                  f"{score_bytes / 1e9:.2f} GB of summaries and "
                  f"{kv_bytes / 1e6:.0f} MB of selected K/V",
            "parallelism": f"replicas x{world}"},
        # the step's roofline as the method defines it: bytes of every
        # summary, the selected pages' K/V, q and o over the step time
        "roofline": {
            "bound": "hbm",
            "kernel": "whole step (score + select + sparse decode + merge)",
            "achieved": round(step_gbs, 1), "peak": peak, "unit": "GB/s",
            "frac": round(step_gbs / peak, 4),
            "frac_of_8tbs": round(step_gbs / 8000.0, 4),
            "traffic": traffic,
            "traffic_per_kernel": per_kernel,
            "traffic_source": "small-case ncu captures scaled per unit of "
                              "work (profiles/step_traffic.json)",
            "peak_source": peak_src,
            "algorithmic_bytes": step_bytes,
            "ms_per_step": round(step_ms, 4),
            "dominant_kernel": {
                "kernel": "score (summary stream)",
                "achieved": round(score_gbs, 1),
                "frac": round(score_gbs / peak, 4),
                "algorithmic_bytes": score_bytes,
                "traffic": (per_kernel or {}).get("score")
                if traffic is not None else None,
                "ms": round(score_ms, 4),
                "share_of_step": round(score_ms / step_ms, 4)}},
        "kernels_ms": {"score": round(score_ms, 4),
                       "select": round(select_ms, 4),
                       "sparse_decode": round(decode_ms, 4),
                       "sparse_decode_gbs": round(decode_gbs, 1),
                       "from_steps": f"events on every {EV_EVERY}th timed step"},
        "gpu_launches": None, "clocks": clk,
    }
    # the library's own count of the kernels it launched in the timed region
    line["gpu_launches"] = timed_launches
    line["build"] = {"page_heads": n_records, "ms": round(build_ms, 3),
                     "page_heads_per_s": round(n_records / (build_ms / 1e3)),
                     "roofline": build_issue(n_records, build_ms,
                                             clk.get("sm_mhz") or
                                             clk.get("sm_max_mhz"))}

    if args.quick and args.ablation:
        line["quality"] = {"rank_precision_ablation": rank_precision_ablation(
            B, wl, lens, k, spec.h_q, peak)}
    if not args.quick:
        # e2e: pinned host query in, pinned host (o, lse) out, every step,
        # through the C ABI decoder object: the query copy, the kernels and
        # the result copies replay as one CUDA graph per step
        dec = B.LocksDecoder(wl.k_cache, wl.v_cache, wl.page_table, store,
                             spec.h_q, k, graph=True, seq_lens=wl.seq_lens)
        q_host = qs.cpu().pin_memory()
        o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        lse_host = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        n_e2e = max(10, min(args.steps, 500))
        # the C ABI call with host buffers, as a C caller makes it: each
        # step's query, output and status pointers are plain host pointers
        import ctypes
        step_host = B.lib().locks_decoder_step_host
        handle = dec.handle()
        q_ptrs = [ctypes.c_void_p(q_host[i].data_ptr()) for i in range(n_q)]
        o_ptr = ctypes.c_void_p(o_host.data_ptr())
        l_ptr = ctypes.c_void_p(lse_host.data_ptr())
        dev_status = ctypes.c_int32(0)
        st_ref = ctypes.byref(dev_status)
        s_ptr = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        for i in range(3):
            assert step_host(handle, q_ptrs[i % n_q], o_ptr, l_ptr, st_ref,
                             s_ptr) == 0
        barrier()
        rcs = 0
        t0 = time.perf_counter()
        for i in range(n_e2e):
            rcs |= step_host(handle, q_ptrs[i % n_q], o_ptr, l_ptr, st_ref,
                             s_ptr)
        dt = reduce_max(time.perf_counter() - t0)
        assert rcs == 0 and dev_status.value == 0, "e2e step failed"
        # the same result the eager step gives for the last query
        ref_o, ref_lse = B.LocksDecoder(
            wl.k_cache, wl.v_cache, wl.page_table, store, spec.h_q,
            k).step(qs[(n_e2e - 1) % n_q].contiguous(), wl.seq_lens)
        assert torch.equal(ref_o.cpu(), o_host) and \
            torch.equal(ref_lse.cpu(), lse_host), "e2e result differs"
        line["e2e"] = {"value": world * batch * n_e2e / dt, "unit": "tokens/s",
                       "steps": n_e2e,
                       "h2d_bytes_per_step": q_bytes,
                       "d2h_bytes_per_step": q_bytes + batch * spec.h_q * 4 + 4,
                       "api": "locks_decoder_step_host (C ABI, called "
                              "with the step's host pointers): one CUDA graph "
                              "per step: a kernel reading q from pinned host "
                              "memory, then the 4 step kernels, which write "
                              "o, lse and the status word straight into "
                              "pinned host memory"}
        # dense full-cache decode of the same shape, as context
        for _ in range(2):
            B.locks_sparse_decode(qs[0], wl.k_cache, wl.v_cache,
                                  wl.page_table, wl.seq_lens, None, 0, o, lse,
                                  ws)
        torch.cuda.synchronize()
        n_dense = 10
        t_start.record()
        for i in range(n_dense):
            B.locks_sparse_decode(qs[i % n_q], wl.k_cache, wl.v_cache,
                                  wl.page_table, wl.seq_lens, None, 0, o, lse,
                                  ws)
        t_end.record()
        torch.cuda.synchronize()
        dms = t_start.elapsed_time(t_end) / n_dense
        dense_bytes = sum(lens) * h_kv * 2 * 128 * 2
        line["dense_context"] = {
            "value": batch / (dms / 1e3), "unit": "tokens/s",
            "ms_per_step": round(dms, 4),
            "gbs": round(dense_bytes / (dms / 1e3) / 1e9, 1)}
        line["small_configs"] = small_configs(B, W, dev)
        line["append_config"] = append_config(
            B, W, dev, clk.get("sm_mhz") or clk.get("sm_max_mhz"))
        line["ragged_config"] = ragged_config(B, W, dev, peak)
        line["quality"] = selection_quality(B, wl, store, scores, ws, lens,
                                            k, spec.h_q, n_records)
        line["quality"]["rank_precision_ablation"] = rank_precision_ablation(
            B, wl, lens, k, spec.h_q, peak)
        if rank == 0 and world == 1:
            from oracle import locks_oracle as O
            b0 = 0
            n0 = math.ceil(lens[b0] / 16)
            phys = wl.page_table[b0, :n0].long()
            keys = wl.k_cache[phys].float().cpu().numpy()
            vals = wl.v_cache[phys].float().cpu().numpy()
            qn = qs[:, b0].float().cpu().numpy()
            steps_cpu = 4
            v_cpu, dt_cpu = cpu_baseline(O, keys, vals, qn, lens[b0], k,
                                         steps_cpu)
            line["cpu_baseline"] = {
                "value": v_cpu, "unit": "tokens/s", "cores": host_cores(),
                "kind": "oracle", "cpu_model": cpu_model(),
                "blas_threads": blas_threads(),
                "sample": f"sequence 0 of {batch} ({lens[b0]} tokens), all "
                          f"{h_kv} KV heads, {steps_cpu} decode steps (score "
                          "+ select + sparse attention) in "
                          f"{dt_cpu:.1f} s; oracle summaries built outside "
                          "the timed region; extrapolated to the batch as "
                          "tokens/s"}
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the reference arm: the float64 oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    import numpy as np

    from oracle import locks_oracle as O
    from sparse_paged_kv_locks_gb300 import workload as W

    rank, world, _ = dist_env()
    if rank != 0:
        return
    spec = rank_spec(W.SPECS[args.workload], 0, args.batch, args.ctx)
    one = W.generate_sequence(spec, 0, "cpu", steps=min(spec.steps, 8))
    keys = one["keys"].float().numpy()
    vals = one["values"].float().numpy()
    qs = one["queries"].float().numpy().astype(np.float64)
    L = one["seq_len"]
    h_kv, k = spec.h_kv, spec.k
    n_full = L // 16
    # per-step sample: one KV head (rotating) over the first P pages, P sized
    # so warm-up + timed steps take about two minutes
    recs = oracle_records(O, keys, L)
    t0 = time.perf_counter()
    oracle_step(O, recs, keys, vals, qs[0], L, k, [0])
    t_head = time.perf_counter() - t0
    budget = 120.0 / max(1, args.steps + args.warmup)
    P = int(min(n_full, max(4 * k, n_full * budget / max(t_head, 1e-6))))
    P = min(P, n_full)
    Ls = 16 * P
    sub = recs[:, :P]

    def one_step(i):
        h = i % h_kv
        oracle_step(O, sub, keys[:P], vals[:P], qs[i % len(qs)], Ls, k, [h])

    for i in range(args.warmup):
        one_step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one_step(args.warmup + i)
    dt = time.perf_counter() - t0
    frac = P / math.ceil(L / 16) / h_kv        # of one token's decode step
    value = frac * args.steps / dt
    sample = (f"per step: sequence 0 ({L} tokens), one KV head of {h_kv} "
              f"(rotating), first {P} of {math.ceil(L / 16)} pages with the "
              f"budget k={k}; counted as {frac:.4f} of a token")
    line = {"impl": "reference", "metric": METRIC, "value": value,
            "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded generator)",
            "config": {"workload": f"{spec.name}: batch {spec.batch} x "
                                   f"{spec.ctx} tokens, {spec.h_q} query / "
                                   f"{h_kv} KV heads, d=128, page 16, rank 8, "
                                   f"budget k={k} pages",
                       "batch": spec.batch, "context": spec.ctx},
            "cpu_baseline": {"value": value, "unit": "tokens/s",
                             "cores": host_cores(), "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "blas_threads": blas_threads(),
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_locks(args)


if __name__ == "__main__":
    main()
