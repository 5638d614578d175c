"""Benchmark of the DSA indexer + top-k + IndexShare sparse-attention path on GB300.

One step = the whole hot path over the L = 131072 prefill workload: 16 layers in
4 IndexShare groups; per group one indexer + top-k call (the Full layer) and
sparse attention for its 4 layers over the shared index rows.  Inputs are
synthetic (seeded Gaussians, distinct per layer) and resident in HBM before the
timed region; they are larger than L2, so L2 is not flushed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--config C]

Prints one JSON line (rank 0).  With --impl reference the CPU oracle is timed on
the host cores on a bounded row sample of the same workload.
"""
import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "indexer+top-k query rows/s and group prefill tok/s @L=128K; % TC peak / HBM BW"
UNIT = "tok/s"
FP8_PER_BF16 = 2.0  # nominal dense FP8 : BF16 tensor ratio (4.5 : 2.25 PFLOP/s)
NOMINAL_TFLOPS = {"e4m3": 4500.0, "bf16": 2250.0}  # datasheet dense peaks, context only


# ----------------------------------------------------------------------------- helpers

def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def _code_only(text):
    """Source text without comments and blank lines (a comment edit keeps the key)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def _kernel_sources_sha(names):
    h = hashlib.sha256()
    for n in names:
        p = os.path.join(ROOT, "top_selection_indexer_gb300", "csrc", n)
        if os.path.exists(p):
            h.update(_code_only(open(p, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def _profiled_traffic(kernel, src_files, workload):
    """DRAM bytes per launch from profiles/traffic.txt, if taken on the current source for
    this workload (None otherwise)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if workload is None or not os.path.exists(path):
        return None
    sha = _kernel_sources_sha(src_files)
    for line in open(path):
        kv = dict(x.split("=", 1) for x in line.split() if "=" in x)
        if kv.get("kernel") == kernel and kv.get("src_sha") == sha and \
                kv.get("workload") == workload:
            return float(kv["bytes_per_launch"])
    return None


def _kernel_files(kernel):
    """Source files that define a kernel's device code (its traffic is keyed to them)."""
    return {
        "tsi_attn_tc_kernel": ["attn_tc.cu", "latent_gather.cuh", "tc_common.cuh"],
        "attn_generic_kernel": ["attn_generic.cu"],
        # the default call: sample gather, threshold and full scoring passes, short units,
        # then the ranking kernel (indexer_generic.cu)
        "tsi_indexer_tc_kernel": ["indexer_tc.cu", "indexer_generic.cu", "topk_select.cuh",
                                  "rank_sort.cuh", "tc_common.cuh", "kernels_tc.cuh"],
        "indexer_generic_kernel": ["indexer_generic.cu", "topk_select.cuh"],
        "tsi_index_kl_tc_kernel": ["index_kl_tc.cu", "latent_gather.cuh", "tc_common.cuh"],
    }[kernel]


def _traffic_workload(cfg, what):
    """Name of a captured workload in profiles/traffic.txt: whole prefills of one sequence."""
    if cfg.B != 1 or cfg.T != cfg.S:
        return None
    return f"prefill_L{cfg.S}_{what}"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU arm

def run_gpu(args, rank, world):
    import torch
    import torch.distributed as dist

    import top_selection_indexer_gb300 as tsi
    from top_selection_indexer_gb300 import accounting
    from workloads import get_config, make_attn_inputs, make_indexer_inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    tsi.load()
    cfg = get_config(args.config)
    if args.groups:
        cfg = cfg.with_(n_layers=min(cfg.n_layers, args.groups * cfg.group))
    if args.tail_rows:  # chunked prefill: only the last R query rows over the full cache
        cfg = cfg.with_(T=min(args.tail_rows, cfg.S))
    G, L = cfg.n_groups, cfg.S
    stream = torch.cuda.current_stream()

    # --- resident inputs (every layer distinct) --------------------------------------
    t0 = time.time()
    ind = [make_indexer_inputs(cfg, g, dev) for g in range(G)]
    lay = [make_attn_inputs(cfg, l, dev) for l in range(cfg.n_layers)]
    idx = torch.empty((cfg.B, cfg.T, cfg.topk), dtype=torch.int32, device=dev)
    outs = [torch.empty((cfg.B, cfg.T, cfg.H, cfg.Dv), dtype=torch.bfloat16, device=dev)
            for _ in range(cfg.group)]
    ws_i = tsi.indexer_topk_workspace(cfg.B, cfg.T, cfg.S, cfg.H_I, cfg.d_I, cfg.topk,
                                      tsi.E4M3 if cfg.qk_dtype == "e4m3" else tsi.BF16)
    ws_a = tsi.sparse_attn_workspace(cfg.B, cfg.T, cfg.S, cfg.H, cfg.Hkv, cfg.Dqk, cfg.Dv,
                                     cfg.topk)
    ws = torch.empty(max(ws_i, ws_a, 16), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    setup_s = time.time() - t0

    ev = {"idx": [], "attn": []}

    def step(record):
        for g in range(G):
            qI, kI, w = ind[g]
            if record:
                a = torch.cuda.Event(enable_timing=True)
                a.record(stream)
            tsi.indexer_topk(qI, kI, w, cfg.topk, idx=idx, workspace=ws, stream=stream)
            if record:
                b = torch.cuda.Event(enable_timing=True)
                b.record(stream)
                ev["idx"].append((a, b))
            for l0 in range(min(cfg.group, cfg.n_layers - g * cfg.group)):
                Q, K, V = lay[g * cfg.group + l0]
                if record:
                    a = torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                tsi.sparse_attn_group([Q], [K], None if V is None else [V], idx, cfg.scale,
                                      outs=[outs[l0]], workspace=ws, stream=stream, Dv=cfg.Dv)
                if record:
                    b = torch.cuda.Event(enable_timing=True)
                    b.record(stream)
                    ev["attn"].append((a, b))

    for _ in range(args.warmup):
        step(False)
    tsi.device_status(stream)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = tsi.launch_count()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clocks:
        t_start.record(stream)
        for _ in range(args.steps):
            step(True)
        t_end.record(stream)
        torch.cuda.synchronize()
    launches = tsi.launch_count() - launches0
    tsi.device_status(stream)
    ms_total = t_start.elapsed_time(t_end)
    if world > 1:
        tt = torch.tensor([ms_total], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms_total = float(tt.item())
        dist.barrier()
    ms_step = ms_total / args.steps
    ms_idx = statistics.mean(a.elapsed_time(b) for a, b in ev["idx"])
    ms_attn = statistics.mean(a.elapsed_time(b) for a, b in ev["attn"]) if ev["attn"] else 0.0

    # --- rates and roofline ------------------------------------------------------------
    rows = cfg.B * cfg.T
    pairs = accounting.causal_pairs(cfg.B, cfg.T, cfg.S)
    valid_k = accounting.selected_pairs(cfg.B, cfg.T, cfg.S, cfg.topk)
    tok_per_group = cfg.B * cfg.T
    value = world * G * tok_per_group / (ms_step / 1e3)  # group prefill tok/s, all ranks
    peaks = _peaks()
    qk_bytes = 1 if cfg.qk_dtype == "e4m3" else 2
    idx_flops = accounting.indexer_flops(pairs, cfg.H_I, cfg.d_I)
    tc_peak = peaks["bf16_tflops_sustained"] * (FP8_PER_BF16 if cfg.qk_dtype == "e4m3" else 1.0)
    idx_achieved = idx_flops / (ms_idx / 1e3) / 1e12
    attn_bytes = accounting.attn_bytes(valid_k, rows, cfg.H, cfg.Hkv, cfg.Dqk, cfg.Dv,
                                       cfg.topk, cfg.v_from_k)
    attn_achieved = attn_bytes / (ms_attn / 1e3) / 1e9 if ms_attn else 0.0
    attn_tc = accounting.attn_flops(valid_k, cfg.H, cfg.Dqk, cfg.Dv) / (ms_attn / 1e3) / 1e12 \
        if ms_attn else 0.0
    qk_code = tsi.E4M3 if cfg.qk_dtype == "e4m3" else tsi.BF16 if cfg.qk_dtype == "bf16" else tsi.F32
    attn_kernel = "tsi_attn_tc_kernel" if tsi.attn_path(cfg.H, cfg.Hkv, cfg.Dqk, cfg.Dv,
                                                        cfg.v_from_k) == 1 else "attn_generic_kernel"
    idx_kernel = "tsi_indexer_tc_kernel" if tsi.indexer_path(qk_code, cfg.H_I, cfg.d_I) == 1 \
        else "indexer_generic_kernel"
    roof_attn = {"kernel": attn_kernel, "bound": "hbm", "achieved": round(attn_achieved, 1),
                 "peak": peaks["hbm_gbs"], "unit": "GB/s",
                 "frac": round(attn_achieved / peaks["hbm_gbs"], 4),
                 "traffic": _profiled_traffic(attn_kernel, _kernel_files(attn_kernel),
                                              _traffic_workload(cfg, "layer")),
                 "algorithmic_bytes_per_launch": attn_bytes, "ms_per_launch": round(ms_attn, 4),
                 "tc_tflops": round(attn_tc, 1),
                 "peak_source": f"{peaks['source']} hbm_gbs"}
    roof_idx = {"kernel": idx_kernel, "bound": "tensor", "achieved": round(idx_achieved, 1),
                "peak": round(tc_peak, 1), "unit": "TFLOP/s",
                "frac": round(idx_achieved / tc_peak, 4),
                "traffic": _profiled_traffic(idx_kernel, _kernel_files(idx_kernel),
                                             _traffic_workload(cfg, "group")),
                "algorithmic_flops_per_launch": idx_flops, "ms_per_launch": round(ms_idx, 4),
                "peak_source": f"{peaks['source']} bf16 sustained x {FP8_PER_BF16:g} (fp8)"
                               if cfg.qk_dtype == "e4m3" else f"{peaks['source']} bf16 sustained",
                "frac_of_burst": round(idx_achieved / (peaks["bf16_tflops"] * (
                    FP8_PER_BF16 if cfg.qk_dtype == "e4m3" else 1.0)), 4),
                "frac_of_nominal": round(idx_achieved / NOMINAL_TFLOPS.get(cfg.qk_dtype, 1e30), 4),
                "scores_to_hbm": False}
    if cfg.T == 1:
        # decode: one query per sequence scans its whole key cache once -- HBM-bound
        idx_bytes = accounting.indexer_bytes(rows, cfg.B * cfg.S, cfg.H_I, cfg.d_I, qk_bytes,
                                             2 if cfg.w_dtype == "bf16" else 4, cfg.topk)
        idx_gbs = idx_bytes / (ms_idx / 1e3) / 1e9
        roof_idx = {"kernel": idx_kernel, "bound": "hbm", "achieved": round(idx_gbs, 1),
                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(idx_gbs / peaks["hbm_gbs"], 4), "traffic": None,
                    "algorithmic_bytes_per_launch": idx_bytes, "ms_per_launch": round(ms_idx, 4),
                    "tc_tflops": round(idx_flops / (ms_idx / 1e3) / 1e12, 2),
                    "peak_source": f"{peaks['source']} hbm_gbs"}
    dominant = roof_attn if ms_attn * cfg.n_layers >= ms_idx * G else roof_idx

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"{cfg.qk_dtype}+bf16", "data": "synthetic",
        "config": {"workload": f"{_phase(cfg)}, {cfg.n_layers} layers = {G} IndexShare groups "
                               f"(1 Full + {cfg.group - 1} Shared), indexer H_I={cfg.H_I} "
                               f"d_I={cfg.d_I} {cfg.qk_dtype}, k={cfg.topk}, MQA {cfg.H} heads "
                               f"over a {cfg.Dqk}-d bf16 latent (value = first {cfg.Dv})",
                   "config_id": cfg.id, "L": L, "query_rows": cfg.B * cfg.T,
                   "layers": cfg.n_layers, "topk": cfg.topk,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (not flushed)"},
        "indexer_topk_rows_per_s": round(world * rows / (ms_idx / 1e3), 1),
        "tok_s_all_layers": round(world * tok_per_group / (ms_step / 1e3), 2),
        "stage_ms": {"indexer_topk": round(ms_idx, 4), "sparse_attn_layer": round(ms_attn, 4)},
        "roofline": dominant,
        "roofline_indexer": roof_idx,
        "roofline_attention": roof_attn,
        "gpu_launches": int(launches),
        "setup_s": round(setup_s, 1),
    }
    result["clocks"] = clocks.summary()
    if cfg.T == 1:
        # MTP draft steps of a decode (index_share_for_mtp_iteration): the first step runs
        # the indexer, the later ones reuse its rows; from the measured stage times
        n = 4
        result["mtp"] = {"draft_steps": n, "ms_first_step": round(ms_idx + ms_attn, 4),
                         "ms_later_step": round(ms_attn, 4),
                         "ms_draft_reusing_indices": round(ms_idx + n * ms_attn, 4),
                         "ms_draft_recomputing_indices": round(n * (ms_idx + ms_attn), 4)}
    if cfg.T == 1:
        result["decode_graph"] = measure_decode_graph(cfg, ind, lay, idx, outs, ws)
    elif cfg.id == 4 and not args.no_decode and not args.tail_rows and not args.groups:
        result["decode"] = measure_decode(dev)
    if G >= 2 and not args.no_overlap:
        result["overlap"] = measure_overlap(cfg, ind, idx, ws, stream)
    if not args.no_cp:
        result["context_parallel"] = measure_cp(cfg, ind, idx, stream)
    if cfg.T > 1 and tsi.indexer_path(qk_code, cfg.H_I, cfg.d_I) == 1 and not args.no_two_pass:
        result["indexer_two_pass"] = measure_two_pass(cfg, ind, idx, stream, idx_flops, tc_peak,
                                                      ms_idx, qk_code)
    if not args.no_kl and cfg.n_layers >= 1 and \
            tsi.attn_path(cfg.H, cfg.Hkv, cfg.Dqk, cfg.Dv, cfg.v_from_k) == 1:
        result["index_kl"] = measure_index_kl(cfg, ind, lay, idx, outs, ws, stream)

    # --- end to end through the C ABI with host buffers ---------------------------------
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, cfg, ind, lay, idx, outs, ws, stream, world,
                                n_copy_streams=args.copy_streams)
    return result


def _phase(cfg):
    """Name of the workload's phase: a whole prefill, the last rows of one, or a decode."""
    if cfg.T == cfg.S:
        return f"prefill L={cfg.S}"
    if cfg.T == 1:
        return f"decode B={cfg.B} over L={cfg.S}"
    return f"chunked prefill: last {cfg.T} rows of L={cfg.S}"


def _balanced_edges(cfg, shards, align=128):
    """Key-shard edges that give every shard the same number of causal pairs (a prefill's
    early keys are seen by more rows than its late keys), rounded to `align` keys."""
    import numpy as np

    p = np.arange(cfg.T, dtype=np.int64) + (cfg.S - cfg.T)  # row positions, kv_len = S

    def pairs_below(e):
        return int(np.minimum(p + 1, e).clip(min=0).sum())

    total = pairs_below(cfg.S)
    edges = [0]
    for i in range(1, shards):
        lo, hi = edges[-1], cfg.S
        while lo < hi:  # smallest e with pairs_below(e) >= i / shards of the total
            mid = (lo + hi) // 2
            if pairs_below(mid) * shards >= i * total:
                hi = mid
            else:
                lo = mid + 1
        edges.append(min(cfg.S, max(edges[-1], (lo + align // 2) // align * align)))
    edges.append(cfg.S)
    return edges


def measure_two_pass(cfg, ind, idx, stream, flops, peak, ms_default, qk_code, reps=2):
    """Group 0's indexer + top-k through the two-pass alternative (tsi_indexer_topk_two_pass:
    every score stored to HBM, then selected by a second kernel) beside the default, which
    keeps every score on chip: time per call, the fraction of the tensor peak, and whether
    the rows equal the default's."""
    import torch

    import top_selection_indexer_gb300 as tsi

    qI, kI, w = ind[0]
    out = torch.empty_like(idx)
    ws = torch.empty(max(1, tsi.indexer_topk_workspace(cfg.B, cfg.T, cfg.S, cfg.H_I, cfg.d_I,
                                                       cfg.topk, qk_code, two_pass=True)),
                     dtype=torch.uint8, device=idx.device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for r in range(reps + 1):  # the first call warms up
        if r:
            ev[r - 1][0].record(stream)
        tsi.indexer_topk(qI, kI, w, cfg.topk, idx=out, workspace=ws, stream=stream,
                         two_pass=True)
        if r:
            ev[r - 1][1].record(stream)
    tsi.device_status(stream)
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    del ws
    tsi.indexer_topk(qI, kI, w, cfg.topk, idx=idx, stream=stream)
    same = bool(torch.equal(out, idx))
    tf = flops / (ms / 1e3) / 1e12
    return {"ms_per_call": round(ms, 3), "achieved_tflops": round(tf, 1),
            "frac": round(tf / peak, 4), "ms_default_onchip": round(ms_default, 3),
            "equals_default": same,
            "workspace_bytes": int(tsi.indexer_topk_workspace(cfg.B, cfg.T, cfg.S, cfg.H_I,
                                                              cfg.d_I, cfg.topk, qk_code,
                                                              two_pass=True)),
            "note": "scores stored to HBM by the scoring kernel, then selected by a second "
                    "kernel; the default keeps them on chip (selection in the scoring "
                    "kernel's epilogue from a sampled threshold)"}


def measure_cp(cfg, ind, idx, stream, shards=2, reps=3):
    """Context-parallel indexer of group 0 with its keys in `shards` shards of equal causal
    work, run one after another on this GPU (each standing in for a rank): per-shard kernel
    time, the merge of the gathered lists, and whether the result equals the unsharded rows."""
    import torch

    import top_selection_indexer_gb300 as tsi

    qI, kI, w = ind[0]
    S = cfg.S
    edges = _balanced_edges(cfg, shards)
    kparts = [kI[:, lo:hi].contiguous() for lo, hi in zip(edges[:-1], edges[1:])]
    rows = cfg.B * cfg.T
    cand = torch.empty((shards, rows, cfg.topk), dtype=torch.int64, device=idx.device)
    cnt = torch.empty((shards, rows), dtype=torch.int32, device=idx.device)
    out = torch.empty((rows, cfg.topk), dtype=torch.int32, device=idx.device)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(shards + 2)] for _ in range(reps)]
    for r in range(reps + 1):  # the first pass warms up
        rec = ev[r - 1] if r else None
        for i, (lo, kp) in enumerate(zip(edges[:-1], kparts)):
            if rec:
                rec[i].record(stream)
            tsi.indexer_topk_shard(qI, kp, w, cfg.topk, S, lo, cand=cand[i], cand_cnt=cnt[i],
                                   stream=stream)
        if rec:
            rec[shards].record(stream)
        tsi.topk_merge(cand, cnt, idx=out, stream=stream)
        if rec:
            rec[shards + 1].record(stream)
    tsi.device_status(stream)
    shard_ms = [statistics.mean(e[i].elapsed_time(e[i + 1]) for e in ev) for i in range(shards)]
    merge_ms = statistics.mean(e[shards].elapsed_time(e[shards + 1]) for e in ev)
    tsi.indexer_topk(qI, kI, w, cfg.topk, idx=idx, stream=stream)
    same = bool(torch.equal(out, idx.view(rows, cfg.topk)))
    return {"shards": shards, "key_edges": edges, "ms_per_shard": [round(x, 3) for x in shard_ms],
            "ms_merge": round(merge_ms, 3), "equals_unsharded": same,
            "note": "shards run one after another on this GPU, each standing in for a rank; "
                    "the exchange between ranks (all-gather of the lists) is not timed"}


def measure_overlap(cfg, ind, idx, ws, stream, reps=5):
    """Cross-layer top-k overlap of the Full layers of groups 0 and 1 (tsi_topk_overlap),
    outside the timed step: its kernel time and the mean overlap rate of the rows."""
    import torch

    import top_selection_indexer_gb300 as tsi

    idx_b = torch.empty_like(idx)
    for g, out in ((0, idx), (1, idx_b)):
        qI, kI, w = ind[g]
        tsi.indexer_topk(qI, kI, w, cfg.topk, idx=out, workspace=ws, stream=stream)
    rows = cfg.B * cfg.T
    inter = torch.empty(rows, dtype=torch.int32, device=idx.device)
    card = torch.empty_like(inter)
    tsi.topk_overlap(idx, idx_b, inter, card, stream=stream)  # warm-up
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        tsi.topk_overlap(idx, idx_b, inter, card, stream=stream)
    b.record(stream)
    tsi.device_status(stream)
    ms = a.elapsed_time(b) / reps
    nbytes = 2 * rows * cfg.topk * 4 + 2 * rows * 4  # both index buffers in, counts out
    rate = (inter.double() / card.clamp(min=1).double())[card > 0].mean().item()
    return {"layers": "Full layers of groups 0 and 1", "rows": rows, "ms_per_launch": round(ms, 4),
            "achieved_gbs": round(nbytes / (ms / 1e3) / 1e9, 1),
            "algorithmic_bytes_per_launch": nbytes, "mean_overlap_rate": round(rate, 5)}


def measure_decode_graph(cfg, ind, lay, idx, outs, ws, reps=20, flush=None):
    """Latency of one IndexShare group of a decode step (the Full layer's indexer + top-k,
    then the group's sparse attention layers) replayed from a CUDA graph, against the same
    calls launched one by one.  With ``flush`` (a device buffer larger than L2) the buffer is
    overwritten before every timed repetition, so no repetition finds the previous one's
    keys in L2."""
    import torch

    import top_selection_indexer_gb300 as tsi

    qI, kI, w = ind[0]
    layers = lay[:cfg.group]
    qs = [Q for Q, _, _ in layers]
    ks = [K for _, K, _ in layers]

    def group_step(stream):
        tsi.indexer_topk(qI, kI, w, cfg.topk, idx=idx, workspace=ws, stream=stream)
        tsi.sparse_attn_group(qs, ks, None, idx, cfg.scale, outs=outs[:len(layers)],
                              workspace=ws, stream=stream, Dv=cfg.Dv)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    n0 = tsi.launch_count()
    with torch.cuda.stream(side):
        for _ in range(3):
            group_step(side)
    launches = (tsi.launch_count() - n0) // 3
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        group_step(side)
    torch.cuda.synchronize()

    def timed(fn):
        with torch.cuda.stream(side):
            for _ in range(3):
                fn()
            if flush is None:
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(side)
                for _ in range(reps):
                    fn()
                b.record(side)
                b.synchronize()
                return a.elapsed_time(b) / reps * 1e3
            evs = []
            for _ in range(reps):
                flush.add_(1)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(side)
                fn()
                b.record(side)
                evs.append((a, b))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3

    us_graph = timed(graph.replay)
    us_eager = timed(lambda: group_step(side))
    tsi.device_status(side)
    return {"what": f"one group of a decode step: indexer + top-k of the Full layer, then "
                    f"{len(layers)} sparse-attention layers (B={cfg.B}, one query each)",
            "kernel_launches": int(launches), "us_graph_replay": round(us_graph, 2),
            "us_eager": round(us_eager, 2), "reps": reps,
            "l2": "flushed before every repetition" if flush is not None else "not flushed"}


def measure_decode(dev, reps=30):
    """The decode workload (B = 8 sequences, one new query each over a 131072-token cache,
    one IndexShare group of 4 layers), timed after the prefill step: the indexer + top-k
    and each attention layer with CUDA events (median over repetitions, L2 flushed before
    each), the group replayed from a CUDA graph, and their HBM fractions in algorithmic
    bytes.  Its tensors are freed afterwards."""
    import torch

    import top_selection_indexer_gb300 as tsi
    from top_selection_indexer_gb300 import accounting
    from workloads import get_config, make_attn_inputs, make_indexer_inputs

    cfg = get_config(5)
    stream = torch.cuda.current_stream()
    ind = [make_indexer_inputs(cfg, 0, dev)]
    lay = [make_attn_inputs(cfg, l, dev) for l in range(cfg.group)]
    idx = torch.empty((cfg.B, cfg.T, cfg.topk), dtype=torch.int32, device=dev)
    outs = [torch.empty((cfg.B, cfg.T, cfg.H, cfg.Dv), dtype=torch.bfloat16, device=dev)
            for _ in range(cfg.group)]
    code = tsi.E4M3
    ws = torch.empty(max(16, tsi.indexer_topk_workspace(cfg.B, cfg.T, cfg.S, cfg.H_I, cfg.d_I,
                                                        cfg.topk, code),
                         tsi.sparse_attn_workspace(cfg.B, cfg.T, cfg.S, cfg.H, cfg.Hkv,
                                                   cfg.Dqk, cfg.Dv, cfg.topk)),
                     dtype=torch.uint8, device=dev)
    flush = torch.zeros(64 << 20, dtype=torch.float32, device=dev)  # 256 MB > L2
    qI, kI, w = ind[0]

    def stage(fn):
        for _ in range(3):
            fn()
        evs = []
        for _ in range(reps):
            flush.add_(1)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3

    us_idx = stage(lambda: tsi.indexer_topk(qI, kI, w, cfg.topk, idx=idx, workspace=ws,
                                            stream=stream))
    us_attn = [stage(lambda l=l: tsi.sparse_attn_group(
        [lay[l][0]], [lay[l][1]], None, idx, cfg.scale, outs=[outs[l]], workspace=ws,
        stream=stream, Dv=cfg.Dv)) for l in range(cfg.group)]
    tsi.device_status(stream)
    graph = measure_decode_graph(cfg, ind, lay, idx, outs, ws, reps=reps, flush=flush)
    peaks = _peaks()
    rows = cfg.B * cfg.T
    idx_bytes = accounting.indexer_bytes(rows, cfg.B * cfg.S, cfg.H_I, cfg.d_I, 1, 2, cfg.topk)
    valid_k = accounting.selected_pairs(cfg.B, cfg.T, cfg.S, cfg.topk)
    attn_bytes = accounting.attn_bytes(valid_k, rows, cfg.H, cfg.Hkv, cfg.Dqk, cfg.Dv, cfg.topk,
                                       cfg.v_from_k)
    us_attn_mean = statistics.mean(us_attn)
    res = {"workload": f"decode B={cfg.B} over L={cfg.S}: indexer H_I={cfg.H_I} d_I={cfg.d_I} "
                       f"e4m3, k={cfg.topk}, {cfg.group} layers of MQA {cfg.H} heads over a "
                       f"{cfg.Dqk}-d bf16 latent cache",
           "us_indexer_topk": round(us_idx, 2),
           "us_attn_per_layer": round(us_attn_mean, 2),
           "us_group_graph": graph["us_graph_replay"], "us_group_eager": graph["us_eager"],
           "kernel_launches_per_group": graph["kernel_launches"],
           "tok_s": round(rows / (graph["us_graph_replay"] / 1e6), 1),
           "indexer_hbm": {"algorithmic_bytes": idx_bytes,
                           "achieved_gbs": round(idx_bytes / (us_idx / 1e6) / 1e9, 1),
                           "frac": round(idx_bytes / (us_idx / 1e6) / 1e9 / peaks["hbm_gbs"], 4)},
           "attn_hbm": {"algorithmic_bytes": attn_bytes,
                        "achieved_gbs": round(attn_bytes / (us_attn_mean / 1e6) / 1e9, 1),
                        "frac": round(attn_bytes / (us_attn_mean / 1e6) / 1e9 / peaks["hbm_gbs"],
                                      4)},
           "peak_source": f"{peaks['source']} hbm_gbs",
           "l2": "a 256 MB buffer is overwritten before every timed repetition"}
    del ind, lay, idx, outs, ws, flush
    torch.cuda.empty_cache()
    return res


def measure_index_kl(cfg, ind, lay, idx, outs, ws, stream, reps=2):
    """Group-centroid KL target of group 0's Full-layer indexer over every query row: the
    indexer's scores and each layer's attention with its log-partition are computed first
    (untimed), then tsi_index_kl (loss and gradient) is timed on its own."""
    import torch

    import top_selection_indexer_gb300 as tsi
    from top_selection_indexer_gb300 import accounting

    qI, kI, w = ind[0]
    dev = idx.device
    score = torch.empty(idx.shape, dtype=torch.float32, device=dev)
    tsi.indexer_topk(qI, kI, w, cfg.topk, idx=idx, score=score, workspace=ws, stream=stream)
    layers = lay[:cfg.group]
    qs = [Q for Q, _, _ in layers]
    ks = [K for _, K, _ in layers]
    lses = [torch.empty((cfg.B, cfg.T, cfg.H), dtype=torch.float32, device=dev)
            for _ in layers]
    tsi.sparse_attn_group(qs, ks, None, idx, cfg.scale, outs=outs[:len(layers)], workspace=ws,
                          stream=stream, Dv=cfg.Dv, lses=lses)
    loss = torch.empty((cfg.B, cfg.T), dtype=torch.float32, device=dev)
    grad = torch.empty(idx.shape, dtype=torch.float32, device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for r in range(reps + 1):  # the first call warms up
        if r:
            ev[r - 1][0].record(stream)
        tsi.index_kl(qs, ks, lses, idx, score, cfg.scale, loss=loss, grad=grad, stream=stream)
        if r:
            ev[r - 1][1].record(stream)
    tsi.device_status(stream)
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    rows = cfg.B * cfg.T
    valid_k = accounting.selected_pairs(cfg.B, cfg.T, cfg.S, cfg.topk)
    nbytes = accounting.index_kl_bytes(valid_k, rows, len(layers), cfg.H, cfg.Dqk, cfg.topk)
    flops = accounting.index_kl_flops(valid_k, len(layers), cfg.H, cfg.Dqk)
    peaks = _peaks()
    achieved = nbytes / (ms / 1e3) / 1e9
    kernel = "tsi_index_kl_tc_kernel"
    return {"layers": f"group 0: 1 Full + {len(layers) - 1} Shared", "rows": rows,
            "outputs": "loss and gradient per row", "ms_per_launch": round(ms, 3),
            "rows_per_s": round(rows / (ms / 1e3), 1),
            "mean_loss": round(float(loss.double().mean().item()), 6),
            "roofline": {"kernel": kernel, "bound": "hbm", "achieved": round(achieved, 1),
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "traffic": _profiled_traffic(kernel, _kernel_files(kernel),
                                                      _traffic_workload(cfg, "group_kl")),
                         "algorithmic_bytes_per_launch": nbytes,
                         "tc_tflops": round(flops / (ms / 1e3) / 1e12, 1),
                         "peak_source": f"{peaks['source']} hbm_gbs"}}


def run_e2e(args, cfg, ind, lay, idx, outs, ws, stream, world, n_copy_streams=4):
    """Same step with inputs copied host->device and results device->host inside the
    timed region (pinned host buffers; every tensor moves as n_copy_streams contiguous
    pieces, one cudaMemcpyAsync each, on as many streams, so several copy engines share
    the transfer).

    Copies overlap the kernels, as a pipelined caller would run them: the upload streams
    move each layer's Q and latent (and each group's indexer inputs) into that layer's
    own device buffers ahead of the compute stream; the read-back streams copy each
    layer's output (and each group's index rows) to the host behind it -- with
    --readback result (the default) only the step's result, the stack's last output, as
    a caller that keeps the intermediate layers on the device would.  Events order
    every reuse of a buffer: an upload waits until the previous step's kernels are done
    with its destination, a kernel waits for its inputs and for the read-back of the
    output buffer it overwrites, and the timer stops after the last read-back.
    """
    import torch

    import top_selection_indexer_gb300 as tsi

    G, nl = cfg.n_groups, cfg.n_layers
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)  # noqa: E731
    h_ind = tuple(pin(x) for x in ind[0])
    for hx, dx in zip(h_ind, ind[0]):
        hx.copy_(dx)
    h_Q = h_K = h_V = h_O = None
    if nl:  # one pinned host copy of a layer's Q and latent serves every layer's upload
        Q0, K0, V0 = lay[0]
        h_Q, h_K = pin(Q0), pin(K0)
        h_Q.copy_(Q0)
        h_K.copy_(K0)
        h_V = None if V0 is None else pin(V0)
        if h_V is not None:
            h_V.copy_(V0)
        h_O = pin(outs[0])
    h_idx = pin(idx)
    idx_bufs = [idx, torch.empty_like(idx)]
    ups = [torch.cuda.Stream(device=idx.device) for _ in range(n_copy_streams)]
    downs = [torch.cuda.Stream(device=idx.device) for _ in range(n_copy_streams)]
    ev = lambda: torch.cuda.Event()  # noqa: E731
    h2d = d2h = 0
    steps = max(5, min(args.steps, 8))
    decode = cfg.T == 1  # a decode step uploads the new token only, not the caches
    # events of the previous step: layer / group kernels done, read-backs done
    attn_done = [None] * nl
    idx_done = [None] * G
    out_read = [None] * cfg.group
    idx_read = [None] * 2

    def split_copy(dst, src, streams, after):
        """dst <- src as len(streams) contiguous pieces, piece i on streams[i] once the
        events `after` have fired; returns the events that mark each piece done."""
        fd, fs = dst.view(-1), src.view(-1)
        n = fd.numel()
        per = (n + len(streams) - 1) // len(streams)
        done = []
        for i, st in enumerate(streams):
            lo, hi = i * per, min(n, (i + 1) * per)
            if lo >= hi:
                continue
            with torch.cuda.stream(st):
                for e in after:
                    if e is not None:
                        st.wait_event(e)
                fd[lo:hi].copy_(fs[lo:hi], non_blocking=True)
                e = ev()
                e.record(st)
                done.append(e)
        return done

    def new_token_copy(cache, h_cache, after):
        """The newest cached row of every sequence (position S - 1) from the pinned host
        copy: one small copy per sequence, on the first upload stream."""
        st = ups[0]
        with torch.cuda.stream(st):
            for e in after:
                if e is not None:
                    st.wait_event(e)
            for b in range(cache.shape[0]):
                cache[b, -1].copy_(h_cache[b, -1], non_blocking=True)
            e = ev()
            e.record(st)
        return [e], cache.shape[0] * cache[0, -1].numel() * cache.element_size()

    def step():
        nonlocal h2d, d2h
        in_ready, ind_ready = [], []
        for g in range(G):  # uploads, in the order the kernels need them
            evs = []
            for j, (hx, dx) in enumerate(zip(h_ind, ind[g])):
                if decode and j == 1:  # the key cache: only the new token's row
                    e, n = new_token_copy(dx, hx, [idx_done[g]])
                    evs += e
                    h2d += n
                    continue
                evs += split_copy(dx, hx, ups, [idx_done[g]])
                h2d += hx.numel() * hx.element_size()
            ind_ready.append(evs)
            for l0 in range(min(cfg.group, nl - g * cfg.group)):
                layer = g * cfg.group + l0
                Q, K, V = lay[layer]
                evs = split_copy(Q, h_Q, ups, [attn_done[layer]])
                h2d += h_Q.numel() * 2
                if decode:
                    e, n = new_token_copy(K, h_K, [attn_done[layer]])
                    evs += e
                    h2d += n
                else:
                    evs += split_copy(K, h_K, ups, [attn_done[layer]])
                    h2d += h_K.numel() * 2
                if V is not None:  # separate values (MHA); the MQA latent carries them
                    evs += split_copy(V, h_V, ups, [attn_done[layer]])
                    h2d += h_V.numel() * 2
                in_ready.append(evs)
        for g in range(G):
            qI, kI, w = ind[g]
            ib = idx_bufs[g % 2]
            for e in ind_ready[g]:
                stream.wait_event(e)
            for e in idx_read[g % 2] or []:
                stream.wait_event(e)
            tsi.indexer_topk(qI, kI, w, cfg.topk, idx=ib, workspace=ws, stream=stream)
            e = ev()
            e.record(stream)
            idx_done[g] = e
            if args.readback == "all" or (nl == 0 and g == G - 1):  # no layers: the rows
                idx_read[g % 2] = split_copy(h_idx, ib, downs, [e])
                d2h += ib.numel() * ib.element_size()
            for l0 in range(min(cfg.group, nl - g * cfg.group)):
                layer = g * cfg.group + l0
                Q, K, V = lay[layer]
                for e in in_ready[layer]:
                    stream.wait_event(e)
                for e in out_read[l0] or []:
                    stream.wait_event(e)
                tsi.sparse_attn_group([Q], [K], None, ib, cfg.scale, outs=[outs[l0]],
                                      workspace=ws, stream=stream, Dv=cfg.Dv)
                e = ev()
                e.record(stream)
                attn_done[layer] = e
                if args.readback == "all" or layer == nl - 1:
                    out_read[l0] = split_copy(h_O, outs[l0], downs, [e])
                    d2h += h_O.numel() * 2

    step()  # warm the copy path
    torch.cuda.synchronize()
    h2d = d2h = 0
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for st in ups:
        st.wait_event(a)  # no upload starts before the timer
    for _ in range(steps):
        step()
    for st in ups + downs:
        stream.wait_stream(st)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    return {"value": round(world * G * cfg.B * cfg.T / (ms / 1e3), 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d // steps, "d2h_bytes_per_step": d2h // steps,
            "ms_per_step": round(ms, 2), "steps": steps,
            "note": (f"decode: every step uploads the new token only (queries, gate weights, "
                     f"each layer's Q, and the newest row of the key and latent caches), the "
                     f"caches stay resident; " if decode else
                     f"every layer uploads Q and the latent from one pinned host buffer; ")
                    + f"copies run on {n_copy_streams} streams per direction, overlapping the "
                    f"kernels; read back: "
                    + ("every layer's output and the index rows" if args.readback == "all"
                       else "the step's result (the last layer's output; the index rows "
                            "when there are no layers)")}


# ----------------------------------------------------------------------------- CPU oracle

def run_cpu_oracle(cfg_id, n_idx_rows=None, n_att_rows=None, phase=0):
    """Time the CPU oracle on a bounded, stratified row sample of one IndexShare group of
    the workload and scale it to the metric (group prefill tok/s).

    Default sample: every row up to L = 8192, 512 rows at L = 32768, 256 beyond (the
    indexer + top-k), and 64 of them through the group's attention layers; ``phase``
    shifts the sample so repeated calls cover different rows."""
    import torch

    import oracle
    from top_selection_indexer_gb300 import accounting
    from workloads import get_config
    from workloads.gen import draw

    cfg = get_config(cfg_id)
    cores = oracle.n_threads_default()
    T, S = cfg.T, cfg.S
    n_all = cfg.B * T
    if n_idx_rows is None:
        n_idx_rows = n_all if T <= 8192 else 512 if T <= 32768 else 256
    n_idx_rows = min(n_idx_rows, n_all)
    if n_att_rows is None:
        n_att_rows = 64
    step = n_all / n_idx_rows
    off = (phase * 0.618034 * step) % step if n_idx_rows < n_all else 0.0
    rows = np.unique(np.minimum(n_all - 1, (np.arange(n_idx_rows) * step + off).astype(np.int64)))
    rows = rows[::-1].copy()  # longest rows first
    # keys of row r (sequence r // T, query r % T at position S - T + r % T)
    n_keys = lambda r: max(0, S - T + int(r) % T + 1)  # noqa: E731
    # inputs of the sampled rows only (same distributions as the workload)
    kI = draw((cfg.B, S, cfg.d_I), cfg.qk_dist, cfg.qk_dtype, 1, "cpu", cfg.d_I)
    q_rows = draw((len(rows), cfg.H_I, cfg.d_I), cfg.qk_dist, cfg.qk_dtype, 2, "cpu", cfg.d_I)
    w_rows = draw((len(rows), cfg.H_I), cfg.w_dist, cfg.w_dtype, 3, "cpu")
    t0 = time.perf_counter()
    idx_rows, _ = oracle.indexer_topk_rows(q_rows, kI, w_rows, cfg.topk, T, rows)
    t_idx = time.perf_counter() - t0
    work_idx = sum(n_keys(r) for r in rows)
    t_idx_full = t_idx * accounting.causal_pairs(cfg.B, T, S) / work_idx
    # attention: the group's layers on a subset of those rows
    arows = rows[np.unique(np.linspace(0, len(rows) - 1, min(n_att_rows, len(rows))).astype(int))]
    n_lay = min(cfg.group, cfg.n_layers)
    t_att = t_att_full = 0.0
    if n_lay:
        K = draw((cfg.B, S, cfg.Hkv, cfg.Dqk), "normal", "bf16", 4, "cpu")
        Qr = draw((len(arows), cfg.H, cfg.Dqk), "normal", "bf16", 5, "cpu")
        V = None if cfg.v_from_k else draw((cfg.B, S, cfg.Hkv, cfg.Dv), "normal", "bf16", 6, "cpu")
        pos = {int(r): i for i, r in enumerate(rows)}
        idx_sel = idx_rows[[pos[int(r)] for r in arows]]
        t0 = time.perf_counter()
        for _ in range(n_lay):
            oracle.sparse_attn(Qr, K, V, idx_sel, cfg.scale, T, arows, Dv=cfg.Dv)
        t_att = time.perf_counter() - t0
        work_att = n_lay * sum(min(cfg.topk, n_keys(r)) for r in arows)
        t_att_full = t_att * n_lay * accounting.selected_pairs(cfg.B, T, S, cfg.topk) / work_att
    t_group = t_idx_full + t_att_full
    return {"value": round(cfg.B * T / t_group, 4), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"{len(rows)} stratified query rows (indexer + top-k, fp64) and "
                      f"{len(arows)} of them x {n_lay} layers (sparse attention, fp64) of "
                      f"one IndexShare group ({cfg.B} x {T} query rows over L={S}); scaled "
                      f"by causal pairs / selected keys",
            "sample_seconds": round(t_idx + t_att, 2)}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    vals = []
    info = None
    cores = __import__("oracle").n_threads_default()
    for i in range(args.warmup + args.steps):
        # each step a bounded sample (two rows per core), shifted so the steps cover
        # different rows of the workload
        info = run_cpu_oracle(args.config, n_idx_rows=2 * cores, n_att_rows=cores, phase=i)
        vals.append(info["value"])
    v = statistics.mean(vals[args.warmup:]) if args.steps else vals[-1]
    from workloads import get_config

    cfg = get_config(args.config)
    ms_step = cfg.n_groups * cfg.B * cfg.T / v * 1e3
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 1), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"prefill L={cfg.T}, {cfg.n_layers} layers = {cfg.n_groups} "
                                   "IndexShare groups (CPU oracle on a row sample)",
                       "config_id": cfg.id, "L": cfg.T, "layers": cfg.n_layers},
            "cpu_baseline": {k: info[k] for k in ("kind", "cores", "sample")} | {"value": round(v, 4),
                                                                                "unit": UNIT},
            "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-cp", action="store_true",
                    help="skip the context-parallel indexer measurement after the timed steps")
    ap.add_argument("--copy-streams", type=int, default=4,
                    help="streams per direction for the end-to-end host copies")
    ap.add_argument("--readback", choices=("result", "all"), default="result",
                    help="end-to-end read-back: the step's result (the last layer's output) "
                         "or every layer's output and the index rows")
    ap.add_argument("--no-kl", action="store_true",
                    help="skip the group-centroid KL measurement")
    ap.add_argument("--no-overlap", action="store_true",
                    help="skip the cross-layer top-k overlap measurement after the timed steps")
    ap.add_argument("--no-two-pass", action="store_true",
                    help="skip timing the two-pass indexer beside the default")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the decode measurement (B = 8 over 131072 keys) after the "
                         "prefill step")
    ap.add_argument("--tail-rows", type=int, default=0,
                    help="profiling: only the last R query rows of the prefill")
    ap.add_argument("--groups", type=int, default=0, help="profiling: only the first G groups")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    import torch
    import torch.distributed as dist

    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(
            "cuda", int(os.environ.get("LOCAL_RANK", 0))))
    res = run_gpu(args, rank, world)
    if rank == 0:
        if not args.no_cpu:
            res["cpu_baseline"] = run_cpu_oracle(args.config)
        print(json.dumps(res), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
