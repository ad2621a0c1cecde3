#!/usr/bin/env python
"""Benchmark of adaptive-precision attention prefill on GB300.

One step = one call of the whole path (key/value statistics, NVFP4 quantizer,
pass 1 with the hot test, pass 2 on the hot tiles, log-sum-exp merge) on one
synthetic seeded workload with its bf16 inputs resident in HBM.  By default the
2048-query x 122880-key Llama-3.2-3B-shaped GQA layer (B=1, Hq=24, Hkv=8, d=128,
tail-aligned causal, eps=0.005; 516 MB of inputs, larger than L2); --workload
names any of the five (tiny, llama3b_2048x122880, prefill_8k, batched_32k,
shortq_131k_d256).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gpu|reference] [--workload NAME]

Prints one JSON line.  Under torchrun every rank processes its own layer
(weak scaling, no data-path collective); the time is the max over ranks.
The reference arm times the CPU oracle (FP64 emulation of the same method)
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from mixed_precision_attention_gb300 import synth  # noqa: E402

WORKLOAD = "llama3b_2048x122880"  # the layer the headline metric is quoted on
METRIC = "ms and effective TFLOP/s, 2048q x 122880k GQA layer; % of tensor-core roofline"
UNIT = "TFLOP/s"
PAGE_APA_MS = 5.200  # the blog's APA time for this layer on an RTX 5090 (context)
FP4_PER_BF16 = 13.5 / 2.25  # nominal dense FP4 : BF16 tensor ratio
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNELS_PER_STEP = 6  # stats, finalize, quantize, pass 1, pass-2 ranking, pass 2 (+merge)
KERNELS_PER_STEP_EPS0 = 3  # FP16 copy of V (two launches), pass 2 (+merge)


# ----------------------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK}, "measured"
    return dict(FALLBACK), "fallback"


def visible_counts(w: synth.Workload):
    """[ng, T] visible (row, key) pairs per (16-row group, 64-key tile) of one KV head."""
    G, R, T, off = w.G, w.G * w.Nq, (w.Nkv + 63) // 64, w.Nkv - w.Nq
    ng = (R + 15) // 16
    p = np.arange(ng * 16)
    valid = p < R
    last = (p // G + off) if w.causal else np.full(p.shape, w.Nkv - 1)
    t0 = np.arange(T) * 64
    cnt = np.clip(np.minimum(last[:, None] + 1, w.Nkv) - t0[None, :], 0, 64) * valid[:, None]
    return cnt.reshape(ng, 16, T).sum(1)


def algorithmic(w: synth.Workload, hot_mask):
    """Algorithmic work: FP4 flops of pass 1, 16-bit flops of pass 2, pair counts."""
    vis = visible_counts(w)  # [ng, T]
    T = vis.shape[1]
    m = np.ascontiguousarray(hot_mask).view(np.uint32)
    bits = np.unpackbits(m.view(np.uint8), bitorder="little").reshape(m.shape[:-1] + (-1,))[..., :T].astype(bool)
    pairs = int(vis.sum()) * w.B * w.Hkv
    hot_pairs = int((bits * vis[None, None]).sum())
    cold_pairs = pairs - hot_pairs
    d = w.d
    # QK^T on every pair, the ones product of the row sums (N = 16 per pair, as the
    # method states it; the default kernel sums the codes on CUDA cores instead), PV
    # on cold pairs
    F1 = pairs * (2 * d + 32) + cold_pairs * 2 * d
    F2 = hot_pairs * 4 * d                         # exact QK^T and PV on hot pairs
    tiles_vis = int((vis > 0).sum()) * w.B * w.Hkv
    hot_tiles = int((bits & (vis > 0)[None, None]).sum())
    # pass 2 walks, per 128-row block (8 groups), the union of its groups' hot tiles
    ng = vis.shape[0]
    nb = (ng + 7) // 8
    gb = np.zeros(bits.shape[:2] + (nb * 8, T), bool)
    gb[:, :, :ng] = bits & (vis > 0)[None, None]
    union = gb.reshape(bits.shape[:2] + (nb, 8, T)).any(3)
    vb = np.zeros((nb * 8, T), bool)
    vb[:ng] = vis > 0
    block_tiles_vis = int(vb.reshape(nb, 8, T).any(1).sum()) * w.B * w.Hkv
    block_tiles_hot = int(union.sum())
    return dict(pairs=pairs, hot_pairs=hot_pairs, cold_pairs=cold_pairs, F1=F1, F2=F2,
                hot_frac=hot_tiles / max(1, tiles_vis), hot_pair_frac=hot_pairs / max(1, pairs),
                block_tiles_hot=block_tiles_hot, block_tiles_vis=block_tiles_vis)


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "mixed_precision_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, pci_bus_id=None):
        self.pci = (pci_bus_id or "").lower()
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                if self.pci and self.pci[-12:] not in parts[1].lower():
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2])]
        smax = [num(r[3]) for r in rows if num(r[3])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup():
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    """The largest x over all ranks (every rank gets it); x itself on one rank."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_layer_seed(w: synth.Workload, rank: int) -> int:
    """Each rank runs its own layer (weak scaling): the workload's seed plus the rank."""
    return w.seed + rank


def whole_job_tflops(world: int, flops_per_rank: float, ms_max: float) -> float:
    """Throughput of the whole job: every rank's work over the slowest rank's time."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


def cpu_sample(w: synth.Workload, q, k, v, heads=(0,), groups_per_head=16, seed=0, b=0):
    """The oracle's APA emulation on a bounded sample: `groups_per_head` 16-row
    groups spread over the rows of each listed KV head of sequence b.  Returns
    (seconds, flops of exact attention on the sampled rows, rows, threads)."""
    import oracle
    ng = oracle.n_groups(w.Hq, w.Hkv, w.Nq)
    rng = np.random.default_rng(seed)
    units = []
    for h in heads:
        for g in np.sort(rng.choice(ng, size=min(groups_per_head, ng), replace=False)):
            units.append((b, h, int(g)))
    units = np.array(units, np.int32)
    rows = [rr for (b, h, g) in units for rr in oracle.group_rows(w.Hq, w.Hkv, w.Nq, b, h, g)]
    off = w.Nkv - w.Nq
    flops = sum(4.0 * w.d * (min(w.Nkv, pos + off + 1) if w.causal else w.Nkv) for (_, _, pos) in rows)
    t0 = time.perf_counter()
    oracle.apa(q, k, v, causal=w.causal, eps=w.eps, units=units)
    return time.perf_counter() - t0, flops, len(rows), oracle.num_threads()


def config_dict(w):
    mb = (w.B * w.Hq * w.Nq + 2 * w.B * w.Hkv * w.Nkv) * w.d * 2 / 1e6
    l2 = (f"inputs larger than L2 (bf16 Q/K/V {mb:.0f} MB vs 126 MB L2); no flush" if mb > 126 else
          f"inputs ({mb:.1f} MB) fit in L2: timed back to back, L2-warm")
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq, "Nkv": w.Nkv, "d": w.d,
            "causal": w.causal, "eps": w.eps, "key_tile": 64, "gqa_packing": True, "l2": l2}


def pass1_hosts_kv_quantizer(w: synth.Workload, sms: int) -> bool:
    """Whether the library quantizes the K/V tiles inside the pass-1 launch for this
    workload (it does when the pass-1 CTAs leave at least 8 SMs free: three 128-row
    blocks per CTA at d <= 128, one at d = 256)."""
    nblk = (w.G * w.Nq + 127) // 128
    ctas = w.B * w.Hkv * (nblk if w.d > 128 else (nblk + 2) // 3)
    return sms - ctas >= 8


def stage_bytes(w: synth.Workload, kv_in_pass1: bool):
    """Algorithmic DRAM bytes of the quantizer stage and of the pass-1 stage.

    Statistics: K, V and Q read once (bf16), per-tile key sums written and read.
    K/V quantizer: K and V read again, E2M1 codes + UE4M3 scales written
    (0.5625 B per element), the FP16 copy of V written (2 B per element).  Q
    blocks: Q read, codes + scales written.  Pass 1: the K/V blobs read once per
    KV head (1.125 d B per key), the Q codes read, the state (d + 3 floats per
    packed row) written.  The K/V quantizer counts where it runs."""
    BH, d, T = w.B * w.Hkv, w.d, (w.Nkv + 63) // 64
    kv_el, q_el = BH * w.Nkv * d, w.B * w.Hq * w.Nq * d
    rows = BH * ((w.G * w.Nq + 127) // 128) * 128
    stats = 2 * kv_el * 2 + q_el * 2 + 2 * BH * T * d * 4
    qblocks = q_el * 2 + q_el * 0.5625
    kvq = 2 * kv_el * 2 + 2 * kv_el * 0.5625 + kv_el * 2
    p1 = 1.125 * d * w.Nkv * BH + q_el * 0.5625 + rows * (d + 3) * 4
    return (stats + qblocks + (0 if kv_in_pass1 else kvq), p1 + (kvq if kv_in_pass1 else 0))


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    _, rank, _ = dist_setup()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    w = synth.WORKLOADS[args.workload]
    q, k, v = synth.generate(w)
    times, flops_all, nrows, threads = [], [], 0, 1
    for step in range(args.warmup + args.steps):
        b = step % w.B
        dt, fl, nrows, threads = cpu_sample(w, q, k, v, heads=(step % w.Hkv,), groups_per_head=8, seed=step, b=b)
        if step >= args.warmup:
            times.append(dt)
            flops_all.append(fl)
    t = float(np.sum(times))
    value = float(np.sum(flops_all)) / t / 1e12
    cores = len(os.sched_getaffinity(0))
    sample = (f"oracle APA emulation (FP64, OpenMP) of 8 sixteen-row groups of one KV head per step "
              f"({nrows} query rows x up to {w.Nkv} keys, incl. that head's NVFP4 quantization), "
              f"KV head = step mod {w.Hkv}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(cores, threads), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm
def profiled_traffic_for(w: synth.Workload, src_hash: str):
    """DRAM bytes per pass-1 launch from the committed ncu summary of this workload."""
    path = os.path.join(ROOT, "profiles", f"pass1_{w.name}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    hm = re.search(r"source hash:\s*`?([0-9a-f]{16})", text)
    tm = re.search(r"dram bytes per launch:\s*`?([0-9.eE+]+)", text)
    if not hm or not tm or hm.group(1) != src_hash:
        return None
    return float(tm.group(1))


def run_gpu(args):
    import torch

    import mixed_precision_attention_gb300 as apa
    from mixed_precision_attention_gb300 import _lib

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = _lib.load()

    w = synth.WORKLOADS[args.workload]
    q, k, v = synth.generate(w, seed=rank_layer_seed(w, rank))  # each rank: its own layer
    tq, tk, tv = (synth.to_torch_bf16(a, dev) for a in (q, k, v))
    B, Hq, Hkv, Nq, Nkv, d = w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.d
    workspace = torch.empty(apa.workspace_bytes(B, Hq, Hkv, Nq, Nkv, d, w.eps), dtype=torch.uint8, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    # one untimed call with the hot mask: the algorithmic work of this layer
    _, _, mask = apa.attention(tq, tk, tv, causal=w.causal, eps=w.eps, return_hot_mask=True, workspace=workspace)
    apa.check_error(dev)
    work = algorithmic(w, mask.cpu().numpy())
    flops_exact = w.flops_exact

    def timed(eps, steps, warmup, ws_tensor, sample_clocks=False, **options):
        for _ in range(warmup):
            apa.attention(tq, tk, tv, causal=w.causal, eps=eps, workspace=ws_tensor, **options)
        torch.cuda.synchronize(dev)
        barrier(world)
        torch.cuda.synchronize(dev)
        clk = None
        if sample_clocks:
            pci = getattr(torch.cuda.get_device_properties(dev), "pci_bus_id", None)
            clk = ClockSampler(pci if isinstance(pci, str) else None)
            clk.start()
        lib.apa_stage_timing(1)
        stream = torch.cuda.current_stream(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            apa.attention(tq, tk, tv, causal=w.causal, eps=eps, workspace=ws_tensor, **options)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        torch.cuda.synchronize(dev)
        ms3 = (ctypes.c_float * 3)()
        calls = ctypes.c_int()
        lib.apa_stage_timing_read(ms3, ctypes.byref(calls))
        lib.apa_stage_timing(0)
        clocks = clk.stop() if clk else None
        apa.check_error(dev)
        return e0.elapsed_time(e1) / steps, [x / max(1, calls.value) for x in ms3], clocks

    ms, stages, clocks = timed(w.eps, args.steps, args.warmup, workspace, sample_clocks=True)
    ms = max_over_ranks(ms, world, dev)
    value = whole_job_tflops(world, flops_exact, ms)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": PAGE_APA_MS / ms if w.name == WORKLOAD else None,
            "dtype": "nvfp4 (e2m1 x ue4m3) + bf16, fp32 accumulate",
            "data": "synthetic", "config": config_dict(w), "gpu_launches": KERNELS_PER_STEP * args.steps}

    pk, pk_kind = peaks()
    # pass 1 is timed as a stage of its own (a burst of at most a few ms): the burst
    # BF16 peak times the nominal FP4 : BF16 ratio; pass 2 likewise
    fp4_peak = pk["bf16_tflops"] * FP4_PER_BF16
    bf16_peak = pk["bf16_tflops"]
    t_q, t_p1, t_p2 = stages
    kv_in_p1 = pass1_hosts_kv_quantizer(w, sms)
    q_bytes, p1_bytes = stage_bytes(w, kv_in_p1)
    src = kernel_source_hash(["apa_pass1.cu", "quant_tile.cuh", "tc.cuh", "apa_internal.h"])
    p1_ach = work["F1"] / (t_p1 * 1e-3) / 1e12
    p1_gbs = p1_bytes / (t_p1 * 1e-3) / 1e9
    kernel = "pass1 (tcgen05 kind::mxf4nvf4" + (", K/V quantizer in the same launch)" if kv_in_p1 else ")")
    if d > 128:
        # the short-query d = 256 shape streams K/V: its pass-1 launch (with the K/V
        # quantizer) is bound by HBM, not by the tensor cores
        line["roofline"] = {"kernel": kernel, "bound": "hbm", "achieved": p1_gbs, "peak": pk["hbm_gbs"],
                            "unit": "GB/s", "frac": p1_gbs / pk["hbm_gbs"], "traffic": profiled_traffic_for(w, src),
                            "peak_note": f"{pk_kind} copy bandwidth", "bytes_per_launch": p1_bytes,
                            "ms_per_launch": t_p1}
    else:
        line["roofline"] = {"kernel": kernel, "bound": "tensor", "achieved": p1_ach,
                            "peak": fp4_peak, "unit": "TFLOP/s", "frac": p1_ach / fp4_peak,
                            "traffic": profiled_traffic_for(w, src),
                            "peak_note": f"dense NVFP4 = {pk_kind} burst bf16 x {FP4_PER_BF16:g} (nominal ratio)",
                            "flops_per_launch": work["F1"], "ms_per_launch": t_p1}
    p2_ach = work["F2"] / (t_p2 * 1e-3) / 1e12 if t_p2 > 0 else 0.0
    line["stages"] = {
        "quantize": {"ms": t_q, "bytes": q_bytes, "hbm_gbs": q_bytes / (t_q * 1e-3) / 1e9,
                     "hbm_frac": q_bytes / (t_q * 1e-3) / 1e9 / pk["hbm_gbs"],
                     "holds": "statistics, key mean, Q blocks" + ("" if kv_in_p1 else ", K/V tiles")},
        "pass1": {"ms": t_p1, "tflops_fp4": p1_ach, "frac_fp4_peak": p1_ach / fp4_peak, "bytes": p1_bytes,
                  "hbm_gbs": p1_gbs, "hbm_frac": p1_gbs / pk["hbm_gbs"], "kv_quantizer_inside": kv_in_p1},
        "pass2_merge": {"ms": t_p2, "tflops_16bit": p2_ach, "frac_bf16_peak": p2_ach / bf16_peak},
    }
    line["tensor_roofline_frac"] = (work["F1"] / fp4_peak + work["F2"] / bf16_peak) / 1e12 / (ms * 1e-3)
    line["hot_tile_frac"] = work["hot_frac"]
    line["hot_pair_frac"] = work["hot_pair_frac"]
    # what pass 2 computes: 128 x 64 (row, key) slots per block-tile in the union
    line["pass2_union"] = {"block_tiles": work["block_tiles_hot"],
                           "frac_of_visible_block_tiles": work["block_tiles_hot"] / max(1, work["block_tiles_vis"]),
                           "pair_slots_per_hot_pair": work["block_tiles_hot"] * 128 * 64 / max(1, work["hot_pairs"])}
    line["peaks"] = {"source": pk_kind, **pk}
    line["clocks"] = clocks

    if not args.skip_extras:
        # the same library at eps = 0: every visible tile exact (BF16 Q K^T, FP16 P.V)
        ws0 = torch.empty(apa.workspace_bytes(B, Hq, Hkv, Nq, Nkv, d, 0.0), dtype=torch.uint8, device=dev)
        ms0, st0, _ = timed(0.0, max(3, args.steps // 4), 3, ws0)
        del ws0
        ms0 = max_over_ranks(ms0, world, dev)
        line["eps0_all_exact"] = {"ms_per_step": ms0, "tflops": whole_job_tflops(world, flops_exact, ms0),
                                  "frac_bf16_peak": flops_exact / (ms0 * 1e-3) / 1e12 / bf16_peak,
                                  "stages_ms": {"v_fp16_copy": st0[0], "pass2": st0[2]},
                                  "speedup_of_apa": ms0 / ms, "gpu_launches_per_step": KERNELS_PER_STEP_EPS0}
        for sweep_eps in w.eps_sweep:
            if sweep_eps in (0.0, w.eps):
                continue
            ms_e, st_e, _ = timed(sweep_eps, max(3, args.steps // 4), 3, workspace)
            _, _, m_e = apa.attention(tq, tk, tv, causal=w.causal, eps=sweep_eps, return_hot_mask=True,
                                      workspace=workspace)
            line.setdefault("eps_sweep", {})[str(sweep_eps)] = {
                "ms_per_step": max_over_ranks(ms_e, world, dev), "stages_ms": st_e,
                "hot_pair_frac": algorithmic(w, m_e.cpu().numpy())["hot_pair_frac"]}
        # the accuracy option: Q as two FP4 terms in pass 1 (one block per pass-1 CTA)
        ws_q2 = torch.empty(apa.workspace_bytes(B, Hq, Hkv, Nq, Nkv, d, w.eps, q_residual=True),
                            dtype=torch.uint8, device=dev)
        msq2, stq2, _ = timed(w.eps, max(3, args.steps // 4), 3, ws_q2, q_residual=True)
        del ws_q2
        msq2 = max_over_ranks(msq2, world, dev)
        line["q_residual"] = {"ms_per_step": msq2, "tflops": whole_job_tflops(world, flops_exact, msq2),
                              "cost_vs_apa": msq2 / ms - 1.0, "stages_ms": stq2}
        # the other accuracy option: least-squared-error block scales (quantizer only)
        mslse, stlse, _ = timed(w.eps, max(3, args.steps // 4), 3, workspace, lse_scales=True)
        mslse = max_over_ranks(mslse, world, dev)
        line["lse_scales"] = {"ms_per_step": mslse, "cost_vs_apa": mslse / ms - 1.0, "stages_ms": stlse}
        # the row sums by the ones-MMA (the page's form) instead of in registers
        msmma, stmma, _ = timed(w.eps, max(3, args.steps // 4), 3, workspace, rowsum_mma=True)
        msmma = max_over_ranks(msmma, world, dev)
        line["rowsum_mma"] = {"ms_per_step": msmma, "cost_vs_apa": msmma / ms - 1.0, "stages_ms": stmma}
        # the hot test weighted by value norm: its own hot set, so its own pass-2 work
        ws_vw = torch.empty(apa.workspace_bytes(B, Hq, Hkv, Nq, Nkv, d, w.eps, value_weighted=True),
                            dtype=torch.uint8, device=dev)
        _, _, mvw = apa.attention(tq, tk, tv, causal=w.causal, eps=w.eps, return_hot_mask=True, workspace=ws_vw,
                                  value_weighted=True)
        msvw, stvw, _ = timed(w.eps, max(3, args.steps // 4), 3, ws_vw, value_weighted=True)
        del ws_vw
        msvw = max_over_ranks(msvw, world, dev)
        line["value_weighted"] = {"ms_per_step": msvw, "cost_vs_apa": msvw / ms - 1.0, "stages_ms": stvw,
                                  "hot_pair_frac": algorithmic(w, mvw.cpu().numpy())["hot_pair_frac"]}
        # end to end through the host-buffer entry point: H2D of q, k, v from pinned
        # memory, the whole path, D2H of out and lse, every step
        hq, hk, hv = (synth.to_torch_bf16(a).pin_memory() for a in (q, k, v))
        hout, hlse, _ = apa.attention_host(hq, hk, hv, causal=w.causal, eps=w.eps)  # pinned outputs, reused
        n_e2e = max(3, min(args.steps, 10))
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            apa.attention_host(hq, hk, hv, causal=w.causal, eps=w.eps, out=hout, lse=hlse)
        e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / n_e2e, world, dev)
        line["e2e"] = {"value": whole_job_tflops(world, flops_exact, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
                       "h2d_bytes_per_step": q.nbytes + k.nbytes + v.nbytes,
                       "d2h_bytes_per_step": B * Hq * Nq * d * 4 + B * Hq * Nq * 4}
        if rank == 0 and world == 1:
            heads = (0, min(5, Hkv - 1)) if Hkv > 1 else (0,)
            dt, fl, nrows, threads = cpu_sample(w, q, k, v, heads=heads, groups_per_head=8)
            line["cpu_baseline"] = {
                "value": fl / dt / 1e12, "unit": UNIT, "cores": min(threads, len(os.sched_getaffinity(0))),
                "kind": "oracle", "seconds": dt,
                "sample": f"oracle APA emulation (FP64, OpenMP) of {8 * len(heads)} sixteen-row groups "
                          f"({nrows} query rows) of KV heads {', '.join(map(str, heads))}, all {w.Nkv} keys "
                          f"each, incl. the per-head NVFP4 quantization"}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--workload", choices=sorted(synth.WORKLOADS), default=WORKLOAD,
                    help="which synthetic workload (default: the 2048 x 122880 Llama-3.2-3B layer)")
    ap.add_argument("--skip-extras", action="store_true",
                    help="time the main loop only (no eps=0 / host / CPU legs); used for profiler runs")
    args = ap.parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
