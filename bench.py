#!/usr/bin/env python
"""Benchmark of the GB300 Gated DeltaNet layer library.

Headline: batched decode at B=64 rows (K-heads 16, V-heads 48, dk = dv = 128, bf16 inputs,
f32 state pool of 128 slots), reported as GB/s of recurrent-state traffic (each step reads and
writes 64 x 48 x 128 x 128 x 4 B = 402.65 MB) and as a fraction of the measured HBM peak.  The
same JSON line carries the chunked prefill of one T = 4096 sequence (tokens/s, contraction
TFLOP/s), the slot compaction on retire (GB/s), the multi-token and CUDA-graph decode, and the
bf16 projections around the step (weight-streaming GB/s at B=64, TFLOP/s at 4096 rows).  A step is one batched decode step; the
state working set (402.65 MB) exceeds the 129 MB L2, so no L2 flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the float64 CPU oracle on the same decode workload on this host's cores.
Under torchrun (N > 1) every rank runs its own independent replica (weak scaling: decode rows
and slots shard with no exchange); rank 0 prints the line.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "GDN decode state GB/s (% of HBM peak) at B=64; chunked prefill tokens/s"
UNIT = "GB/s"
DECODE_WL = 2
PREFILL_WL = 3
MULTI_T = 4   # tokens per row of the multi-token decode line
E2E_RING = 64   # pinned input buffers cycled by the end-to-end lines (64 x 2.1 MB > L2)

# Per-launch DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the decode kernel
# from one ncu capture at B=64, keyed by the SHA-256 of the kernel source it was taken on.  A
# changed kernel reports null until it is captured again.
DECODE_TRAFFIC = {"ca7142ef62f2d9c6": 353341952}
# The same for the projection kernel's B=64 input projection (hidden 5120, 16480 features).
PROJ_IN_TRAFFIC = {"e339b96ae862774e": 173261568}


def _src_sha(name: str) -> str:
    p = os.path.join(ROOT, "gated_deltanet_linear_09_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_over_ranks(dist, ms: float, units: float, device="cpu"):
    """(max over ranks of the timed region in ms, sum over ranks of the work done).

    Every rank runs an independent replica of the workload (decode rows and slots shard with no
    exchange), so the job's throughput is the summed work over the slowest rank's time."""
    if dist is None:
        return ms, units
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def decode_config(wl, ws: int) -> dict:
    geo = wl.geo
    return {"workload": wl.name, "batch_rows": wl.batch, "k_heads": geo.Hk, "v_heads": geo.Hv,
            "head_dim": geo.dk, "slots": wl.num_slots, "act_dtype": "bf16", "state_dtype": "f32",
            "l2": "no flush: 402.65 MB state working set per step > 129 MB L2",
            "parallelism": f"replicas x{ws} (rows/slots shard, no exchange)"}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while the GPU is busy."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for nm, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = sorted(sm)[len(sm) // 2:]        # upper half: samples taken under load
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------ ours

def run_ours(args, ws, rank, local):
    import torch
    from gated_deltanet_linear_09_gb300 import build as gbuild
    from gated_deltanet_linear_09_gb300 import gdn, synth
    from gated_deltanet_linear_09_gb300.runtime import DecodeGraphs, GatedDeltaNetLayer

    gbuild.build()
    gdn.load()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    hbm_peak, bf16_peak, peak_kind = peaks()

    if args.only == "prefill":
        p_ms, T = time_prefill(torch, synth, GatedDeltaNetLayer, args.steps, args.warmup)
        if rank == 0:
            print(json.dumps({"only": "prefill", "ms": p_ms, "tokens_per_s": T / (p_ms * 1e-3)}))
        return
    if args.only == "proj":
        pr = time_proj(torch, gdn, synth, GatedDeltaNetLayer, hbm_peak, bf16_peak, args.steps)
        if rank == 0:
            print(json.dumps({"only": "proj", **pr}))
        return
    # ---------------- decode, B = 64
    wl = synth.workloads()[DECODE_WL]
    geo = wl.geo
    w = synth.make_weights(geo, wl.seed)
    layer = GatedDeltaNetLayer(geo, w, wl.num_slots)
    rec, conv = synth.make_pool(geo, wl.num_slots, wl.seed, True)
    layer.load_state(rec, conv)
    del rec, conv
    slots = torch.from_numpy(synth.make_slot_idx(wl.num_slots, wl.batch, wl.seed)).cuda()
    # a ring of distinct per-step inputs resident in HBM
    ring = [layer.inputs(synth.decode_step_inputs(wl, t)) for t in range(8)]
    out = torch.empty((wl.batch, geo.zdim), dtype=layer.act, device="cuda")
    stream = torch.cuda.current_stream()
    state_bytes = 2 * wl.batch * geo.Hv * geo.dk * geo.dv * 4
    total_bytes = state_bytes + wl.batch * (2 * 3 * geo.cqkv * 2 + geo.cqkv * 2 + 2 * geo.zdim * 2
                                            + 2 * geo.Hv * 2)

    def step(i):
        x = ring[i % len(ring)]
        layer.decode_step(slots, x["qkv"], x["z"], x["a"], x["b"], out)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    # keep the GPU busy (not idle) between the warm-up and the timed region, so that the clocks
    # and the memory system are in their loaded state when timing starts
    t_busy = time.time() + 0.3
    i = 0
    while time.time() < t_busy:
        for _ in range(50):
            step(i)
            i += 1
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = ev0.elapsed_time(ev1)
    # keep the same load a little longer so the clock sampler sees it
    t_end = time.time() + (1.0 if args.only == "all" else 0.0)
    i = 0
    while time.time() < t_end:
        for _ in range(200):
            step(i)
            i += 1
        torch.cuda.synchronize()
    clocks = sampler.stop()
    ms_local = ms
    ms, total_bytes_moved = reduce_over_ranks(dist, ms, float(state_bytes) * args.steps, "cuda")
    ms_step = ms / args.steps
    gbs = total_bytes_moved / (ms * 1e-3) / 1e9
    per_launch_gbs = state_bytes / (ms_local / args.steps * 1e-3) / 1e9

    if args.only == "decode":
        if rank == 0:
            print(json.dumps({"only": "decode", "ms_per_step": ms_step, "gbs": gbs}), flush=True)
        if dist:
            dist.destroy_process_group()
        return
    # ---------------- e2e: the same step through the public API with host buffers
    # a step's inputs are staged the way a serving loop stages them: packed into one pinned host
    # buffer, brought in with one copy, and handed to the API as views of one device buffer
    keys = list(ring[0].keys())
    nbytes = [ring[0][k].numel() * ring[0][k].element_size() for k in keys]
    offs, o = [], 0
    for nb in nbytes:   # 16-byte aligned views
        offs.append(o)
        o += (nb + 15) // 16 * 16
    h2d = o
    # E2E_RING distinct pinned buffers (> L2 in total): every step's inputs are fresh host data
    host = []
    for j in range(E2E_RING):
        hb = torch.empty(h2d, dtype=torch.uint8).pin_memory()
        src = ring[j % len(ring)] if j < len(ring) else layer.inputs(synth.decode_step_inputs(wl, j))
        for k, o, nb in zip(keys, offs, nbytes):
            hb[o:o + nb].copy_(src[k].cpu().contiguous().view(-1).view(torch.uint8))
        host.append(hb)
    dev_pack = torch.empty(h2d, dtype=torch.uint8, device="cuda")
    dev_in = {k: dev_pack[o:o + nb].view(ring[0][k].dtype).view(ring[0][k].shape)
              for k, o, nb in zip(keys, offs, nbytes)}
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step(i):
        dev_pack.copy_(host[i % len(host)], non_blocking=True)
        layer.decode_step(slots, dev_in["qkv"], dev_in["z"], dev_in["a"], dev_in["b"], out)
        host_out.copy_(out, non_blocking=True)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms, e2e_bytes = reduce_over_ranks(dist, e2e_ms, float(state_bytes) * args.steps, "cuda")
    e2e_gbs = e2e_bytes / (e2e_ms * 1e-3) / 1e9

    # the same step with the kernel reading its inputs from, and writing its output to, the
    # pinned host buffers directly (zero-copy over the coherent CPU-GPU link): the host<->device
    # transfers happen inside the kernel's own loads and stores
    hviews = [{k: host[j][o:o + nb].view(ring[0][k].dtype).view(ring[0][k].shape)
               for k, o, nb in zip(keys, offs, nbytes)} for j in range(len(host))]

    def zc_step(i):
        hv = hviews[i % len(hviews)]
        layer.decode_step(slots, hv["qkv"], hv["z"], hv["a"], hv["b"], host_out)

    for i in range(args.warmup):
        zc_step(i)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        zc_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    zc_ms = e0.elapsed_time(e1)
    zc_ms, zc_bytes = reduce_over_ranks(dist, zc_ms, float(state_bytes) * args.steps, "cuda")
    zc_gbs = zc_bytes / (zc_ms * 1e-3) / 1e9
    del ring, host, dev_in, dev_pack, hviews

    # ---------------- multi-token decode: the same 64 rows, MULTI_T tokens per row per call
    mt_in = []
    for j in range(2):
        toks = [synth.decode_step_inputs(wl, 1000 + MULTI_T * j + t, wl.batch) for t in range(MULTI_T)]
        mt_in.append(layer.inputs({k: np.ascontiguousarray(np.stack([x[k] for x in toks], axis=1))
                                   for k in toks[0]}))
    mt_out = torch.empty((wl.batch, MULTI_T, geo.zdim), dtype=layer.act, device="cuda")
    for j in range(3):
        layer.decode_multi(slots, out=mt_out, **mt_in[j % 2])
    torch.cuda.synchronize()
    m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    mreps = 50
    m0.record(stream)
    for j in range(mreps):
        layer.decode_multi(slots, out=mt_out, **mt_in[j % 2])
    m1.record(stream)
    torch.cuda.synchronize()
    multi_ms = m0.elapsed_time(m1) / mreps
    del mt_in, mt_out

    # ---------------- CUDA-graph decode against eager calls: one row and all 64 rows, per-step
    # time on the GPU timeline (the gaps between eager launches included)
    graphs = DecodeGraphs(layer, [1, 2, 4, 8, 16, 32, 64])
    graph_us = {}
    for B in (1, wl.batch):
        gx = layer.inputs(synth.decode_step_inputs(wl, 2000, B))
        graphs.slot_idx[:B].copy_(slots[:B])
        for k in ("qkv", "z", "a", "b"):
            getattr(graphs, k)[:B].copy_(gx[k])
        eo = torch.empty((B, geo.zdim), dtype=layer.act, device="cuda")
        for mode in ("eager", "graph"):
            def one():
                if mode == "graph":
                    graphs.step(B)
                else:
                    layer.decode_step(slots[:B], gx["qkv"], gx["z"], gx["a"], gx["b"], eo)
            for _ in range(10):
                one()
            torch.cuda.synchronize()
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            greps = 200
            g0.record(stream)
            for _ in range(greps):
                one()
            g1.record(stream)
            torch.cuda.synchronize()
            graph_us[f"B{B}_{mode}_us"] = round(g0.elapsed_time(g1) / greps * 1e3, 2)
    graphs.close()
    del graphs

    # ---------------- compaction at step 256 of the B=64 workload (56 survivors -> [0,56))
    retire = synth.retire_choice(wl.seed, wl.batch, 8, 256)
    keep = [i for i in range(wl.batch) if i not in set(retire.tolist())]
    src = slots.cpu().numpy()[keep].tolist()
    dst = list(range(len(keep)))
    slot_bytes = gdn.gdn_state_slot_bytes(layer.dims, gdn.act_code(layer.act))
    comp_bytes = 2 * len(keep) * slot_bytes
    for _ in range(3):
        layer.compact(src, dst)
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 20
    c0.record(stream)
    for _ in range(reps):
        layer.compact(src, dst)
    c1.record(stream)
    torch.cuda.synchronize()
    comp_ms = c0.elapsed_time(c1) / reps
    del layer
    torch.cuda.empty_cache()

    # ---------------- workload 1: B=16 decode with an L2 flush between steps; workload 4: mixed
    # serving (varlen prefill, decode steps, retire / compact / admit)
    b16 = time_decode_b16(torch, synth, GatedDeltaNetLayer, hbm_peak)
    mixed = time_mixed(torch, synth, GatedDeltaNetLayer)

    # ---------------- the projections around the step
    proj = time_proj(torch, gdn, synth, GatedDeltaNetLayer, hbm_peak, bf16_peak)

    # ---------------- chunked prefill, one sequence of T = 4096
    p_ms, T = time_prefill(torch, synth, GatedDeltaNetLayer, 10, 3)
    pwl = synth.workloads()[PREFILL_WL]
    pgeo = pwl.geo
    Hk, Hv, d, C = pgeo.Hk, pgeo.Hv, pgeo.dk, pwl.chunk
    flops = T * (Hv * (8 * C * d + 6 * d * d) + Hk * 4 * C * d)
    p_tflops = flops / (p_ms * 1e-3) / 1e12
    p_bytes = T * (pgeo.cqkv * 2 + pgeo.zdim * 2 * 2 + 2 * Hv * 2) + Hv * d * d * 4
    # launches of one call: the library pipelines windows of chunks, the first a wave of intra
    # CTAs (SMs // Hk chunks), the others the chunks whose intra CTAs fit beside the Hv chains
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    nch = (T + C - 1) // C
    win = max(1, (nsm - Hv) // Hk)
    win0 = max(win, nsm // Hk)
    p_windows = 1 + max(0, -(-(nch - win0) // win))
    # 64-dim heads (zero-padded to 128 on the tensor-core path): same sequence and head counts
    g64 = synth.Geometry(Hk, Hv, 64, 64, 4, synth.BF16)
    p64_ms, _ = time_prefill(torch, synth, GatedDeltaNetLayer, 5, 2, geo=g64)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    traffic = None
    ent = DECODE_TRAFFIC.get(_src_sha("gdn_decode.cu"))
    if ent:
        traffic = ent
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": decode_config(wl, ws),
        "row_steps_per_s": round(wl.batch * ws * args.steps / (ms * 1e-3), 1),
        "hbm_frac_state": round(per_launch_gbs / hbm_peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(per_launch_gbs, 2), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(per_launch_gbs / hbm_peak, 4),
                     "traffic": traffic, "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": state_bytes,
                     "total_bytes_per_launch_incl_conv_io": total_bytes,
                     "kernel": "decode_kernel<128,128,bf16>"},
        "e2e": {"value": round(zc_gbs, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(zc_ms / args.steps, 5),
                "mode": "gdn_decode_step called with pinned host buffers: the kernel reads the "
                        "inputs and writes the output over the CPU-GPU link",
                "host_buffers": E2E_RING},
        "e2e_copies": {"value": round(e2e_gbs, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / args.steps, 5),
                       "mode": "one packed pinned-host to device copy, the call on device "
                               "buffers, one device to pinned-host copy of the output"},
        "gpu_launches": args.steps,
        "prefill": {"workload": pwl.name, "tokens_per_s": round(T / (p_ms * 1e-3), 1),
                    "ms": round(p_ms, 4), "contraction_gflop": round(flops / 1e9, 3),
                    "tflops": round(p_tflops, 3),
                    "roofline": {"bound": "tensor", "achieved": round(p_tflops, 3),
                                 "peak": bf16_peak, "unit": "TFLOP/s",
                                 "frac": round(p_tflops / bf16_peak, 5), "peak_kind": peak_kind},
                    "io_bytes": p_bytes, "windows_per_call": p_windows,
                    "launches_per_call": 2 * p_windows},
        "prefill_d64": {"workload": f"prefill_T{T}_Hk{Hk}_Hv{Hv}_d64_bf16",
                        "path": "tensor-core path, heads zero-padded to 128",
                        "ms": round(p64_ms, 4), "tokens_per_s": round(T / (p64_ms * 1e-3), 1)},
        "decode_multi": {"tokens_per_row": MULTI_T, "rows": wl.batch, "ms": round(multi_ms, 5),
                         "tokens_per_s": round(wl.batch * MULTI_T / (multi_ms * 1e-3), 1),
                         "state_gbs": round(state_bytes / (multi_ms * 1e-3) / 1e9, 1),
                         "state_bytes_per_token": state_bytes // (wl.batch * MULTI_T),
                         "single_step_tokens_per_s": round(wl.batch / (ms_step * 1e-3), 1)},
        "decode_graphs": dict(graph_us, buckets=[1, 2, 4, 8, 16, 32, 64]),
        "decode_b16": b16,
        "mixed_serving": mixed,
        "proj": proj,
        "compact": {"pairs": len(keep), "bytes": comp_bytes, "ms": round(comp_ms, 4),
                    "gbs": round(comp_bytes / (comp_ms * 1e-3) / 1e9, 1),
                    "hbm_frac": round(comp_bytes / (comp_ms * 1e-3) / 1e9 / hbm_peak, 4)},
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and ws == 1:   # the oracle baseline: rank 0 at N = 1 only
        line["cpu_baseline"] = cpu_baseline(args)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def time_proj(torch, gdn, synth, GatedDeltaNetLayer, hbm_peak, bf16_peak, reps=20):
    """The projections around the step.  Decode-shaped: in_proj and out_proj of the 64 rows of
    the B=64 workload (hidden 5120), weight-streaming bound, reported as GB/s of algorithmic
    bytes (weights + activations + outputs) against the HBM peak; each launch reads weights
    the previous launches did not touch (copies rotated, > 2 x L2 per rotation).
    Prefill-shaped: in_proj of the T = 4096 sequence (hidden 4096), tensor bound, TFLOP/s
    against the bf16 peak."""
    from gated_deltanet_linear_09_gb300.runtime import pack_weight
    stream = torch.cuda.current_stream()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    res = {}

    def randn(shape, scale):
        return (torch.randn(shape, device="cuda", generator=gen) * scale).to(torch.bfloat16)

    def timed(fn, n):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    wl = synth.workloads()[DECODE_WL]
    geo = wl.geo
    H = synth.PROJ_HIDDEN[geo.Hv]
    layer = GatedDeltaNetLayer(geo, synth.make_weights(geo, wl.seed), 1)
    B = wl.batch
    n_in, n_out = synth.proj_rows(geo), H
    l2 = 129e6
    r_in = max(2, int(2 * l2 // (n_in * H * 2)) + 1)
    r_out = max(2, int(2 * l2 // (n_out * geo.zdim * 2)) + 1)
    w_in = [pack_weight(randn((n_in, H), H ** -0.5)) for _ in range(r_in)]
    w_out = [pack_weight(randn((n_out, geo.zdim), geo.zdim ** -0.5)) for _ in range(r_out)]
    x = randn((B, H), 1.0)
    o = randn((B, geo.zdim), 1.0)
    t = {"qkv": torch.empty((B, geo.cqkv), dtype=torch.bfloat16, device="cuda"),
         "z": torch.empty((B, geo.zdim), dtype=torch.bfloat16, device="cuda"),
         "a": torch.empty((B, geo.Hv), dtype=torch.bfloat16, device="cuda"),
         "b": torch.empty((B, geo.Hv), dtype=torch.bfloat16, device="cuda")}
    y = torch.empty((B, H), dtype=torch.bfloat16, device="cuda")
    ms_in = timed(lambda i: gdn.gdn_in_proj(layer.dims, x, w_in[i % r_in], t["qkv"], t["z"],
                                            t["b"], t["a"], layer.status), reps)
    ms_out = timed(lambda i: gdn.gdn_out_proj(layer.dims, o, w_out[i % r_out], y, layer.status),
                   reps)
    b_in = n_in * H * 2 + B * H * 2 + B * n_in * 2
    b_out = n_out * geo.zdim * 2 + B * geo.zdim * 2 + B * H * 2
    for name, ms, nbytes, n, k in (("in_proj", ms_in, b_in, n_in, H),
                                   ("out_proj", ms_out, b_out, n_out, geo.zdim)):
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[f"decode_{name}"] = {
            "rows": B, "features": n, "hidden" if name == "in_proj" else "k": k,
            "us": round(ms * 1e3, 2), "bytes": nbytes, "gbs": round(gbs, 1),
            "hbm_frac": round(gbs / hbm_peak, 4),
            "tflops": round(2.0 * B * n * k / (ms * 1e-3) / 1e12, 2)}
    res["decode_in_proj"]["roofline"] = {
        "bound": "hbm", "achieved": res["decode_in_proj"]["gbs"], "peak": hbm_peak,
        "unit": "GB/s", "frac": res["decode_in_proj"]["hbm_frac"],
        "traffic": PROJ_IN_TRAFFIC.get(_src_sha("gdn_proj.cu"))}
    del w_in, w_out, layer
    torch.cuda.empty_cache()

    pwl = synth.workloads()[PREFILL_WL]
    pgeo = pwl.geo
    PH = synth.PROJ_HIDDEN[pgeo.Hv]
    T = pwl.seq_lens[0]
    player = GatedDeltaNetLayer(pgeo, synth.make_weights(pgeo, pwl.seed), 1)
    pn = synth.proj_rows(pgeo)
    pw = pack_weight(randn((pn, PH), PH ** -0.5))
    px = randn((T, PH), 1.0)
    pt = {"qkv": torch.empty((T, pgeo.cqkv), dtype=torch.bfloat16, device="cuda"),
          "z": torch.empty((T, pgeo.zdim), dtype=torch.bfloat16, device="cuda"),
          "a": torch.empty((T, pgeo.Hv), dtype=torch.bfloat16, device="cuda"),
          "b": torch.empty((T, pgeo.Hv), dtype=torch.bfloat16, device="cuda")}
    ms_p = timed(lambda i: gdn.gdn_in_proj(player.dims, px, pw, pt["qkv"], pt["z"], pt["b"],
                                           pt["a"], player.status), max(5, reps // 4))
    fl = 2.0 * T * pn * PH
    tf = fl / (ms_p * 1e-3) / 1e12
    res["prefill_in_proj"] = {"rows": T, "features": pn, "hidden": PH, "us": round(ms_p * 1e3, 2),
                              "tflops": round(tf, 1), "bf16_frac": round(tf / bf16_peak, 4)}
    res["hidden_sizes"] = {str(k): v for k, v in synth.PROJ_HIDDEN.items()}
    res["kernel"] = ("proj_kernel: 256 features x 64 rows per CTA (two tcgen05 M=128 x N=64 "
                     "accumulators), packed weight blocks, cp.async ring, cluster split-K; from "
                     "512 unsplit rows 256 features x 256 rows (N=256 accumulators)")
    return res


def time_decode_b16(torch, synth, GatedDeltaNetLayer, hbm_peak, steps=64):
    """Workload 1: B=16 rows of a 64-slot pool, Hk=16, Hv=32.  Its 67.1 MB of state traffic per
    step would sit in the 129 MB L2, so every timed step is preceded (outside its events) by a
    write of a 256 MB buffer that evicts it; the step times are summed from per-step events."""
    wl = synth.workloads()[1]
    geo = wl.geo
    layer = GatedDeltaNetLayer(geo, synth.make_weights(geo, wl.seed), wl.num_slots)
    rec, conv = synth.make_pool(geo, wl.num_slots, wl.seed, True)
    layer.load_state(rec, conv)
    del rec, conv
    slots = torch.from_numpy(synth.make_slot_idx(wl.num_slots, wl.batch, wl.seed)).cuda()
    ring = [layer.inputs(synth.decode_step_inputs(wl, t)) for t in range(4)]
    out = torch.empty((wl.batch, geo.zdim), dtype=layer.act, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    state_bytes = 2 * wl.batch * geo.Hv * geo.dk * geo.dv * 4
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for i in range(3):
        layer.decode_step(slots, out=out, **ring[i % 4])
    for i in range(steps):
        flush.zero_()
        evs[i][0].record(stream)
        layer.decode_step(slots, out=out, **ring[i % 4])
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in evs) / steps
    gbs = state_bytes / (ms * 1e-3) / 1e9
    del layer, flush, ring
    torch.cuda.empty_cache()
    return {"workload": wl.name, "rows": wl.batch, "us_per_step": round(ms * 1e3, 2),
            "state_bytes_per_step": state_bytes, "gbs": round(gbs, 1),
            "hbm_frac": round(gbs / hbm_peak, 4),
            "row_steps_per_s": round(wl.batch / (ms * 1e-3), 1),
            "l2": "256 MB buffer written between steps, outside the timed events", "steps": steps}


def time_mixed(torch, synth, GatedDeltaNetLayer):
    """Workload 4, mixed serving: varlen prefill of 8 sequences (lengths ~ U[128, 8192]) into a
    16-slot pool, then 512 decode steps over the 8 rows; every 64 steps 2 rows retire, the live
    slots are compacted to the pool's prefix and 2 new sequences are admitted by prefill.  Every
    input is staged on the device first; each call is timed with its own events and the phases
    are summed (prefill tokens/s over all prefills, decode row-steps/s over all decode steps)."""
    wl = synth.workloads()[4]
    geo = wl.geo
    layer = GatedDeltaNetLayer(geo, synth.make_weights(geo, wl.seed), wl.num_slots)
    B = wl.batch
    stream = torch.cuda.current_stream()

    def i32(x):
        return torch.from_numpy(np.asarray(x, np.int32)).cuda()

    # the schedule, staged: (kind, args) in call order
    plan = []
    lens = synth.mixed_seq_lens(wl.seed, B, tag=0)
    row_slots = synth.make_slot_idx(wl.num_slots, B, wl.seed)
    plan.append(("prefill", lens, row_slots.copy(), 0))
    for t in range(wl.steps):
        if t > 0 and t % 64 == 0:
            retire = synth.retire_choice(wl.seed, B, 2, t)
            keep = np.array([i for i in range(B) if i not in set(retire.tolist())], np.int32)
            dst = np.arange(len(keep), dtype=np.int32)
            plan.append(("compact", row_slots[keep].tolist(), dst.tolist(), t))
            new_lens = synth.mixed_seq_lens(wl.seed, 2, tag=t)
            new_slots = np.array([len(keep), len(keep) + 1], np.int32)
            plan.append(("prefill", new_lens, new_slots, t))
            row_slots = np.concatenate([dst, new_slots]).astype(np.int32)
        plan.append(("decode", None, row_slots.copy(), t))
    staged = []
    for kind, a, sl, t in plan:
        if kind == "prefill":
            cu = synth.cu_seqlens(a)
            xs = layer.inputs(synth.make_token_inputs(geo, int(cu[-1]), wl.seed, 7, t))
            staged.append((kind, (i32(cu), i32(sl), xs, int(cu[-1]))))
        elif kind == "decode":
            staged.append((kind, (i32(sl), layer.inputs(synth.make_token_inputs(geo, B, wl.seed, 100, t)))))
        else:
            staged.append((kind, (a, sl)))
    max_tokens = max(v[3] for k, v in staged if k == "prefill")
    layer.workspace(B, max_tokens)
    out_p = torch.empty((max_tokens, geo.zdim), dtype=layer.act, device="cuda")
    out_d = torch.empty((B, geo.zdim), dtype=layer.act, device="cuda")
    torch.cuda.synchronize()
    times = {"prefill": [], "decode": [], "compact": []}
    tokens = 0
    for kind, v in staged:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if kind == "prefill":
            cu, sl, xs, T = v
            layer.prefill(cu, sl, None, out=out_p[:T], **xs)
            tokens += T
        elif kind == "decode":
            sl, xs = v
            layer.decode_step(sl, out=out_d, **xs)
        else:
            layer.compact(*v)
        e1.record(stream)
        times[kind].append((e0, e1))
    torch.cuda.synchronize()
    ms = {k: sum(a.elapsed_time(b) for a, b in evs) for k, evs in times.items()}
    status = int(layer.status.item())
    del layer, staged, out_p
    torch.cuda.empty_cache()
    return {"workload": wl.name, "prefill_tokens": tokens, "prefill_calls": len(times["prefill"]),
            "prefill_ms": round(ms["prefill"], 3),
            "prefill_tokens_per_s": round(tokens / (ms["prefill"] * 1e-3), 1),
            "decode_steps": len(times["decode"]), "rows": B, "decode_ms": round(ms["decode"], 3),
            "decode_row_steps_per_s": round(B * len(times["decode"]) / (ms["decode"] * 1e-3), 1),
            "compactions": len(times["compact"]), "compact_ms": round(ms["compact"], 3),
            "total_ms": round(sum(ms.values()), 3), "status": status}


def time_prefill(torch, synth, GatedDeltaNetLayer, reps, warmup, geo=None):
    """Average time of one chunked prefill of the T = 4096 sequence (inputs resident in HBM), on
    the workload's geometry or on `geo`."""
    pwl = synth.workloads()[PREFILL_WL]
    pgeo = geo if geo is not None else pwl.geo
    player = GatedDeltaNetLayer(pgeo, synth.make_weights(pgeo, pwl.seed), pwl.num_slots)
    T = pwl.seq_lens[0]
    px = player.inputs(synth.make_token_inputs(pgeo, T, pwl.seed, 0))
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    psl = torch.tensor([0], dtype=torch.int32, device="cuda")
    pout = torch.empty((T, pgeo.zdim), dtype=player.act, device="cuda")
    for _ in range(warmup):
        player.prefill(cu, psl, None, px["qkv"], px["z"], px["a"], px["b"], pout)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(reps):
        player.prefill(cu, psl, None, px["qkv"], px["z"], px["a"], px["b"], pout)
    p1.record(stream)
    torch.cuda.synchronize()
    return p0.elapsed_time(p1) / reps, T


# ------------------------------------------------------------------------------ oracle timing

def _oracle_decode_setup(rows):
    import oracle
    from gated_deltanet_linear_09_gb300 import synth
    wl = synth.workloads()[DECODE_WL]
    geo = wl.geo
    w = {k: np.asarray(v, np.float64) for k, v in synth.make_weights(geo, wl.seed).items()}
    rng = np.random.default_rng(0)
    rec = rng.normal(0, 0.02, (rows, geo.Hv, geo.dk, geo.dv))
    conv = np.asarray(synth.in_dtype(rng.normal(0, 1, (rows, geo.K - 1, geo.cqkv)), geo.act),
                      np.float64)
    return oracle, wl, geo, w, rec, conv


def _oracle_decode_steps(n_steps, rows):
    oracle, wl, geo, w, rec, conv = _oracle_decode_setup(rows)
    slots = np.arange(rows, dtype=np.int32)
    xs = [{k: np.asarray(v, np.float64) for k, v in
           synth_inputs(wl, t, rows).items()} for t in range(min(n_steps, 4))]
    t0 = time.perf_counter()
    for t in range(n_steps):
        oracle.decode_step(geo.oracle_dims(), w, rec, conv, slots, **xs[t % len(xs)])
    return time.perf_counter() - t0, geo


def _oracle_rows_worker(job):
    """One worker of the all-core oracle run: rows [r0, r1) of the B=64 sample, n_steps steps.
    Returns its own compute seconds (process start-up and imports are not oracle work)."""
    n_steps, r0, r1, total_rows = job
    oracle, wl, geo, w, rec, conv = _oracle_decode_setup(r1 - r0)
    slots = np.arange(r1 - r0, dtype=np.int32)
    xs = [{k: np.ascontiguousarray(np.asarray(v, np.float64)[r0:r1]) for k, v in
           synth_inputs(wl, t, total_rows).items()} for t in range(min(n_steps, 4))]
    t0 = time.perf_counter()
    for t in range(n_steps):
        oracle.decode_step(geo.oracle_dims(), w, rec, conv, slots, **xs[t % len(xs)])
    return time.perf_counter() - t0


def _oracle_rows_parallel(n_steps, rows):
    """The oracle on all host cores: the rows split over spawned worker processes (the GPU
    context of this process is never forked).  Returns (span seconds, workers)."""
    import multiprocessing as mp
    nw = max(1, min(os.cpu_count() or 1, rows))
    bounds = [(rows * j // nw, rows * (j + 1) // nw) for j in range(nw)]
    with mp.get_context("spawn").Pool(nw) as pool:
        secs = pool.map(_oracle_rows_worker, [(n_steps, a, b, rows) for a, b in bounds])
    return max(secs), nw


def _oracle_prefill_worker(job):
    """One worker of the oracle prefill sample: the T-token prefix of the T = 4096 workload's
    sequence, run by the float64 oracle over the given K-heads (each with its V-heads and its
    slice of the [q | k | v] channels; heads are independent).  Returns its compute seconds."""
    T, k_heads = job
    import oracle
    from gated_deltanet_linear_09_gb300 import synth
    wl = synth.workloads()[PREFILL_WL]
    geo = wl.geo
    w = synth.make_weights(geo, wl.seed)
    xs = synth.make_token_inputs(geo, T, wl.seed, 0)
    r = geo.Hv // geo.Hk
    secs = 0.0
    for kh in k_heads:
        vh = list(range(kh * r, kh * r + r))
        ch = ([kh * geo.dk + e for e in range(geo.dk)] +
              [geo.Hk * geo.dk + kh * geo.dk + e for e in range(geo.dk)] +
              [2 * geo.Hk * geo.dk + h * geo.dv + e for h in vh for e in range(geo.dv)])
        zc = [h * geo.dv + e for h in vh for e in range(geo.dv)]
        sub = synth.Geometry(1, r, geo.dk, geo.dv, geo.K, geo.act)
        ws = dict(A_log=np.asarray(w["A_log"], np.float64)[vh],
                  dt_bias=np.asarray(w["dt_bias"], np.float64)[vh],
                  conv_w=np.asarray(w["conv_w"], np.float64)[ch],
                  norm_w=np.asarray(w["norm_w"], np.float64))
        xin = dict(qkv=np.ascontiguousarray(np.asarray(xs["qkv"], np.float64)[:, ch]),
                   z=np.ascontiguousarray(np.asarray(xs["z"], np.float64)[:, zc]),
                   a=np.ascontiguousarray(np.asarray(xs["a"], np.float64)[:, vh]),
                   b=np.ascontiguousarray(np.asarray(xs["b"], np.float64)[:, vh]))
        rec = np.zeros((1, r, geo.dk, geo.dv))
        conv = np.zeros((1, geo.K - 1, sub.cqkv))
        t0 = time.perf_counter()
        oracle.prefill(sub.oracle_dims(), ws, rec, conv, [0, T], [0], None, **xin)
        secs += time.perf_counter() - t0
    return secs


def _oracle_prefill(T, workers):
    """(span seconds, workers used): the 16 K-heads split over spawned worker processes."""
    import multiprocessing as mp
    from gated_deltanet_linear_09_gb300 import synth
    Hk = synth.workloads()[PREFILL_WL].geo.Hk
    nw = max(1, min(workers, Hk))
    jobs = [(T, list(range(j, Hk, nw))) for j in range(nw)]
    if nw == 1:
        return _oracle_prefill_worker(jobs[0]), 1
    with mp.get_context("spawn").Pool(nw) as pool:
        secs = pool.map(_oracle_prefill_worker, jobs)
    return max(secs), nw


def synth_workload():
    from gated_deltanet_linear_09_gb300 import synth
    return synth.workloads()[DECODE_WL]


def synth_inputs(wl, t, rows):
    from gated_deltanet_linear_09_gb300 import synth
    return synth.make_token_inputs(wl.geo, rows, wl.seed, 100, t)


def cpu_baseline(args):
    """The oracle as it stands (float64) on a bounded sample of the decode workload: on all host
    cores (rows split over processes), and on one thread."""
    import oracle
    oracle.build()
    rows = 64
    geo = synth_workload().geo
    per_row_step = 2 * geo.Hv * geo.dk * geo.dv * 4
    n_par = 96
    span, nw = _oracle_rows_parallel(n_par, rows)
    n_one = 48
    sec, _ = _oracle_decode_steps(n_one, rows)
    # the chunked prefill's workload (T = 4096, Hk = 16, Hv = 32): the oracle's sequential
    # recurrence over a prefix of the sequence, all K-heads, on all cores and on one thread
    tp_all, tp_one = 4096, 1024
    p_span, p_nw = _oracle_prefill(tp_all, os.cpu_count() or 1)
    p_one, _ = _oracle_prefill(tp_one, 1)
    prefill = {"tokens_per_s": round(tp_all / p_span, 1), "unit": "tokens/s", "cores": p_nw,
               "kind": "oracle",
               "sample": f"{tp_all} tokens of the T=4096 workload's sequence, all 16 "
                         f"K-heads split over {p_nw} processes, float64 C oracle",
               "seconds": round(p_span, 2),
               "single_thread": {"tokens_per_s": round(tp_one / p_one, 1), "cores": 1,
                                 "sample": f"the first {tp_one} tokens, all 16 K-heads, one thread",
                                 "seconds": round(p_one, 2)}}
    return {"value": round(per_row_step * rows * n_par / span / 1e9, 4), "unit": UNIT,
            "cores": nw, "kind": "oracle",
            "sample": f"{n_par} decode steps x {rows} rows of the B=64 workload, rows split over "
                      f"{nw} processes, float64 C oracle",
            "seconds": round(span, 2),
            "single_thread": {"value": round(per_row_step * rows * n_one / sec / 1e9, 4),
                              "unit": UNIT, "cores": 1,
                              "sample": f"{n_one} decode steps x {rows} rows, one thread",
                              "seconds": round(sec, 2)},
            "prefill": prefill}


def run_reference(args, ws, rank):
    """--impl reference: the oracle on the host cores, same metric and workload shape."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    rows = 64
    # one step = one full B=64 decode step of the oracle, its rows split over the host cores
    # (the warm-up steps run inside the same workers, untimed)
    geo = synth_workload().geo
    _oracle_rows_parallel(max(1, min(args.warmup, 2)), rows)
    sec, nw = _oracle_rows_parallel(args.steps, rows)
    state_bytes = 2 * rows * args.steps * geo.Hv * geo.dk * geo.dv * 4
    v = state_bytes / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": decode_config(synth_workload(), ws),
        "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": nw, "kind": "oracle",
                         "sample": f"{args.steps} full B=64 decode steps, rows split over {nw} "
                                   "processes, float64 C oracle"},
        "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default="all", choices=["all", "decode", "prefill", "proj"],
                    help="decode: only the B=64 decode timing (used for profiling captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)


if __name__ == "__main__":
    main()
