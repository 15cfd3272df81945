"""Benchmark of the CSA2 decode hot path on GB300.

One step = one decode pass of the whole index-and-attend path for a batch of
sequences of the Full-layer decode workload (32 sequences x 65,536 visible
entries; 32 x 128 MXFP4 indexer, Top-512, 64 x 512 attention over the 512
selected FP4 latents + 128 FP8 SWA rows):

    csa2_index_topk_bf16 (indexer q -> MXFP4 in the scan's prologue, scan,
      Top-512)  ->  csa2_sparse_attn_decode

with the KV cache resident in HBM. The timed region holds exactly --steps
steps, each bracketed by CUDA events on the launching stream, with an L2
flush between steps outside the events: a 512 MiB write followed by a
512 MiB read, so that no input of the step is cached and the step is not
charged for writing back the flush's dirty lines.

Prints one JSON line. `value` is queries/s over all ranks; `e2e` is the same
metric with each step's inputs copied from pinned host memory and its
outputs copied back inside the timed region; `roofline` reports the indexer
scan kernel (68 algorithmic bytes per scored entry) against the measured HBM
copy bandwidth, timed in a second loop of csa2_index_score on the same
inputs (the same kernel; inside csa2_index_topk it also builds the Top-K
histogram in its epilogue); `cpu_baseline` is the CPU oracle on a bounded
sample.

The line's `workloads` object holds the other workloads, each measured the
same way on its own caches: the single-query decode (4,096 entries; its
latency per query), the Reindex decode with the 2,048 x 8 block pool (8 x
1,048,576 entries), the long-context decode with 1 Full + 3 Reuse layers
(4 x 1,048,576), and the prefill chunk as a pipeline (4,096 queries after
126,976 entries: q -> MXFP4, causal scan, Top-512, sparse attention).

--impl reference runs the CPU oracle instead (the reference arm).
Multi-GPU: launched with torch.distributed.run, every rank runs its own
batch of sequences (weak scaling, no data-path collective).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD_ID = 1
METRIC = "CSA2 decode queries/s at 64K-1M ctx; indexer-scan HBM GB/s vs GB300 peak"
IK_BYTES_PER_ENTRY = 68        # 64 B E2M1 + 4 B E8M0 per indexer key
KV_BYTES_PER_ENTRY = 288       # 256 B E2M1 + 32 B E4M3 per main-KV latent
L2_FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------------------- host logic

def dist_env():
    """(rank, world_size, local_rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_sequences(rank: int, B: int) -> list[int]:
    """Sequence ids this rank owns: each rank runs its own batch of B."""
    return list(range(rank * B, (rank + 1) * B))


def reduce_max(value: float, world: int, device=None) -> float:
    """Max over ranks (barrier semantics come from the collective)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


FP4_PER_BF16 = 13.5 / 2.25   # nominal dense FP4 : BF16 tensor rate


def tensor_peak_tflops():
    """(bf16 TFLOP/s of a kernel timed alone, its source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
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
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def step_config(wl, B, N, L, K, W, world):
    """The `config` object of the bench line, shared by both arms."""
    return {"workload": wl.name if B == wl.B else f"{wl.name}_batch{B}", "sequences_per_gpu": B,
            "visible_entries": N, "layers_sharing_topk": L,
            "indexer": "32 heads x 128 MXFP4", "topk": K, "heads": 64, "head_dim": 512, "swa": W,
            "l2": "flushed between steps (512 MiB write + 512 MiB read)", "parallelism": f"dp{world} (sequences)"}


# ---------------------------------------------------------------------------- GPU arm

def build_inputs(csa2, torch, wid, B, N, L, reindex, seqs, device, planted_blocks=0):
    """Synthetic resident caches and per-step inputs, packed with the library's
    own packers on the device (indexer K: MXFP4; main KV: E2M1 + E4M3/16;
    SWA: E4M3). With planted_blocks, each sequence's keys hold that many
    blocks of 8 aligned with its Full-layer query (the Reindex workload)."""
    from fp4_kv_cache_02_gb300.inputs import (CAP_ALIGN, device_normal, device_planted_keys, device_uniform,
                                              round_up, seed_for)
    cap = round_up(N, CAP_ALIGN)
    ik_data = torch.empty(B, cap, 64, dtype=torch.uint8, device=device)
    ik_scale = torch.empty(B, cap, 4, dtype=torch.uint8, device=device)
    kv_data = torch.empty(B, cap, 256, dtype=torch.uint8, device=device)
    kv_scale = torch.empty(B, cap, 32, dtype=torch.uint8, device=device)
    q_idx = torch.empty(B, 32, 128, dtype=torch.bfloat16, device=device)
    w = torch.empty(B, 32, dtype=torch.float32, device=device)
    Q = torch.empty(B, L, 64, 512, dtype=torch.bfloat16, device=device)
    swa = torch.empty(B, L, 128, 512, dtype=torch.uint8, device=device)
    q_re = torch.empty(B, 32, 128, dtype=torch.bfloat16, device=device) if reindex else None
    w_re = torch.empty(B, 32, dtype=torch.float32, device=device) if reindex else None
    for b, s in enumerate(seqs):
        seed = seed_for(wid, s)
        q_idx[b] = device_normal((32, 128), 4 * seed + 3, device)
        w[b] = device_uniform((32,), 4 * seed + 3, device)
        ik = device_normal((cap, 128), 4 * seed + 1, device)
        if planted_blocks:
            device_planted_keys(ik, q_idx[b], w[b], N, planted_blocks, 4 * seed + 7)
        csa2.csa2_quant_mxfp4(ik, ik_data[b], ik_scale[b])
        del ik
        kv = device_normal((cap, 512), 4 * seed + 2, device)
        csa2.csa2_pack_kv_fp4(kv, kv_data[b], kv_scale[b])
        del kv
        Q[b] = device_normal((L, 64, 512), 4 * seed + 4, device, scale=1.0 / math.sqrt(512))
        csa2.csa2_pack_fp8_e4m3(device_normal((L, 128, 512), 4 * seed + 5, device), swa[b])
        if reindex:
            q_re[b] = device_normal((32, 128), 4 * seed + 6, device)
            w_re[b] = device_uniform((32,), 4 * seed + 6, device)
    n_visible = torch.full((B,), N, dtype=torch.int32, device=device)
    torch.cuda.synchronize()
    return dict(cap=cap, ik_data=ik_data, ik_scale=ik_scale, kv_data=kv_data, kv_scale=kv_scale, q_idx=q_idx, w=w,
                Q=Q, swa=swa, n_visible=n_visible, q_re=q_re, w_re=w_re)


class Ctx:
    """What every measurement of one process shares: device, stream, ranks
    and the L2 flush."""

    def __init__(self, torch, device, world, rank, local_rank):
        self.torch, self.device, self.world, self.rank, self.local_rank = torch, device, world, rank, local_rank
        self.stream = torch.cuda.current_stream(device)
        self._flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self._flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)

    def flush_l2(self):
        self._flush.fill_(1)
        self._flush_rd.max()

    def timed(self, fn, n):
        """Mean CUDA-event time (ms) of fn over n launches, L2 flushed before each."""
        torch = self.torch
        tot = 0.0
        for _ in range(n):
            self.flush_l2()
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(self.stream)
            fn()
            b_.record(self.stream)
            b_.synchronize()
            tot += a.elapsed_time(b_)
        return tot / n


def measure_decode(csa2, ctx, wid, B, steps, warmup, use_graph=True, with_e2e=True):
    """One decode workload, measured four ways: (1) eager steps with an event
    between stages (the per-stage breakdown), (2) the step captured as a CUDA
    graph and replayed (the timed number, under clock sampling), (3) the
    indexer scan alone, scheduled as inside the step (its roofline), and (4)
    end to end with host copies. Each of the `steps` timed steps is preceded
    by an L2 flush outside its events."""
    torch, device, stream, world = ctx.torch, ctx.device, ctx.stream, ctx.world
    from fp4_kv_cache_02_gb300.inputs import WORKLOADS
    wl = WORKLOADS[wid]
    reindex = wl.kind == "reindex"
    N, L, K, W = wl.N, wl.L, 512, 128
    seqs = rank_sequences(ctx.rank, B)
    inp = build_inputs(csa2, torch, wid, B, N, L, reindex, seqs, device,
                       planted_blocks=wl.planted_blocks if reindex else 0)
    cap = inp["cap"]
    flush_l2 = ctx.flush_l2

    q_data = torch.empty(B, 32, 64, dtype=torch.uint8, device=device)
    q_sc = torch.empty(B, 32, 4, dtype=torch.uint8, device=device)
    idx = torch.empty(B, K, dtype=torch.int32, device=device)
    out = torch.empty(B, L, 64, 512, dtype=torch.bfloat16, device=device)
    NBLK = 2048
    iws = csa2.index_topk_workspace(B, cap, K, NBLK if reindex else 0, device=device)
    aws = csa2.attn_workspace(B * L, K, W, device=device)
    pool = idx_full = rws = None
    if reindex:
        pool = torch.empty(B, NBLK * 8, dtype=torch.int32, device=device)
        idx_full = torch.empty(B, K, dtype=torch.int32, device=device)
        rws = csa2.index_topk_workspace(B, NBLK * 8, K, device=device)

    # the step as named stages (each a sequence of public C-ABI calls); the
    # per-step inputs and outputs are looked up in `io`, which the end-to-end
    # loop points at one of two buffer sets
    io = {k_: inp[k_] for k_ in ("q_idx", "w", "Q", "swa", "q_re", "w_re")}
    io["out"], io["idx"] = out, idx

    # the indexer q goes in as bf16: the scan quantises it to MXFP4 in its prologue
    def st_index():
        if reindex:
            csa2.csa2_index_topk_bf16(io["q_idx"], io["w"], inp["ik_data"], inp["ik_scale"], inp["n_visible"], K,
                                      idx_full, iws, pool_blocks=NBLK, pool=pool)
        else:
            csa2.csa2_index_topk_bf16(io["q_idx"], io["w"], inp["ik_data"], inp["ik_scale"], inp["n_visible"], K,
                                      io["idx"], iws)

    def st_reindex():
        csa2.csa2_index_topk_bf16(io["q_re"], io["w_re"], inp["ik_data"], inp["ik_scale"], inp["n_visible"], K,
                                  io["idx"], rws, positions=pool)

    def st_attn():
        csa2.csa2_sparse_attn_decode(io["Q"], inp["kv_data"], inp["kv_scale"], inp["n_visible"], io["idx"], io["swa"],
                                     io["out"], aws)

    stages = [("index_topk_pool" if reindex else "index_topk", st_index)]
    if reindex:
        stages.append(("reindex_topk", st_reindex))
    stages.append(("sparse_attn", st_attn))
    # our kernels per step: workspace clear + scan (q quantisation, fused histogram and, with the pool,
    # block maxima) + select + finalize 4; pool: clear, histogram, select, finalize, expand 5; reindex:
    # clear, scan, select, finalize 4; attention: as the library plans it for B * L query-layers
    n_launches = 4 + (5 + 4 if reindex else 0) + csa2.lib().csa2_sparse_attn_kernel_launches(B * L, K, W)

    def step(ev=None):
        for j, (_, fn) in enumerate(stages):
            if ev is not None:
                ev[j].record(stream)
            fn()
        if ev is not None:
            ev[len(stages)].record(stream)

    for _ in range(warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    assert csa2.csa2_get_last_error() == 0

    nst = len(stages)
    # (1) eager steps with an event between stages: the per-stage breakdown
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(steps)]
    for i in range(steps):
        flush_l2()
        step(evs[i])
    torch.cuda.synchronize()
    stage = [0.0] * nst
    eager_total = 0.0
    for e in evs:
        for j in range(nst):
            stage[j] += e[j].elapsed_time(e[j + 1])
        eager_total += e[0].elapsed_time(e[nst])
    stage_ms = {nm: s_ / steps for (nm, _), s_ in zip(stages, stage)}
    eager_ms = eager_total / steps

    # (2) the step captured once as a CUDA graph (the kernels' programmatic
    # dependent launches become graph edges) and replayed: the timed number
    graph = None
    if use_graph:
        side = torch.cuda.Stream(device)
        side.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream(device).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(warmup):
            flush_l2()
            graph.replay()
        torch.cuda.synchronize()
        assert csa2.csa2_get_last_error() == 0
    run_step = graph.replay if graph is not None else step
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with ClockSampler(ctx.local_rank) as clk:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("timed_steps")   # lets ncu filter to the timed region
        for i in range(steps):
            flush_l2()                     # L2 flush between timed steps, outside the events
            ev_a[i].record(stream)
            run_step()
            ev_b[i].record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
    ms = sum(a_.elapsed_time(b_) for a_, b_ in zip(ev_a, ev_b)) / steps
    ms_max = reduce_max(ms, world, device)

    # (3) the scan kernel alone, for its roofline (same inputs, L2 flushed),
    # scheduled as inside the step: tiles claimed from per-sequence counters
    csa2.csa2_quant_mxfp4(inp["q_idx"], q_data, q_sc)
    tile_ctr = torch.zeros(2 * B, dtype=torch.int32, device=device)
    scores = torch.empty(B, cap, dtype=torch.float32, device=device)
    scan_ms = ctx.timed(lambda: csa2.csa2_index_score_claimed(q_data, q_sc, inp["w"], inp["ik_data"],
                                                              inp["ik_scale"], inp["n_visible"], scores, tile_ctr,
                                                              stream=stream), steps)
    del scores

    # (3b) Reuse layers: the attention alone, per layer (the step's call) and
    # fused (each selected tile gathered once per pair of layers), on the
    # step's indices, L2 flushed before each
    attn_alone = None
    if L >= 2:
        attn_alone = {
            "per_layer_ms": ctx.timed(st_attn, steps),
            "fused_reuse_ms": ctx.timed(lambda: csa2.csa2_sparse_attn_reuse(
                io["Q"], inp["kv_data"], inp["kv_scale"], inp["n_visible"], io["idx"], io["swa"], io["out"], aws),
                steps)}
        assert csa2.csa2_get_last_error() == 0

    res = {"wl": wl, "B": B, "N": N, "L": L, "K": K, "W": W, "reindex": reindex, "ms": ms_max,
           "eager_ms": eager_ms, "stage_ms": stage_ms, "scan_ms": scan_ms, "n_launches": n_launches,
           "graph": graph is not None, "clocks": clk.summary(), "attn_alone": attn_alone}
    if not with_e2e:
        return res

    # (4) end to end: per-step inputs from pinned host memory, outputs back.
    # Each step copies its inputs host -> device and its outputs (attention
    # output, Top-K indices) device -> host, each as one packed buffer (one copy
    # a direction keeps the host's enqueue work small). The copies run on their own streams
    # and overlap the neighbouring steps' compute (two buffer sets); the number
    # is the span from the first input copy to the last output copy over K
    # steps. No L2 flush here: the step's inputs exceed L2.
    in_keys = [k_ for k_ in ("q_idx", "w", "Q", "swa", "q_re", "w_re") if inp.get(k_) is not None]

    def flat(specs, alloc):
        # one buffer holding every tensor of `specs` at 256-byte aligned offsets:
        # a step moves its inputs (outputs) with one copy
        offs, off = [], 0
        for k_, ref in specs:
            nb = ref.numel() * ref.element_size()
            offs.append((k_, off, nb, ref))
            off = (off + nb + 255) // 256 * 256
        buf = alloc(off)
        return buf, {k_: buf[o:o + nb].view(ref.dtype).view(ref.shape) for k_, o, nb, ref in offs}

    pinned = lambda n: torch.empty(n, dtype=torch.uint8).pin_memory()
    on_dev = lambda n: torch.empty(n, dtype=torch.uint8, device=device)
    host_in_flat, host_in = flat([(k_, inp[k_]) for k_ in in_keys], pinned)
    for k_ in in_keys:
        host_in[k_].copy_(inp[k_].cpu())
    slot_io = []
    for _ in range(2):
        in_flat, d = flat([(k_, inp[k_]) for k_ in in_keys], on_dev)
        out_flat, o = flat([("out", out), ("idx", idx)], on_dev)
        h_out_flat, h = flat([("out", out), ("idx", idx)], pinned)
        d.update(o)
        d["in_flat"], d["out_flat"], d["h_out_flat"] = in_flat, out_flat, h_out_flat
        d["h_idx"] = h["idx"]
        slot_io.append(d)
    h2d = host_in_flat.numel()
    d2h = slot_io[0]["h_out_flat"].numel()
    default_io = dict(io)
    slot_run = []
    for d in slot_io:
        io.update({k_: d[k_] for k_ in in_keys + ["out", "idx"]})
        for k_ in in_keys:
            d[k_].copy_(inp[k_])
        step()  # eager warm-up with this buffer set
        if graph is not None:
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_):
                step()
            slot_run.append(g_.replay)
        else:
            sio = {k_: d[k_] for k_ in in_keys + ["out", "idx"]}
            slot_run.append(lambda sio=sio: (io.update(sio), step()))
    io.update(default_io)
    torch.cuda.synchronize()
    main = torch.cuda.current_stream(device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_loop(n):
        for i in range(n):
            sl = i % 2
            d = slot_io[sl]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[sl])   # step i-2 has read this buffer set
                d["in_flat"].copy_(host_in_flat, non_blocking=True)
                h2d_done[sl].record(s_in)
            main.wait_event(h2d_done[sl])
            if i >= 2:
                main.wait_event(d2h_done[sl])        # step i-2's outputs have left this buffer set
            slot_run[sl]()
            comp_done[sl].record(main)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[sl])
                d["h_out_flat"].copy_(d["out_flat"], non_blocking=True)
                d2h_done[sl].record(s_out)

    e2e_loop(max(warmup, 2))
    torch.cuda.synchronize()
    t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_a.record(main)
    s_in.wait_stream(main)
    h0 = time.perf_counter()
    e2e_loop(steps)
    host_ms = (time.perf_counter() - h0) * 1e3 / steps
    s_out.wait_stream(main)
    t_b.record(s_out)
    t_b.synchronize()
    e2e_ms = reduce_max(t_a.elapsed_time(t_b) / steps, world, device)
    assert torch.equal(slot_io[(steps - 1) % 2]["h_idx"].to(device), idx)  # same result as the timed steps
    res.update({"e2e_ms": e2e_ms, "host_ms": host_ms, "h2d": h2d, "d2h": d2h})
    return res


def decode_summary(res, world, hbm_peak, peak_kind):
    """The figures of one decode workload: queries/s (device-timed graph
    replays and end to end), stage times, the indexer scan's HBM roofline and
    the attention stage's algorithmic bytes over its time."""
    B, N, L, K, W = res["B"], res["N"], res["L"], res["K"], res["W"]
    ms = res["ms"]
    scan_bytes = B * N * IK_BYTES_PER_ENTRY
    scan_gbs = scan_bytes / (res["scan_ms"] * 1e-3) / 1e9
    # attention: gathered latents + SWA rows + Q in + bf16 O out, per query-layer
    attn_bytes = B * L * (K * KV_BYTES_PER_ENTRY + W * 512 + 2 * 64 * 512 * 2)
    attn_ms = res["stage_ms"]["sparse_attn"]
    out = {
        "workload": res["wl"].name, "sequences": world * B, "visible_entries": N, "layers_sharing_topk": L,
        "queries_per_s": round(world * B / (ms * 1e-3), 1), "ms_per_step": round(ms, 5),
        "us_per_query": round(ms * 1e3 / B, 3),
        "entries_scored_per_s": round(world * B * (N + (2048 * 8 if res["reindex"] else 0)) / (ms * 1e-3), 1),
        "ms_per_step_eager": round(res["eager_ms"], 5),
        "stages_ms": {k_: round(v, 5) for k_, v in res["stage_ms"].items()},
        "scan_roofline": {"kernel": "index_score", "bound": "hbm", "achieved": round(scan_gbs, 1),
                          "peak": hbm_peak, "peak_kind": f"{peak_kind} HBM copy bandwidth", "unit": "GB/s",
                          "frac": round(scan_gbs / hbm_peak, 4), "ms": round(res["scan_ms"], 5),
                          "algorithmic_bytes_per_launch": scan_bytes},
        "attention": {"algorithmic_bytes_per_step": attn_bytes, "ms": round(attn_ms, 5),
                      "achieved_gbs": round(attn_bytes / (attn_ms * 1e-3) / 1e9, 1),
                      "frac": round(attn_bytes / (attn_ms * 1e-3) / 1e9 / hbm_peak, 4),
                      "hbm_floor_us": round(attn_bytes / (hbm_peak * 1e9) * 1e6, 2)},
        "gpu_launches_per_step": res["n_launches"],
        "clocks": res["clocks"],
    }
    if res.get("attn_alone"):
        # the Reuse layers' attention timed alone: the step's per-layer call and
        # the fused call (bit-identical outputs), with the selected rows' bytes
        # read once per sequence for the fused one
        aa = res["attn_alone"]
        out["reuse_attention"] = {
            "per_layer_ms": round(aa["per_layer_ms"], 5), "fused_reuse_ms": round(aa["fused_reuse_ms"], 5),
            "note": "csa2_sparse_attn_decode vs csa2_sparse_attn_reuse on the step's indices, eager, L2 flushed"}
    if "e2e_ms" in res:
        out["e2e"] = {"value": round(world * B / (res["e2e_ms"] * 1e-3), 1), "unit": "queries/s",
                      "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                      "ms_per_step": round(res["e2e_ms"], 5)}
    return out


def run_gpu(args):
    import torch
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    from fp4_kv_cache_02_gb300 import csa2
    from fp4_kv_cache_02_gb300.inputs import WORKLOADS

    ctx = Ctx(torch, device, world, rank, local_rank)
    wid = args.workload
    wl = WORKLOADS[wid]
    B = args.batch or wl.B
    res = measure_decode(csa2, ctx, wid, B, args.steps, args.warmup, use_graph=not args.no_graph)
    torch.cuda.empty_cache()

    # ---- the fused KV append, for its roofline and its decode latency ----
    app = measure_append(csa2, torch, B, device, args.steps, ctx.flush_l2, ctx.stream)
    pre = measure_prefill(csa2, ctx, max(3, min(args.steps, 10)), *args.prefill_shape) if args.prefill else None
    torch.cuda.empty_cache()

    # ---- the other workloads, each its own decode step (or prefill pipeline) ----
    hbm_peak, peak_kind = peaks()
    extra = {}
    for w_ in args.workloads:
        if w_ == wid or w_ not in WORKLOADS:
            continue
        if WORKLOADS[w_].kind == "prefill":
            continue  # the prefill pipeline comes from measure_prefill
        r_ = measure_decode(csa2, ctx, w_, WORKLOADS[w_].B, min(args.steps, 100), args.warmup,
                            use_graph=not args.no_graph)
        extra[str(w_)] = decode_summary(r_, world, hbm_peak, peak_kind)
        del r_
        torch.cuda.empty_cache()
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return None

    ms_max = res["ms"]
    main_sum = decode_summary(res, world, hbm_peak, peak_kind)
    scan_bytes = main_sum["scan_roofline"]["algorithmic_bytes_per_launch"]
    scan_gbs = main_sum["scan_roofline"]["achieved"]
    traffic = None
    tp = os.path.join(ROOT, "profiles", "index_score_traffic.json")
    if os.path.exists(tp):
        try:
            rec = json.load(open(tp))
            # the ncu figure of this workload's scan launch, when one was taken
            if rec.get("workload") == wl.name and B == wl.B:
                traffic = rec.get("dram_bytes_per_launch")
        except (ValueError, OSError):
            traffic = None
    L = res["L"]
    qps = world * B / (ms_max * 1e-3)
    line = {
        "metric": METRIC,
        "value": round(qps, 1),
        "unit": "queries/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e2m1/e4m3/e8m0 storage; fp32 scores; bf16 attention with fp32 accumulate",
        "data": "synthetic N(0,1) caches drawn on the device, packed by the library",
        "config": step_config(wl, B, res["N"], L, res["K"], res["W"], world),
        "launch": "CUDA graph of the step (programmatic dependent launches)" if res["graph"] else "eager",
        "ms_per_step_eager": round(res["eager_ms"], 5),
        "stages_ms": dict([(nm, round(v, 5)) for nm, v in res["stage_ms"].items()] +
                          [("index_score_alone", round(res["scan_ms"], 5))]),
        "entries_scored_per_s": main_sum["entries_scored_per_s"],
        "indexer_scan_gbs": scan_gbs,
        "roofline": {"kernel": "index_score", "bound": "hbm", "achieved": scan_gbs,
                     "peak": hbm_peak, "peak_kind": f"{peak_kind} HBM copy bandwidth", "unit": "GB/s",
                     "frac": main_sum["scan_roofline"]["frac"], "traffic": traffic,
                     "algorithmic_bytes_per_launch": scan_bytes},
        "kernel_rooflines": {
            "sparse_attn": {"bound": "hbm", "achieved": main_sum["attention"]["achieved_gbs"], "peak": hbm_peak,
                            "unit": "GB/s", "frac": main_sum["attention"]["frac"],
                            "algorithmic_bytes_per_step": main_sum["attention"]["algorithmic_bytes_per_step"]},
            "kv_append": {"bound": "hbm", "achieved": round(app["bulk_bytes"] / (app["bulk_ms"] * 1e-3) / 1e9, 1),
                          "peak": hbm_peak, "unit": "GB/s",
                          "frac": round(app["bulk_bytes"] / (app["bulk_ms"] * 1e-3) / 1e9 / hbm_peak, 4),
                          "algorithmic_bytes_per_launch": app["bulk_bytes"], "entries_per_launch": app["entries"],
                          "decode_append_us": round(app["decode_us"], 2),
                          "note": "timed alone, outside the step: bf16 latent + key in, 356 B entry out"}},
        "e2e": {"value": main_sum["e2e"]["value"], "unit": "queries/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "ms_per_step": round(res["e2e_ms"], 5), "host_enqueue_ms_per_step": round(res["host_ms"], 5),
                "note": "one host-to-device copy of the step's inputs and one device-to-host copy of its outputs "
                        "(each a packed buffer), on their own streams, overlapping neighbouring steps (two buffer "
                        "sets); inputs exceed L2"},
        "gpu_launches": args.steps * res["n_launches"],
        "clocks": res["clocks"],
    }
    workloads = {str(wid): main_sum}
    workloads.update(extra)
    if pre is not None:
        bf16_peak, bf16_kind = tensor_peak_tflops()
        fp4_peak = bf16_peak * FP4_PER_BF16
        sc_tf = pre["scan_flops"] / (pre["scan_ms"] * 1e-3) / 1e12
        at_tf = pre["attn_flops"] / (pre["attn_ms"] * 1e-3) / 1e12
        rp_tf = pre["attn_flops"] / (pre["replay_ms"] * 1e-3) / 1e12
        line["kernel_rooflines"]["prefill_index_score"] = {
            "bound": "tensor", "achieved": round(sc_tf, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
            "frac": round(sc_tf / fp4_peak, 4), "ms": round(pre["scan_ms"], 4), "pairs": pre["pairs"],
            "peak_kind": f"{bf16_kind} bf16 x {FP4_PER_BF16:g} (nominal FP4:BF16)",
            "note": "4,096 queries at 126,976.., causal; 2 x 4,096 FLOP per (query, entry) pair"}
        cs_tf = pre["cscan_flops"] / (pre["cscan_ms"] * 1e-3) / 1e12
        line["kernel_rooflines"]["prefill_index_score_compressed_m2"] = {
            "bound": "tensor", "achieved": round(cs_tf, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
            "frac": round(cs_tf / fp4_peak, 4), "ms": round(pre["cscan_ms"], 4), "pairs": pre["cpairs"],
            "peak_kind": f"{bf16_kind} bf16 x {FP4_PER_BF16:g} (nominal FP4:BF16)",
            "note": "encoder Full layer: 4,096 queries at token 253,952.. over complete 2-token entries"}
        cmp_gbs = pre["cmp_bytes"] / (pre["cmp_ms"] * 1e-3) / 1e9
        line["kernel_rooflines"]["compress_kv_m2"] = {
            "bound": "hbm", "achieved": round(cmp_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(cmp_gbs / hbm_peak, 4), "ms": round(pre["cmp_ms"], 4),
            "algorithmic_bytes_per_launch": pre["cmp_bytes"], "entries_per_launch": pre["cmp_entries"],
            "note": f"{2 * pre['cmp_entries']:,} tokens of C and Z (bf16) in, {pre['cmp_entries']:,} packed "
                    "288-byte entries out"}
        line["kernel_rooflines"]["prefill_attention"] = {
            "bound": "tensor", "achieved": round(at_tf, 1), "peak": round(bf16_peak, 1), "unit": "TFLOP/s",
            "frac": round(at_tf / bf16_peak, 4), "ms": round(pre["attn_ms"], 4),
            "peak_kind": f"{bf16_kind} bf16",
            "note": "4,096 queries x (512 selected + 128 SWA rows); QK + PV FLOPs"}
        line["kernel_rooflines"]["prefill_attention_replay"] = {
            "bound": "tensor", "achieved": round(rp_tf, 1), "peak": round(bf16_peak, 1), "unit": "TFLOP/s",
            "frac": round(rp_tf / bf16_peak, 4), "ms": round(pre["replay_ms"], 4),
            "peak_kind": f"{bf16_kind} bf16",
            "note": "as prefill_attention with the Bounded-Replay cut at swa row 64 (FLOPs counted over 640 rows)"}
        workloads["3"] = {
            "workload": (WORKLOADS[3].name if (pre["T"], pre["N"] - pre["T"]) == (PREFILL_T, PREFILL_P0)
                         else f"prefill_t{pre['T']}_after_{pre['N'] - pre['T']}"),
            "queries": pre["T"], "visible_entries_max": pre["N"],
            "queries_per_s": round(pre["T"] / (pre["pipeline_ms"] * 1e-3), 1),
            "ms_per_step": round(pre["pipeline_ms"], 4),
            "stages_ms": {k_: round(v, 4) for k_, v in pre["stages_ms"].items()},
            "scan_roofline": {"bound": "tensor", "achieved": round(sc_tf, 1), "peak": round(fp4_peak, 1),
                              "unit": "TFLOP/s", "frac": round(sc_tf / fp4_peak, 4)},
            "steps": pre["steps"],
            "note": "one step = q -> MXFP4, causal scan, Top-512 per query (n_valid = position + 1), sparse "
                    "attention over 512 selected + the 128-row causal SWA window; eager, L2 flushed before "
                    "each step"}
    line["workloads"] = workloads
    if not args.no_cpu_baseline and wid == WORKLOAD_ID:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget)
    if world > 1:
        torch.distributed.destroy_process_group()
    return line


APPEND_ENTRIES = 131072            # bulk append: entries per launch, over the batch
APPEND_BYTES_PER_ENTRY = 512 * 2 + 128 * 2 + KV_BYTES_PER_ENTRY + IK_BYTES_PER_ENTRY   # bf16 in, packed out


PREFILL_T, PREFILL_P0, PREFILL_REPLAY_ROW = 4096, 126976, 64


def measure_prefill(csa2, ctx, steps, T=None, p0=None):
    """The prefill workload (4,096 queries at positions 126,976 .. 131,071 of
    one sequence) as a pipeline, eager, with an event between stages: indexer
    q -> MXFP4, the causal indexer scan (4,096 MAC per query-entry pair, FP4
    tensor cores), the Top-512 of each query's visible prefix, and the sparse
    attention over the 512 selected + the 128-row SWA window (QK and PV on
    bf16 tensor cores). Beside it, timed alone: the attention with the
    Bounded-Replay cut, the indexer scan of an encoder Full layer over 2-token
    compressed entries, and the compressor."""
    torch, device, stream = ctx.torch, ctx.device, ctx.stream
    from fp4_kv_cache_02_gb300.inputs import device_normal, device_uniform
    T = PREFILL_T if T is None else T
    p0 = PREFILL_P0 if p0 is None else p0
    W, K = 128, 512
    N = p0 + T
    q_bf = device_normal((T, 32, 128), 71, device)
    q_data = torch.empty(T, 32, 64, dtype=torch.uint8, device=device)
    q_sc = torch.empty(T, 32, 4, dtype=torch.uint8, device=device)
    w = device_uniform((T, 32), 72, device).float().contiguous()
    ik_data, ik_sc = csa2.quant_mxfp4(device_normal((N, 128), 73, device))
    scores = torch.empty(T, N, dtype=torch.float32, device=device)
    kv_data, kv_sc = csa2.pack_kv_fp4(device_normal((N, 512), 74, device))
    Q = device_normal((T, 64, 512), 75, device, scale=1.0 / math.sqrt(512))
    swa = csa2.pack_fp8(device_normal((T + W - 1, 512), 76, device))
    n_valid = torch.arange(p0 + 1, p0 + T + 1, dtype=torch.int32, device=device)
    idx = torch.empty(T, K, dtype=torch.int32, device=device)
    tws = csa2.topk_workspace(T, N, K, device=device)
    out = torch.empty(T, 64, 512, dtype=torch.bfloat16, device=device)
    aws = csa2.attn_workspace(T, K, W, device=device)

    stages = [
        ("quant_q", lambda: csa2.csa2_quant_mxfp4(q_bf, q_data, q_sc, stream=stream)),
        ("index_score", lambda: csa2.csa2_prefill_index_score(q_data, q_sc, w, ik_data, ik_sc, p0, scores,
                                                              stream=stream)),
        ("topk", lambda: csa2.csa2_topk(scores, K, idx, tws, n_valid=n_valid, stream=stream)),
        ("sparse_attn", lambda: csa2.csa2_sparse_attn_prefill(Q, kv_data, kv_sc, idx, swa, W, out, aws,
                                                              stream=stream)),
    ]
    nst = len(stages)
    for _ in range(2):
        ctx.flush_l2()
        for _, fn in stages:
            fn()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(steps)]
    for i in range(steps):
        ctx.flush_l2()
        for j, (_, fn) in enumerate(stages):
            evs[i][j].record(stream)
            fn()
        evs[i][nst].record(stream)
    torch.cuda.synchronize()
    assert csa2.csa2_get_last_error() == 0
    stage_ms = {nm: sum(e[j].elapsed_time(e[j + 1]) for e in evs) / steps for j, (nm, _) in enumerate(stages)}
    pipeline_ms = sum(e[0].elapsed_time(e[nst]) for e in evs) / steps
    del tws

    replay = lambda: csa2.csa2_sparse_attn_prefill_replay(Q, kv_data, kv_sc, idx, swa, W, PREFILL_REPLAY_ROW, out,
                                                          aws, stream=stream)
    # encoder Full layer at m = 2: the same 4,096 queries at token positions
    # 253,952 .. see the complete compressed entries (126,976 .. 129,024 of them)
    m, tok0 = 2, 2 * p0
    cscan = lambda: csa2.csa2_prefill_index_score_compressed(q_data, q_sc, w, ik_data, ik_sc, tok0, m, scores,
                                                               stream=stream)
    ctx.timed(replay, 2)
    replay_ms = ctx.timed(replay, steps)
    ctx.timed(cscan, 2)
    cscan_ms = ctx.timed(cscan, steps)
    del scores
    # the compressor: 2 N tokens of C and Z (bf16) into the N packed entries of
    # the planes above (262,144 tokens into 131,072 entries at the default shape)
    n_tok = 2 * N
    C = device_normal((n_tok, 512), 78, device)
    Z = device_normal((n_tok, 512), 79, device)
    bias = device_normal((m, 512), 80, device).float().contiguous()
    cmp = lambda: csa2.csa2_compress_kv(C, Z, bias, m, kv_data, kv_sc, stream=stream)
    ctx.timed(cmp, 2)
    cmp_ms = ctx.timed(cmp, steps)
    torch.cuda.synchronize()
    assert csa2.csa2_get_last_error() == 0
    pairs = T * p0 + T * (T + 1) // 2
    cpairs = sum((tok0 + t + 1) // m for t in range(T))
    return {"T": T, "N": N, "steps": steps, "pipeline_ms": pipeline_ms, "stages_ms": stage_ms,
            "scan_ms": stage_ms["index_score"], "scan_flops": 2 * 4096 * pairs, "pairs": pairs,
            "attn_ms": stage_ms["sparse_attn"], "attn_flops": 2 * 2 * T * 64 * (K + W) * 512,
            "replay_ms": replay_ms,
            "cscan_ms": cscan_ms, "cscan_flops": 2 * 4096 * cpairs, "cpairs": cpairs,
            "cmp_ms": cmp_ms, "cmp_bytes": n_tok * 2 * 512 * 2 + (n_tok // m) * KV_BYTES_PER_ENTRY,
            "cmp_entries": n_tok // m}


def measure_append(csa2, torch, B, device, steps, flush_l2, stream):
    """csa2_kv_append timed alone: (1) a bulk append of APPEND_ENTRIES new
    entries spread over the B sequences into empty planes (inputs larger than
    L2, flushed between launches), against the HBM roofline; (2) the decode
    case, one entry per sequence, as a latency."""
    from fp4_kv_cache_02_gb300.inputs import device_normal
    T = APPEND_ENTRIES // B
    kv = device_normal((B, T, 512), 91, device)
    ik = device_normal((B, T, 128), 92, device)
    planes = [torch.empty(B, T, w, dtype=torch.uint8, device=device) for w in (256, 32, 64, 4)]
    nv0 = torch.zeros(B, dtype=torch.int32, device=device)
    nv1 = torch.empty_like(nv0)

    def timed(kv_, ik_, n):
        tot = 0.0
        for _ in range(n):
            flush_l2()
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            csa2.csa2_kv_append(kv_, ik_, *planes, nv0, n_visible_out=nv1, stream=stream)
            b_.record(stream)
            b_.synchronize()
            tot += a.elapsed_time(b_)
        return tot / n

    timed(kv, ik, 3)
    bulk_ms = timed(kv, ik, steps)
    one_kv, one_ik = kv[:, :1].contiguous(), ik[:, :1].contiguous()
    timed(one_kv, one_ik, 3)
    decode_ms = timed(one_kv, one_ik, steps)
    torch.cuda.synchronize()
    assert csa2.csa2_get_last_error() == 0
    nbytes = B * T * APPEND_BYTES_PER_ENTRY
    return {"bulk_ms": bulk_ms, "bulk_bytes": nbytes, "entries": B * T, "decode_us": decode_ms * 1e3}


# ---------------------------------------------------------------------------- CPU oracle

def oracle_sample(n_seq: int, N: int):
    """Host caches of `n_seq` sequences of the workload, quantised by the oracle."""
    import numpy as np

    import oracle
    from fp4_kv_cache_02_gb300.inputs import decode_sequence
    try:
        import torch
        gen_dev = "cuda" if torch.cuda.is_available() else None
    except ImportError:
        gen_dev = None
    qd = np.zeros((n_seq, 32, 64), np.uint8)
    qs = np.zeros((n_seq, 32, 4), np.uint8)
    w = np.zeros((n_seq, 32), np.float32)
    ikd = np.zeros((n_seq, N, 64), np.uint8)
    iks = np.zeros((n_seq, N, 4), np.uint8)
    kvd = np.zeros((n_seq, N, 256), np.uint8)
    kvs = np.zeros((n_seq, N, 32), np.uint8)
    Q = np.zeros((n_seq, 1, 64, 512), np.float32)
    swa = np.zeros((n_seq, 1, 128, 512), np.uint8)
    for b in range(n_seq):
        d = decode_sequence(WORKLOAD_ID, b, N, device=gen_dev)
        qd[b], qs[b] = oracle.quant_mxfp4(d["q_idx"])
        w[b] = d["w"]
        ikd[b], iks[b] = oracle.quant_mxfp4(d["ik"])
        kvd[b], kvs[b] = oracle.pack_kv_fp4(d["kv"])
        Q[b] = d["Q"]
        swa[b] = oracle.pack_fp8(d["swa"].reshape(-1)).reshape(1, 128, 512)
    return dict(n_visible=np.full(n_seq, N, np.int32), qd=qd, qs=qs, w=w, ikd=ikd, iks=iks, kvd=kvd, kvs=kvs, Q=Q,
                swa=swa)


def oracle_time(sample, threads: int, reps: int = 1) -> float:
    import oracle
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.decode_batch(sample["n_visible"], sample["qd"], sample["qs"], sample["w"], sample["ikd"],
                            sample["iks"], sample["kvd"], sample["kvs"], sample["Q"], sample["swa"], k=512,
                            n_threads=threads)
    return time.perf_counter() - t0


def cpu_baseline(budget_s: float = 20.0):
    import oracle
    from fp4_kv_cache_02_gb300.inputs import WORKLOADS
    N = WORKLOADS[WORKLOAD_ID].N
    cores = oracle.max_threads()
    n_seq = max(1, cores)
    sample = oracle_sample(n_seq, N)
    t = oracle_time(sample, cores)
    reps = max(1, int(budget_s / max(t, 1e-3)) - 1)
    t = oracle_time(sample, cores, reps) / reps
    return {"value": round(n_seq / t, 3), "unit": "queries/s", "cores": cores, "kind": "oracle",
            "sample": f"{n_seq} sequences x {N} entries of the Full-layer decode workload "
                      f"(score + Top-512 + attention), {reps} repetitions, OpenMP over sequences"}


def run_reference(args):
    """The reference arm: the CPU oracle, timed on the host cores."""
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    from fp4_kv_cache_02_gb300.inputs import WORKLOADS
    oracle.build()
    N = WORKLOADS[WORKLOAD_ID].N
    cores = oracle.max_threads()
    total_budget = 150.0
    per_step = total_budget / max(1, args.steps + args.warmup)
    probe = oracle_sample(1, N)
    t1 = oracle_time(probe, cores)
    n_seq = int(max(1, min(cores, per_step / max(t1, 1e-3))))
    sample = oracle_sample(n_seq, N) if n_seq > 1 else probe
    for _ in range(args.warmup):
        oracle_time(sample, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_time(sample, cores)
    ms = (time.perf_counter() - t0) / args.steps * 1e3
    qps = n_seq / (ms * 1e-3)
    return {
        "impl": "reference", "metric": METRIC, "value": round(qps, 3), "unit": "queries/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 accumulate (oracle)", "data": "synthetic",
        "config": step_config(WORKLOADS[WORKLOAD_ID], WORKLOADS[WORKLOAD_ID].B, N, WORKLOADS[WORKLOAD_ID].L, 512,
                              128, world),
        "cpu_baseline": {"value": round(qps, 3), "unit": "queries/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n_seq} sequence(s) x {N} entries per step"},
        "e2e": {"value": round(qps, 3), "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches instead of a CUDA graph of the step")
    ap.add_argument("--prefill-shape", default=f"{PREFILL_T},{PREFILL_P0}",
                    help="T,P0 of the prefill workload: T queries at positions P0 .. P0+T-1 (profiling a smaller case)")
    ap.add_argument("--no-prefill", dest="prefill", action="store_false",
                    help="skip the prefill scan and attention timings reported beside the decode step")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--batch", type=int, default=0, help="sequences per GPU (default: the workload's)")
    ap.add_argument("--workload", type=int, default=WORKLOAD_ID, choices=[0, 1, 2, 4],
                    help="decode workload of the headline value (default 1: 32 sequences x 65,536 entries)")
    ap.add_argument("--workloads", default="0,2,3,4",
                    help="comma-separated workloads also measured into the line's `workloads` object ('' for none)")
    args = ap.parse_args(argv)
    args.workloads = [int(x) for x in args.workloads.split(",") if x.strip()]
    args.prefill_shape = tuple(int(x) for x in args.prefill_shape.split(","))
    if 3 not in args.workloads:
        args.prefill = False
    args.warmup = max(args.warmup, 3)  # at least 3 untimed warm-up steps
    line = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
