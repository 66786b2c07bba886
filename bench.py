"""Benchmark of the paged-KV decode step of a looped transformer on GB300.

One step = one decode token for every request of the batch through every
(layer, plane) bank of the model: for each bank, append this step's K/V rows and
run paged decode attention over them (by default one call does both:
rlt_paged_decode_attn / _prefix with k_new, v_new; --append plain times
rlt_kv_append as its own launch);
workloads whose model draws latent noise (Huginn-shaped) also initialise the new
tokens' latent state (rlt_latent_noise_init).  All inputs are seeded and
synthetic; every bank's KV lives in its own region of HBM.

Prints ONE JSON line.  `value` is the step's algorithmic HBM bytes (unique pages
counted once) divided by the device time of a step, in GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ouro] [--impl reference]
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attn: achieved HBM GB/s (% of GB300 peak), µs per layer-plane step"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0
L2_BYTES = 129 * 2**20


# ------------------------------------------------------------------ bytes

def attn_bytes(case: W.PagedCase, unique: bool = True) -> int:
    """Algorithmic bytes of one paged decode attention call over one bank."""
    tokens = case.unique_tokens() if unique else case.kv_tokens()
    kv = tokens * case.num_kv_heads * case.head_dim * 2 * 2
    qo = case.batch * case.num_q_heads * case.head_dim * 2 * 2
    meta = sum(case.pages_of(b) for b in range(case.batch)) * 4 + case.batch * 4
    return kv + qo + meta


def append_bytes(case: W.PagedCase) -> int:
    n = int((case.new_slots >= 0).sum())
    return n * case.num_kv_heads * case.head_dim * 2 * 2 * 2 + case.batch * 8


def fused_append_bytes(case: W.PagedCase) -> int:
    """The append's bytes when the attention call does it: new rows read, pool rows written
    (no slot list: the slot comes from the page table the call reads anyway)."""
    return append_bytes(case) - case.batch * 8


def noise_bytes(case: W.PagedCase) -> int:
    nz = case.noise
    return 0 if nz is None else nz.rows * 16 + nz.rows * nz.channels * 4


def layer_planes(case: W.PagedCase):
    rec = np.asarray(case.recurrent, np.uint8)
    return [(l, t) for t in range(case.num_planes) for l in range(case.num_layers) if t == 0 or rec[l]]


def extend_roofline(case: W.PagedCase, new_lens, ms: float) -> dict:
    """Roofline of one causal extend call: its bound is the one its arithmetic intensity selects.

    flops: QK^T and PV over each new token's causal keys (4 * D * Hq per (token, key) pair);
    bytes: the K/V rows read once per kv head (unique pages, as decode counts them), the new
    tokens' q and out rows, the page-table entries.  Below the ridge (measured bf16 peak / measured
    HBM peak, ~284 flop/B) the call is HBM-bound, above it tensor-bound."""
    D, Hq = case.head_dim, case.num_q_heads
    keys = sum(int(L) - int(n) + i + 1 for L, n in zip(case.seq_lens, new_lens) for i in range(int(n)))
    flops = 4.0 * D * Hq * keys
    rows = int(np.sum(new_lens))
    nbytes = attn_bytes(case) - case.batch * Hq * D * 4 + rows * Hq * D * 4
    hbm, _ = hbm_peak()
    ridge = bf16_peak() * 1e12 / (hbm * 1e9)
    t = ms * 1e-3
    intensity = flops / nbytes
    tensor = intensity >= ridge
    achieved = flops / t / 1e12 if tensor else nbytes / t / 1e9
    peak = bf16_peak() if tensor else hbm
    return {"new_tokens_per_request": int(np.max(new_lens)) if len(new_lens) else 0,
            "us_per_call": round(ms * 1e3, 2), "flop_per_byte": round(intensity, 1), "ridge_flop_per_byte": round(ridge, 1),
            "bound": "tensor" if tensor else "hbm", "achieved": round(achieved, 1),
            "unit": "TFLOP/s" if tensor else "GB/s", "peak": peak, "frac": round(achieved / peak, 4),
            "tflops": round(flops / t / 1e12, 1), "gbs": round(nbytes / t / 1e9, 1)}


# --------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[4:8]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for_smi(torch, dev) -> str:
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if uuid:
            return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    return vis.split(",")[dev.index or 0] if vis else str(dev.index or 0)


# ------------------------------------------------------------ peaks etc.

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak() -> float:
    """Measured dense bf16 TFLOP/s of the GB300s (burst), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return 1900.0


def profiled_traffic(workload: str, fused: bool):
    """DRAM bytes of one attention call (all its kernels) from the committed ncu summary
    profiles/traffic_<workload>.txt, if it was taken on the kernels' current sources and
    with the append in the same form (fused into the call or not)."""
    import hashlib
    try:
        text = open(os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")).read()
    except OSError:
        return None
    lines = {k.strip(): v.strip() for k, v in (l.split(":", 1) for l in text.splitlines() if ":" in l)}
    srcs = lines.get("sources", "").split()
    if not srcs:
        return None
    blob = b"".join(open(os.path.join(ROOT, "paged_kv_looped_gb300", "csrc", f), "rb").read() for f in srcs)
    if lines.get("sources_sha256_16") != hashlib.sha256(blob).hexdigest()[:16] or lines.get("workload") != workload:
        return None
    if (lines.get("append", "plain") == "fused") != fused:
        return None
    try:
        return float(lines["dram_bytes_per_call"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------ GPU arm

def auto_chunk_tiles(rlt, case, tails, num_sms):
    """Tiles per work item of the persistent tensor-core kernel: the library's choice for this
    batch (rlt_choose_chunk_tiles: with private tails the chunk whose contiguous item split has
    the least-loaded busiest CTA, otherwise at least 16 items per CTA)."""
    return rlt.rlt_choose_chunk_tiles(case.page_table, case.seq_lens, case.page_size, case.group, tails,
                                      case.num_kv_heads, num_sms)


def run_gpu(args, rank, world):
    import torch

    import paged_kv_looped_gb300 as rlt
    from paged_kv_looped_gb300 import build as rlt_build
    rlt_build.build()

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    case = W.config(args.workload)
    if args.batch:      # the first N requests alone, on a compact pool (small case for profilers)
        case = W.subcase(case, range(min(args.batch, case.batch)))
    lp = layer_planes(case)
    bmap, nbanks = rlt.rlt_bank_map(case.recurrent, case.num_planes)
    assert nbanks == len(lp)
    if args.banks:
        lp = lp[: args.banks]
        nbanks = len(lp)
        bmap = np.where(bmap < nbanks, bmap, -1)
    assert rlt.rlt_validate_batch(case.page_table, case.seq_lens, case.new_slots, case.num_pages,
                                  case.page_size) == 0

    # resident state: one pool region per bank, page table, lengths
    kpool, vpool = W.device_pool(case, nbanks, dev)
    pool = rlt.KVPool(kpool, vpool)
    rng = np.random.default_rng(case.seed + 77)
    B, Hq, Hkv, D = case.batch, case.num_q_heads, case.num_kv_heads, case.head_dim
    def bf(shape):
        return torch.from_numpy(W.bf16_normal(rng, shape).view(np.int16)).view(torch.bfloat16)
    q_h = bf((nbanks, B, Hq, D)).pin_memory()
    kn_h = bf((nbanks, B, Hkv, D)).pin_memory()
    vn_h = bf((nbanks, B, Hkv, D)).pin_memory()
    loc_h = torch.from_numpy(case.new_slots.copy()).pin_memory()
    pt_h = torch.from_numpy(case.page_table.copy()).pin_memory()
    sl_h = torch.from_numpy(case.seq_lens.astype(np.int32)).pin_memory()
    q, kn, vn = q_h.to(dev), kn_h.to(dev), vn_h.to(dev)
    loc, pt, sl = loc_h.to(dev), pt_h.to(dev), sl_h.to(dev)
    out = torch.empty((nbanks, B, Hq, D), dtype=torch.bfloat16, device=dev)
    out_h = torch.empty_like(out, device="cpu").pin_memory()
    # shared-prefix plan (the scheduler's radix tree, recovered from the page tables)
    plan = None
    # every token on tensor cores once a kv head serves >= 8 query heads; below that the
    # private rest goes to the split-K kernel, run beside the tensor-core kernel
    tails = args.tails == "on" or (args.tails == "auto" and case.group >= 8)
    if args.cascade != "off":
        shared = rlt.rlt_plan_prefix(case.page_table, case.seq_lens, case.page_size, 1, False, case.group)
        if shared.num_segments > 0 or args.cascade == "on":
            if args.chunk_tiles == 0:
                args.chunk_tiles = auto_chunk_tiles(rlt, case, tails,
                                                    torch.cuda.get_device_properties(dev).multi_processor_count)
            plan = rlt.rlt_plan_prefix(case.page_table, case.seq_lens, case.page_size, args.chunk_tiles, tails,
                                       case.group)
            if plan.num_segments == 0:
                plan = None
            else:
                plan.to(dev)
    if plan is not None:
        ws_bytes = rlt.rlt_paged_decode_prefix_workspace_size(B, Hq, Hkv, D, plan.max_rest_len,
                                                              plan.max_prefix_slots, args.split_tokens)
        plan_h = [torch.from_numpy(np.ascontiguousarray(a, np.int32).reshape(-1)).pin_memory()
                  for a in (plan.segments, plan.members, plan.member_limit, plan.request_prefix)]
    else:
        ws_bytes = rlt.rlt_paged_decode_workspace_size(B, Hq, Hkv, D, case.max_seq_len, args.split_tokens)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    nz = case.noise
    if nz is not None:
        seeds_h = torch.from_numpy(nz.seeds.view(np.int64).copy()).pin_memory()
        pos_h = torch.from_numpy(nz.positions.copy()).pin_memory()
        seeds, pos = seeds_h.to(dev), pos_h.to(dev)
        noise = torch.empty((nz.rows, nz.channels), dtype=torch.float32, device=dev)
        noise_h = torch.empty_like(noise, device="cpu").pin_memory()
    stream = torch.cuda.current_stream(dev)
    banks = [int(bmap[l, t]) for (l, t) in lp]
    # fused RoPE append: each new token at its sequence position (the last of its request)
    new_pos = torch.from_numpy(np.maximum(case.seq_lens.astype(np.int64) - 1, 0)).to(dev)
    req_ids = torch.arange(B, dtype=torch.int32, device=dev)
    written = torch.zeros((nbanks, B), dtype=torch.int32, device=dev)
    # early start (programmatic dependent launch of each call behind the kernel ahead of it) is
    # valid when nothing ahead of a call writes its bank: the append fused into the call
    early = args.early_start == "on" and args.append == "fused"


    def step(st, events=None):
        """One decode step; with ``events`` (one pair per bank), each attention call is bracketed."""
        if nz is not None:
            rlt.rlt_latent_noise_init(seeds, pos, nz.channels, nz.initializer_range, out=noise, stream=st)
        for i, bank in enumerate(banks):
            if args.append == "rope":
                rlt.rlt_kv_append_rope(pool, bank, kn[i], vn[i], new_pos, loc, case.head_dim, 10000.0,
                                       request=req_ids, written=written, stream=st)
            elif args.append == "plain":
                rlt.rlt_kv_append(pool, bank, kn[i], vn[i], loc, stream=st)
            if events is not None:
                events[i][0].record(st)
            attend(i, bank, st)
            if events is not None:
                events[i][1].record(st)

    def attend(i, bank, st):
        """One bank's attention call (with the append fused into it under --append fused)."""
        fused = {"k_new": kn[i], "v_new": vn[i]} if args.append == "fused" else {}
        if plan is not None:
            rlt.rlt_paged_decode_attn_prefix(pool, bank, q[i], pt, sl, case.max_seq_len, plan, out=out[i],
                                             workspace=ws, split_tokens=args.split_tokens,
                                             max_ctas=args.prefix_ctas, stream=st, early_start=early, **fused)
        else:
            rlt.rlt_paged_decode_attn(pool, bank, q[i], pt, sl, case.max_seq_len, out=out[i], workspace=ws,
                                      split_tokens=args.split_tokens, stream=st, early_start=early, **fused)

    def attention_only(st):
        """Every bank's attention call and nothing else (for the per-call roofline timing)."""
        for i, bank in enumerate(banks):
            attend(i, bank, st)

    def new_events(external):
        kw = {"external": True} if external else {}
        return [(torch.cuda.Event(enable_timing=True, **kw), torch.cuda.Event(enable_timing=True, **kw))
                for _ in banks]

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step(stream)
    assert rlt.rlt_get_device_error() == 0

    # the whole step as one CUDA-graph submission (every call is stream-capturable); a graph of
    # the attention calls alone gives the roofline's per-call time, and a capture bracketing each
    # attention call with event-record nodes gives each call's time on its own (reported beside it)
    graph = timed_graph = graph_events = attn_graph = None
    if args.graph == "on":
        def capture(events=None, fn=None):
            side = torch.cuda.Stream(dev)
            side.wait_stream(stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                if fn is None:
                    step(side, events)
                else:
                    fn(side)
            stream.wait_stream(side)
            return g
        graph = capture()
        attn_graph = capture(fn=attention_only)
        try:
            graph_events = new_events(external=True)
            timed_graph = capture(graph_events)
        except TypeError:              # a torch without graph-recordable events: time eager calls
            graph_events = timed_graph = None
        for _ in range(args.warmup):
            graph.replay()
        assert rlt.rlt_get_device_error() == 0

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            step(stream)

    # ---- timed region: inputs resident in HBM; each bank's KV (> L2) is read once per step
    gpu_id = gpu_id_for_smi(torch, dev)
    with ClockSampler(gpu_id) as clocks:
        barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            run_step()
        t1.record(stream)
        barrier()
        # the attention calls alone, back to back in one graph as the step submits them: events
        # around the replays, the average call = elapsed / calls
        attn_call_ms = None
        if attn_graph is not None:
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(args.steps):
                attn_graph.replay()
            a1.record(stream)
            torch.cuda.synchronize(dev)
            attn_call_ms = a0.elapsed_time(a1) / (args.steps * len(banks))
        # each attention call on the device, an event pair around it, step by step
        attn_ms = []
        for _ in range(args.steps):
            if timed_graph is not None:
                timed_graph.replay()
                torch.cuda.synchronize(dev)
                attn_ms += [a.elapsed_time(b) for a, b in graph_events]
            else:
                events = new_events(external=False)
                step(stream, events)
                torch.cuda.synchronize(dev)
                attn_ms += [a.elapsed_time(b) for a, b in events]
        barrier()
    ms_total = t0.elapsed_time(t1)
    attn_timing = ("attention-only CUDA graph (every bank's call back to back), events around the replays"
                   if attn_call_ms is not None else "eager event pairs")
    assert rlt.rlt_get_device_error() == 0

    # ---- extend (span) attention, when asked: N new tokens per request attend causally over
    # their request's cached keys (a LOTUS block re-forward / packed prefill chunk), per bank
    extend = None
    if args.extend > 0:
        new = np.minimum(case.seq_lens, args.extend).astype(np.int32)
        eplan = rlt.rlt_plan_extend(case.seq_lens, new, case.page_size, max(1, args.chunk_tiles or 2),
                                    case.group).to(dev)
        qx = torch.randn((int(new.sum()), Hq, D), device=dev).to(torch.bfloat16)
        ox = torch.empty_like(qx)
        wsx = torch.empty(max(16, int(rlt.load().rlt_paged_extend_workspace_size(
            int(new.sum()), Hq, D, max(eplan.max_slots, 1)))), dtype=torch.uint8, device=dev)
        for i, bank in enumerate(banks[: args.warmup]):
            rlt.rlt_paged_extend_attn(pool, bank, qx, pt, eplan, out=ox, workspace=wsx, stream=stream)
        ev = []
        for i, bank in enumerate(banks):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            rlt.rlt_paged_extend_attn(pool, bank, qx, pt, eplan, out=ox, workspace=wsx, stream=stream)
            e1.record(stream)
            ev.append((e0, e1))
        torch.cuda.synchronize(dev)
        assert rlt.rlt_get_device_error() == 0
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        extend = extend_roofline(case, new, ms)

    # ---- the latent-noise kernel alone: a graph of back-to-back launches, events around it
    noise_ms = None
    if nz is not None:
        reps = 20
        for _ in range(3):
            rlt.rlt_latent_noise_init(seeds, pos, nz.channels, nz.initializer_range, out=noise, stream=stream)
        def noise_reps(st):
            for _ in range(reps):
                rlt.rlt_latent_noise_init(seeds, pos, nz.channels, nz.initializer_range, out=noise, stream=st)
        if args.graph == "on":
            ng = capture(fn=noise_reps)
            ng.replay()
        n0, n1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0.record(stream)
        if args.graph == "on":
            ng.replay()
        else:
            noise_reps(stream)
        n1.record(stream)
        torch.cuda.synchronize(dev)
        noise_ms = n0.elapsed_time(n1) / reps

    # ---- end to end: this step's inputs from pinned host memory, outputs back to the host
    def ship_plan(host_bufs, dev_arrays, st):
        """The host plans the step from its page tables, then ships the plan (on stream st)."""
        p2 = rlt.rlt_plan_prefix(case.page_table, case.seq_lens, case.page_size, args.chunk_tiles, tails,
                                 case.group)
        # a captured step stays valid while the plan's shape (grid, slots) is unchanged
        assert graph is None or (p2.num_segments, p2.work_units, p2.max_prefix_slots, p2.max_rest_len) == \
            (plan.num_segments, plan.work_units, plan.max_prefix_slots, plan.max_rest_len)
        for host, arr, devt in zip(host_bufs, (p2.segments, p2.members, p2.member_limit, p2.request_prefix),
                                   dev_arrays):
            host.numpy()[:] = np.ascontiguousarray(arr, np.int32).reshape(-1)
            devt.copy_(host, non_blocking=True)

    # (a) one step after another: copies in, the step, copies out, on one stream
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        if plan is not None:
            torch.cuda.synchronize(dev)     # the pinned plan buffers are rewritten below
            ship_plan(plan_h, plan.dev, stream)
        q.copy_(q_h, non_blocking=True)
        kn.copy_(kn_h, non_blocking=True)
        vn.copy_(vn_h, non_blocking=True)
        loc.copy_(loc_h, non_blocking=True)
        pt.copy_(pt_h, non_blocking=True)
        sl.copy_(sl_h, non_blocking=True)
        if nz is not None:
            seeds.copy_(seeds_h, non_blocking=True)
            pos.copy_(pos_h, non_blocking=True)
        run_step()
        out_h.copy_(out, non_blocking=True)
        if nz is not None:
            noise_h.copy_(noise, non_blocking=True)
    e1.record(stream)
    barrier()
    e2e_serial_ms = e0.elapsed_time(e1)
    e2e_ms, e2e_mode = e2e_serial_ms, "serial"

    # (b) pipelined, as a serving loop runs it: two sets of per-step device buffers, each with
    # its own captured step; while step k computes, one copy stream brings in step k+1's inputs
    # and another takes out step k-1's results.  Every step's copies are inside the timed region.
    if graph is not None:
        import copy as _copy
        set0 = dict(q=q, kn=kn, vn=vn, loc=loc, pt=pt, sl=sl, out=out, plan=plan)
        set1 = {k: torch.empty_like(v) for k, v in set0.items() if k != "plan"}
        if plan is not None:
            set1["plan"] = _copy.copy(plan)
            set1["plan"].dev = tuple(t.clone() for t in plan.dev)
        else:
            set1["plan"] = None
        if nz is not None:
            set0.update(seeds=seeds, pos=pos, noise=noise)
            set1.update(seeds=torch.empty_like(seeds), pos=torch.empty_like(pos), noise=torch.empty_like(noise))
        for k in ("q", "kn", "vn", "loc", "pt", "sl", "seeds", "pos"):
            if k in set1:
                set1[k].copy_(set0[k])
        # the step closure reads these names: bind set 1, capture, bind set 0 back
        q, kn, vn, loc, pt, sl, out, plan = (set1[k] for k in ("q", "kn", "vn", "loc", "pt", "sl", "out", "plan"))
        if nz is not None:
            seeds, pos, noise = set1["seeds"], set1["pos"], set1["noise"]
        graph1 = capture()
        q, kn, vn, loc, pt, sl, out, plan = (set0[k] for k in ("q", "kn", "vn", "loc", "pt", "sl", "out", "plan"))
        if nz is not None:
            seeds, pos, noise = set0["seeds"], set0["pos"], set0["noise"]
        graph1.replay()
        torch.cuda.synchronize(dev)
        assert rlt.rlt_get_device_error() == 0
        sets, graphs = (set0, set1), (graph, graph1)
        out_hs = (out_h, torch.empty_like(out_h).pin_memory())
        noise_hs = (noise_h, torch.empty_like(noise_h).pin_memory()) if nz is not None else None
        plan_hs = (plan_h, [torch.empty_like(t).pin_memory() for t in plan_h]) if plan is not None else None
        in_s, out_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_free = [torch.cuda.Event() for _ in range(2)]
        barrier()
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        p0.record(in_s)
        for k in range(args.steps):
            si = k % 2
            S = sets[si]
            with torch.cuda.stream(in_s):
                if k >= 2:
                    in_s.wait_event(ev_free[si])
                if plan is not None:
                    if k >= 2:
                        ev_free[si].synchronize()     # its pinned plan buffers are rewritten now
                    ship_plan(plan_hs[si], S["plan"].dev, in_s)
                for name, host in (("q", q_h), ("kn", kn_h), ("vn", vn_h), ("loc", loc_h), ("pt", pt_h),
                                   ("sl", sl_h)):
                    S[name].copy_(host, non_blocking=True)
                if nz is not None:
                    S["seeds"].copy_(seeds_h, non_blocking=True)
                    S["pos"].copy_(pos_h, non_blocking=True)
                ev_in[si].record(in_s)
            stream.wait_event(ev_in[si])
            graphs[si].replay()
            ev_done[si].record(stream)
            with torch.cuda.stream(out_s):
                out_s.wait_event(ev_done[si])
                out_hs[si].copy_(S["out"], non_blocking=True)
                if nz is not None:
                    noise_hs[si].copy_(S["noise"], non_blocking=True)
                ev_free[si].record(out_s)
        p1.record(out_s)
        barrier()
        pipe_ms = p0.elapsed_time(p1)
        assert rlt.rlt_get_device_error() == 0
        # the faster schedule is the step's end-to-end time (a host-bound tiny step gains nothing
        # from the extra stream and event calls of the pipelined loop); both are reported
        if pipe_ms < e2e_serial_ms:
            e2e_ms, e2e_mode = pipe_ms, "pipelined"
        pipelined_ms = pipe_ms
    else:
        pipelined_ms = None
    h2d = sum(t.numel() * t.element_size() for t in (q_h, kn_h, vn_h, loc_h, pt_h, sl_h))
    d2h = out_h.numel() * out_h.element_size()
    if nz is not None:
        h2d += seeds_h.numel() * 8 + pos_h.numel() * 8
        d2h += noise_h.numel() * 4
    if plan is not None:
        h2d += sum(t.numel() * 4 for t in plan_h)
        per_lp = 4 if plan.max_rest_len > 0 else 3    # append, tensor-core segments, [split-K], combine
    else:
        per_lp = 3 if ws_bytes > 0 else 2
    if args.append == "fused":
        per_lp -= 1                                   # the append rides in an attention kernel
    combine = ws_bytes > 0
    launches = args.steps * (len(banks) * per_lp + (1 if nz is not None else 0))
    return dict(case=case, banks=banks, cascade=plan is not None, graph=graph is not None, attn_timing=attn_timing,
                extend=extend, noise_ms=noise_ms,
                ms_total=ms_total, attn_ms=attn_ms, attn_call_ms=attn_call_ms, e2e_ms=e2e_ms, h2d=h2d, d2h=d2h,
                e2e_serial_ms=e2e_serial_ms, e2e_mode=e2e_mode, e2e_pipelined_ms=pipelined_ms,
                clocks=clocks.summary(), launches=launches, combine=combine, ws_bytes=ws_bytes)


# ------------------------------------------------------------ CPU oracle

class OracleSample:
    """A bounded sample of the workload for the CPU oracle: k random requests of one
    bank on a compact host pool, generated once; each pass is append + attention."""

    def __init__(self, case: W.PagedCase, k: int, seed: int = 0):
        import oracle
        oracle.build()
        self.oracle = oracle
        rng = np.random.default_rng(seed)
        rows = rng.choice(case.batch, min(k, case.batch), replace=False)
        self.sub = W.subcase(case, rows)
        self.requests = len(rows)
        self.h = W.host_tensors(self.sub, seed=seed + 1)
        self.bytes = attn_bytes(self.sub) + append_bytes(self.sub)
        self.desc = (f"oracle (plain C, fp64, 1 thread): append + paged decode attention of {len(rows)} random "
                     f"requests ({self.sub.kv_tokens()} cached tokens) of one bank of the {case.name} workload; "
                     f"GB/s of the same algorithmic bytes")

    def run(self) -> float:
        """One pass; returns its wall time in seconds."""
        h, sub, o = self.h, self.sub, self.oracle
        kp, vp = h.k_pool.copy(), h.v_pool.copy()
        t = time.perf_counter()
        o.kv_append(kp, vp, h.k_new, h.v_new, sub.new_slots)
        o.decode_attn(h.q, kp, vp, sub.page_table, sub.seq_lens)
        return time.perf_counter() - t


def oracle_sample(case: W.PagedCase, budget_s: float, seed: int = 0):
    """Time the oracle (as it stands, one thread) on a sample of the workload for about
    budget_s of CPU work; returns (GB/s of algorithmic bytes, description, seconds)."""
    s = OracleSample(case, 8, seed)
    spent, passes = 0.0, 0
    while spent < budget_s or passes == 0:
        spent += s.run()
        passes += 1
    return s.bytes * passes / spent / 1e9, s.desc + f"; {passes} passes, {spent:.1f} s", spent


def _oracle_worker(args):
    """One process of the parallel oracle timing: its own sample, timed for budget_s."""
    name, seed, budget_s = args
    s = OracleSample(W.config(name), 8, seed)
    spent, passes = 0.0, 0
    while spent < budget_s or passes == 0:
        spent += s.run()
        passes += 1
    return s.bytes * passes, spent


def oracle_parallel(case: W.PagedCase, procs: int, budget_s: float):
    """The same single-threaded oracle run as `procs` independent processes at once (spawned:
    the parent holds a CUDA context), each on its own sample of the workload for about
    budget_s; returns the summed rate (GB/s) and the process count."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    with ctx.Pool(procs) as pool:
        res = pool.map(_oracle_worker, [(case.name, 1000 + i, budget_s) for i in range(procs)])
    return sum(b / t for b, t in res) / 1e9, procs


def run_reference(args, rank, world):
    """The oracle as it stands on the host cores, on the bench's workload, metric and unit."""
    if rank != 0:
        return None
    case = W.config(args.workload)
    sample = OracleSample(case, 8, seed=1)
    for _ in range(args.warmup):
        sample.run()
    times = [sample.run() for _ in range(args.steps)]
    value = sample.bytes * len(times) / sum(times) / 1e9
    nlp = len(layer_planes(case))
    step_bytes = attn_bytes(case) * nlp + append_bytes(case) * nlp + noise_bytes(case)
    # a timed step is one pass over the sample, not the workload's whole decode step: ms_per_step
    # is what was measured; the whole step's time is an extrapolation, labelled as one
    sample_ms = sum(times) / len(times) * 1e3
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sample_ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(case, args, gpu=False),
        "extrapolation": {"extrapolated": True,
                          "timed_step": f"one pass (append + attention) over {sample.requests} of the workload's "
                                        f"{case.batch} requests in one of its {nlp} layer-plane banks"
                                        + (" (the step's latent-noise draw is not in the sample)"
                                           if noise_bytes(case) else ""),
                          "sample_requests": sample.requests, "sample_bytes": sample.bytes,
                          "full_step_bytes": step_bytes, "scale": round(step_bytes / sample.bytes, 1),
                          "full_step_ms_extrapolated": round(step_bytes / (value * 1e9) * 1e3, 1)},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample.desc + f"; each step one pass, {args.steps} steps, "
                                                 f"{sum(times):.1f} s"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def config_dict(case, args, gpu=True):
    """The workload (both arms) and, for the GPU arm, the launch settings."""
    base = {"workload": f"{case.name}: {case.num_layers} layers x {case.num_planes} planes "
                        f"({len(layer_planes(case))} layer-plane banks), B={case.batch}, Hq={case.num_q_heads}, "
                        f"Hkv={case.num_kv_heads}, head_dim={case.head_dim}, page_size={case.page_size}, "
                        f"L in [{int(case.seq_lens.min())}, {int(case.seq_lens.max())}]",
            "batch": case.batch, "kv_tokens_per_layer_plane": case.kv_tokens(),
            "unique_kv_tokens_per_layer_plane": case.unique_tokens()}
    if not gpu:
        return base
    return {**base,
            "split_tokens": args.split_tokens or "auto",
            "cascade": args.cascade, "chunk_tiles": args.chunk_tiles, "tails": args.tails,
            "prefix_ctas": args.prefix_ctas or "one per SM",
            "banks_run": args.banks or "all", "cuda_graph": args.graph, "append": args.append,
            "early_start": "on" if (args.early_start == "on" and args.append == "fused") else "off",
            "l2": "inputs larger than L2: every bank's KV exceeds the 129 MB L2 and each is read once per step"}


# ------------------------------------------------------------ replicas

def max_over_ranks(times_ms):
    """Each timing's maximum over all ranks of the default process group (any backend)."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return [float(t) for t in times_ms]
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x) for x in times_ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_gbs(step_bytes_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's step time (weak scaling)."""
    return world * step_bytes_per_rank / (ms_max * 1e-3) / 1e9


# ------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="ouro", choices=W.WORKLOADS)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--split-tokens", type=int, default=0)
    ap.add_argument("--cascade", default="auto", choices=["auto", "on", "off"],
                    help="read shared-prefix tiles once (tensor-core cascade) when the page tables share them")
    ap.add_argument("--chunk-tiles", type=int, default=0,
                    help="128-token tiles per work item of the tensor-core kernel (0 = from the plan's size)")
    ap.add_argument("--tails", default="auto", choices=["auto", "on", "off"],
                    help="with a shared prefix, also send each request's unshared tokens through the "
                         "tensor-core kernel (auto: when a kv head serves >= 8 query heads)")
    ap.add_argument("--graph", default="on", choices=["on", "off"],
                    help="submit each decode step as one captured CUDA graph (on) or as eager launches")
    ap.add_argument("--extend", type=int, default=0,
                    help="also time causal extend attention with this many new tokens per request (0: off)")
    ap.add_argument("--append", default="fused", choices=["plain", "fused", "rope"],
                    help="store_kv as its own launch at the given slots (plain), fused into the attention "
                         "call (fused), or with RoPE on the keys and written-prefix counters (rope)")
    ap.add_argument("--early-start", default="on", choices=["on", "off"],
                    help="launch each attention call as a programmatic dependent of the kernel ahead of it "
                         "(RLT_ATTN_EARLY_START; only with the append fused into the call)")
    ap.add_argument("--prefix-ctas", type=int, default=0,
                    help="CTAs of the persistent tensor-core kernel (0 = one per SM)")
    ap.add_argument("--banks", type=int, default=0,
                    help="run only the first N layer-plane banks (small-footprint case for profilers); 0 = all")
    ap.add_argument("--batch", type=int, default=0,
                    help="run only the first N requests of the workload (small case for profilers); 0 = all")
    ap.add_argument("--also", default="auto",
                    help="other workloads timed after the headline one (comma list; auto = every other "
                         "workload unless --batch/--banks slice the run; none = skip)")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle CPU time for cpu_baseline")
    ap.add_argument("--cpu-procs", type=int, default=os.cpu_count() or 1,
                    help="also time the oracle as this many processes at once (cpu_baseline.all_cores; <= 1: skip)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if rank == 0:
            print(json.dumps(line))
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl")
    r = run_gpu(args, rank, world)
    case = r["case"]
    res = summarize(r, args, world)

    cpu = None
    if rank == 0 and args.cpu_budget > 0:
        v, desc, _ = oracle_sample(case, args.cpu_budget)
        cpu = {"value": round(v, 4), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc}
        if args.cpu_procs > 1:
            pv, procs = oracle_parallel(case, args.cpu_procs, args.cpu_budget / 2)
            cpu["all_cores"] = {"value": round(pv, 4), "unit": UNIT, "cores": procs,
                                "sample": f"{procs} processes of the same single-threaded oracle at once, "
                                          f"each on its own 8 random requests for about "
                                          f"{args.cpu_budget / 2:.1f} s; summed rate"}

    # the other workloads, each at full size in the same launch settings, fewer steps: per-call
    # and per-step figures beside the headline (the headline stays the --workload one)
    others = {}
    for name in other_workloads(args):
        import copy
        import gc

        import torch
        del r
        gc.collect()
        torch.cuda.empty_cache()
        a2 = copy.copy(args)
        a2.workload, a2.steps, a2.chunk_tiles, a2.cpu_budget = name, min(args.steps, 10), 0, 0
        r = run_gpu(a2, rank, world)
        others[name] = compact(summarize(r, a2, world), a2, r["case"])

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(res["value"], 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(res["ms_step"], 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 Q/K/V, random page allocation)",
        "config": config_dict(case, args),
        "us_per_layer_plane": res["us_per_layer_plane"],
        "pct_of_peak_hbm": round(100 * res["value"] / world / res["roofline"]["peak"], 2),
        "pct_of_nominal_8tbs": round(100 * res["value"] / world / NOMINAL_HBM_GBS, 2),
        "kv_tokens_per_s": res["kv_tokens_per_s"],
        "roofline": res["roofline"],
        "cpu_baseline": cpu,
        "e2e": res["e2e"],
        "gpu_launches": res["launches"],
        **({"extend_attention": res["extend"]} if res["extend"] else {}),
        **({"noise": res["noise"]} if res["noise"] else {}),
        "clocks": res["clocks"],
        **({"workloads": others} if others else {}),
    }
    print(json.dumps(line))


def other_workloads(args):
    """Workloads timed after the headline one: every other workload in the default run (the
    headline's own launch settings, no profiling slice), none when asked or when slicing."""
    if args.also == "none" or args.batch or args.banks:
        return []
    if args.also == "auto":
        return [w for w in W.WORKLOADS if w != args.workload]
    return [w for w in args.also.split(",") if w and w != args.workload]


def summarize(r, args, world):
    """The figures of one workload's run, times taken as the maximum over ranks."""
    case = r["case"]
    nlp = len(r["banks"])
    step_bytes = attn_bytes(case) * nlp + append_bytes(case) * nlp + noise_bytes(case)
    pipe_total = r["e2e_pipelined_ms"] if r["e2e_pipelined_ms"] is not None else r["e2e_serial_ms"]
    attn_isolated_ms = statistics.mean(r["attn_ms"])
    attn_launch_ms = r["attn_call_ms"] if r["attn_call_ms"] is not None else attn_isolated_ms
    ms_max, e2e_ms_step, e2e_serial_step, e2e_pipe_step, attn_launch_ms, attn_isolated_ms, noise_ms = \
        max_over_ranks([r["ms_total"] / args.steps, r["e2e_ms"] / args.steps, r["e2e_serial_ms"] / args.steps,
                        pipe_total / args.steps, attn_launch_ms, attn_isolated_ms, r["noise_ms"] or 0.0])
    value = job_gbs(step_bytes, world, ms_max)
    e2e_value = job_gbs(step_bytes, world, e2e_ms_step)
    e2e_serial = job_gbs(step_bytes, world, e2e_serial_step)
    e2e_pipe = job_gbs(step_bytes, world, e2e_pipe_step) if r["e2e_pipelined_ms"] is not None else None
    fused = args.append == "fused"
    a_bytes = attn_bytes(case) + (fused_append_bytes(case) if fused else 0)
    peak, peak_kind = hbm_peak()
    achieved = a_bytes / (attn_launch_ms * 1e-3) / 1e9
    traffic = profiled_traffic(case.name, fused)
    roofline = {"bound": "hbm",
                "kernel": ("rlt_paged_decode_attn_prefix (tcgen05 shared-prefix + split-K + combine)"
                           if r["cascade"] else "rlt_paged_decode_attn (split-K partial + combine)")
                          + (", append fused" if fused else ""),
                "achieved": round(achieved, 2),
                "achieved_logical": round((attn_bytes(case, unique=False) + (a_bytes - attn_bytes(case)))
                                          / (attn_launch_ms * 1e-3) / 1e9, 2),
                "peak": peak, "peak_kind": f"{peak_kind} (HBM copy)",
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "frac_logical": round((attn_bytes(case, unique=False) + (a_bytes - attn_bytes(case)))
                                      / (attn_launch_ms * 1e-3) / 1e9 / peak, 4),
                "traffic": traffic,
                "traffic_over_algorithmic": round(traffic / a_bytes, 4) if traffic else None,
                "algorithmic_bytes_per_launch": a_bytes, "launch_us": round(attn_launch_ms * 1e3, 2),
                "timing": r["attn_timing"],
                "launch_us_event_nodes": round(attn_isolated_ms * 1e3, 2)}
    return {"value": value, "ms_step": ms_max, "us_per_layer_plane": round(ms_max * 1e3 / nlp, 2),
            "kv_tokens_per_s": round(world * case.kv_tokens() * nlp / (ms_max * 1e-3), 1),
            "roofline": roofline,
            "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": r["h2d"],
                    "d2h_bytes_per_step": r["d2h"], "mode": r["e2e_mode"],
                    "serial_value": round(e2e_serial, 2),
                    "pipelined_value": round(e2e_pipe, 2) if e2e_pipe is not None else None},
            "extend": r["extend"], "noise": noise_roofline(case, noise_ms) if r["noise_ms"] else None,
            "clocks": r["clocks"], "launches": r["launches"]}


def compact(res, args, case):
    """One other workload's entry: per-call attention, per step, end to end, clocks."""
    rf = res["roofline"]
    return {"config": config_dict(case, args)["workload"], "steps": args.steps,
            "us_per_attention_call": rf["launch_us"], "attention_gbs_unique": rf["achieved"],
            "frac": rf["frac"], "frac_logical": rf["frac_logical"],
            "traffic_over_algorithmic": rf["traffic_over_algorithmic"],
            "attention_kernel": rf["kernel"],
            "step_gbs": round(res["value"], 2), "ms_per_step": round(res["ms_step"], 4),
            "us_per_layer_plane": res["us_per_layer_plane"], "e2e_gbs": res["e2e"]["value"],
            **({"noise": res["noise"]} if res["noise"] else {}), "clocks": res["clocks"]}


def noise_roofline(case: W.PagedCase, ms: float) -> dict:
    """The latent-noise kernel against both of its bounds: the HBM write of 4 bytes per value (plus
    the 16-byte key of each row) and integer issue (instructions per value from the committed ncu
    summary of the current kernel source, else null; peak = SMs x 4 schedulers x 32 lanes x SM clock
    / instructions per value)."""
    nz = case.noise
    values = nz.rows * nz.channels
    nbytes = values * 4 + nz.rows * 16
    t = ms * 1e-3
    hbm, _ = hbm_peak()
    out = {"kernel": "noise_kernel (rlt_latent_noise_init)", "values": values, "us_per_call": round(ms * 1e3, 2),
           "values_per_s": round(values / t, 1), "write_gbs": round(nbytes / t / 1e9, 1),
           "frac_of_hbm_peak": round(nbytes / t / 1e9 / hbm, 4)}
    ipv = profiled_noise_instructions()
    if ipv:
        sms, mhz = sm_count_and_clock()
        peak_vps = sms * 4 * 32 * mhz * 1e6 / ipv
        out["alu"] = {"inst_per_value": ipv, "peak_values_per_s": round(peak_vps, 1),
                      "frac": round(values / t / peak_vps, 4)}
    out["bound"] = "alu" if ipv and values / t / out["alu"]["peak_values_per_s"] > out["frac_of_hbm_peak"] else "hbm"
    return out


def sm_count_and_clock():
    """SMs of the current device and the measured maximum SM clock (MHz) of the GB300s."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f)["sm_max_mhz"])
    except (OSError, KeyError, ValueError):
        mhz = 2070.0
    return sms, mhz


def profiled_noise_instructions():
    """Thread-instructions per value of the noise kernel from profiles/noise_kernel.txt, if that
    summary was taken on the current noise.cu."""
    import hashlib
    try:
        text = open(os.path.join(ROOT, "profiles", "noise_kernel.txt")).read()
    except OSError:
        return None
    f = {k.strip(): v.strip() for k, v in (l.split(":", 1) for l in text.splitlines() if ":" in l)}
    srcs = f.get("sources", "").split()
    if not srcs:
        return None
    blob = b"".join(open(os.path.join(ROOT, "paged_kv_looped_gb300", "csrc", x), "rb").read() for x in srcs)
    if f.get("sources_sha256_16") != hashlib.sha256(blob).hexdigest()[:16]:
        return None
    try:
        return float(f["thread_instructions_per_value"])
    except (KeyError, ValueError):
        return None


if __name__ == "__main__":
    main()
