"""Benchmark: fused RoPE causal attention TFLOP/s and rope_apply GB/s on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one fused RoPE causal attention forward over the long-context GQA
workload (bf16, B=1, 32 q-heads / 8 kv-heads, 16384 new queries after a
4096-row cached prefix, D=128, NeoX, base 5e5): the largest single-GPU
configuration of the attention metric.  The same run also times the
standalone rope_apply_qk on the continuous-batching workload (bf16, 65536
tokens of 256 requests, 32 + 8 heads, D=128, in place) and reports its GB/s,
and the decoder step on the decode workload (512 requests, contexts up to
131072 keys, ~140 GB of cached bf16 K/V): rope_append_kv plus attn_decode,
reported as GB/s of the decode attention (object "decode_step"); the
backward of the long-context workload (object "backward"); and the
configurations small enough to fit in L2, each timed cold (objects "sweep":
the six bf16 GPT-J shapes with their peak extra memory against |O| + |LSE|,
"decode_rope": the decode-batch rope_apply_qk, "fp32_attn": the fp32 case;
"cold_floor": a one-element PyTorch kernel timed the same way, the part of
each of those times that any launch pays).

Timing: W untimed warm-up steps, then K steps, each timed with CUDA events on
the launching stream; L2 is flushed (a 256 MiB write) before every timed
attention step, followed by a ~100 us GPU-side sleep so that the call is
queued before its start event fires (small kernels are then timed on the
device, not behind the host's launch overhead); the rope working set
(1.4 GB) is larger than L2.  A barrier
and a device synchronize bracket the timed region; times are the max over
ranks.  Under torchrun each rank runs an independent replica (the method has
no exchange step), so scaling is weak.

End to end ("e2e"): the same attention through the public API with every
step's q, k, v uploaded from pinned host memory and O, LSE read back, two
buffer sets and two copy streams overlapping the copies with the attention;
"e2e.link" gives one step's upload and download timed alone, so a step
that the host link, not the kernel, bounds is visible as such.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (rows of the attention), same metric and unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "fused RoPE causal attn TFLOPS (% bf16 peak); rope_apply GB/s (% HBM), 1 GB300"
ATTN = wl.LONG_GQA
ROPE = wl.CB_ROPE
DEC = wl.DECODE_ATTN
ATTN_KERNEL_SRC = os.path.join(ROOT, "rope_causal_attention_gb300", "csrc", "attn_tc.cu")
ROPE_KERNEL_SRC = os.path.join(ROOT, "rope_causal_attention_gb300", "csrc", "rope_kernels.cu")
DECODE_KERNEL_SRC = os.path.join(ROOT, "rope_causal_attention_gb300", "csrc", "decode_tc.cu")
BWD_KERNEL_SRC = [os.path.join(ROOT, "rope_causal_attention_gb300", "csrc", f)
                  for f in ("attn_bwd_tc.cu", "attn_bwd_simt.cu")]
PROFILE_JSON = os.path.join(ROOT, "profiles", "counters.json")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def max_over_ranks(value: float) -> float:
    """Max of a per-rank float over all ranks (identity without a process
    group); CUDA tensor under NCCL, CPU tensor under gloo."""
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def src_hash(paths):
    """First 16 hex digits of the SHA-256 of one source file, or of several
    concatenated in order."""
    h = hashlib.sha256()
    for path in [paths] if isinstance(paths, str) else paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def dram_traffic(kernel_key, src):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    try:
        with open(PROFILE_JSON) as f:
            d = json.load(f)[kernel_key]
        if d.get("src_sha256_16") != src_hash(src):
            return None
        return int(d["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during a region."""
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


_CPU_INPUTS = {}


def cpu_oracle_attention(sample_rows: int, seed: int = 0):
    """Times the fp64 oracle on a seeded row sample of the attention workload.
    Returns (TFLOP/s, seconds, threads, description)."""
    import oracle
    oracle.build()
    if "attn" not in _CPU_INPUTS:
        q, k, v = ATTN.inputs()
        _CPU_INPUTS["attn"] = (q.float().numpy(), k.float().numpy(), v.float().numpy())
    qn, kn, vn = _CPU_INPUTS["attn"]
    rng = np.random.default_rng(seed)
    n = ATTN.B * ATTN.Hq * ATTN.Sq
    rows = np.sort(rng.choice(n, size=sample_rows, replace=False))
    i = rows % ATTN.Sq
    flops = float(4.0 * ATTN.D * np.minimum(ATTN.Sk, ATTN.kv_offset + i + 1).sum())
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.attention(qn, kn, vn, kv_offset=ATTN.kv_offset, base=ATTN.base, layout=ATTN.layout,
                     rows=rows, nthreads=threads)
    dt = time.perf_counter() - t0
    desc = (f"{sample_rows} seeded random query rows of {n} (all heads), K rotation of all "
            f"kv heads included; fp64 C oracle, {threads} threads")
    return flops / dt / 1e12, dt, threads, desc


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    sample = args.ref_rows
    vals = []
    for it in range(args.warmup + args.steps):
        tf, dt, threads, desc = cpu_oracle_attention(sample, seed=it)
        if it >= args.warmup:
            vals.append((tf, dt))
    value = statistics.mean(v[0] for v in vals)
    ms = statistics.mean(v[1] for v in vals) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": ATTN.name, "sample": f"{sample} rows per step"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def attn_workload(args):
    if args.attn_workload:
        return next(w for w in wl.ALL_ATTN if w.name == args.attn_workload)
    if args.attn_sq:
        import dataclasses
        return dataclasses.replace(ATTN, Sq=args.attn_sq, Sk=args.attn_sq + ATTN.kv_offset,
                                   name=f"{ATTN.name}__Sq{args.attn_sq}")
    return ATTN


def flush_l2(flush):
    """Overwrite L2 with a buffer larger than it, then hold the stream for
    ~100 us (GPU-side sleep) so that the next call is already queued when its
    start event fires: the events then time the kernel from a cold L2, not
    the host's argument marshalling."""
    flush.zero_()
    torch.cuda._sleep(200_000)


def time_attention(ra, W, args, dev, stream, ws, local, host_e2e=True):
    """Times W warm-up + K steps of the fused attention; returns a dict."""
    q, k, v = W.inputs()
    qg, kg, vg = q.to(dev), k.to(dev), v.to(dev)
    cos, sin = ra.make_tables(max(W.Sk, W.kv_offset + W.Sq), W.r, W.base, device=dev)
    o = torch.empty_like(qg)
    lse = torch.empty(W.B, W.Hq, W.Sq, dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def call():
        ra.attn_fwd_causal_rope(qg, kg, vg, cos, sin, kv_offset=W.kv_offset, layout=W.layout,
                                out=o, lse=lse)

    for _ in range(args.warmup):
        flush_l2(flush)
        call()
    torch.cuda.synchronize()
    if ra.ra_get_device_status() != 0:
        raise RuntimeError("device status error during warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        time.sleep(0.05)  # let the sampler start before the timed region
        t0 = time.perf_counter()
        for s in range(args.steps):
            flush_l2(flush)
            starts[s].record(stream)
            call()
            ends[s].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    if ws > 1:
        torch.distributed.barrier()
    if ra.ra_get_device_status() != 0:
        raise RuntimeError("device status error during timed steps")
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in zip(starts, ends)))
    out = {"ms": ms, "wall": wall, "clocks": clk.summary(), "flops": W.flops()}
    if host_e2e:
        # The same call end to end through the public API: every step uploads
        # its q, k, v from pinned host memory and reads O and LSE back.  As in
        # a serving loop, two device buffer sets and two copy streams let step
        # s+1's upload and step s-1's download overlap step s's attention; the
        # timed region runs from the first upload to the last download.
        qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
        sets = [(qg, kg, vg, o, lse),
                tuple(torch.empty_like(t) for t in (qg, kg, vg, o, lse))]
        outs = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                 torch.empty(lse.shape, dtype=torch.float32).pin_memory()) for _ in range(2)]
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        loaded = [torch.cuda.Event() for _ in range(2)]  # inputs of the set on the device
        done = [torch.cuda.Event() for _ in range(2)]    # attention of the set finished
        read = [torch.cuda.Event() for _ in range(2)]    # outputs of the set copied out

        def e2e_step(i):
            bs = i % 2
            qd, kd, vd, od, ld = sets[bs]
            up.wait_event(done[bs])  # the set's previous attention has read its inputs
            with torch.cuda.stream(up):
                qd.copy_(qh, non_blocking=True)
                kd.copy_(kh, non_blocking=True)
                vd.copy_(vh, non_blocking=True)
            loaded[bs].record(up)
            stream.wait_event(loaded[bs])
            stream.wait_event(read[bs])  # the set's previous outputs are on the host
            ra.attn_fwd_causal_rope(qd, kd, vd, cos, sin, kv_offset=W.kv_offset,
                                    layout=W.layout, out=od, lse=ld, stream=stream)
            done[bs].record(stream)
            down.wait_event(done[bs])
            with torch.cuda.stream(down):
                outs[bs][0].copy_(od, non_blocking=True)
                outs[bs][1].copy_(ld, non_blocking=True)
            read[bs].record(down)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        n = max(4, args.steps)  # as many steps as the device-timed region
        te = time.perf_counter()
        for i in range(n):
            e2e_step(i)
        torch.cuda.synchronize()
        out["e2e_s"] = (time.perf_counter() - te) / n
        if ra.ra_get_device_status() != 0:
            raise RuntimeError("device status error during end-to-end steps")
        out["h2d"] = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
        out["d2h"] = outs[0][0].numel() * outs[0][0].element_size() + outs[0][1].numel() * 4
        # The host link on its own (one step's copies, nothing else running):
        # when these take longer than the attention, the end-to-end step is
        # bound by the copies, not by the kernel.
        qd, kd, vd, od, _ = sets[0]

        def copy_ms(fn, s):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(s)
            with torch.cuda.stream(s):
                fn()
            b.record(s)
            torch.cuda.synchronize()
            return a.elapsed_time(b)
        h2d_ms = min(copy_ms(lambda: [d.copy_(h, non_blocking=True)
                                      for d, h in ((qd, qh), (kd, kh), (vd, vh))], up)
                     for _ in range(3))
        d2h_ms = min(copy_ms(lambda: outs[0][0].copy_(od, non_blocking=True), down)
                     for _ in range(3))
        out["link"] = {"h2d_GBps": out["h2d"] / (h2d_ms * 1e-3) / 1e9, "h2d_ms": h2d_ms,
                       "d2h_GBps": outs[0][0].numel() * outs[0][0].element_size()
                       / (d2h_ms * 1e-3) / 1e9, "d2h_ms": d2h_ms}
    return out


def time_backward(ra, W, args, dev, stream):
    """Times attn_bwd_causal_rope on workload W (the forward's o and LSE are
    computed once, untimed); L2 flushed before every timed call.  FLOPs are
    the algorithmic 2.5x of the forward (the five products S, dP, dV, dK,
    dQ over the admissible pairs)."""
    q, k, v = W.inputs()
    g = torch.Generator("cpu").manual_seed(W.seed + 7)
    dout = wl.randn((W.B, W.Hq, W.Sq, W.D), g, wl.DTYPES[W.dtype])
    qg, kg, vg, dg = q.to(dev), k.to(dev), v.to(dev), dout.to(dev)
    cos, sin = ra.make_tables(max(W.Sk, W.kv_offset + W.Sq), W.r, W.base, device=dev)
    o, lse = ra.attn_fwd_causal_rope(qg, kg, vg, cos, sin, kv_offset=W.kv_offset, layout=W.layout)
    dq, dk, dv = torch.empty_like(qg), torch.empty_like(kg), torch.empty_like(vg)
    wsb = ra.lib().attn_bwd_workspace_size(1, W.B, W.Hq, W.Hkv, W.Sq, W.Sk, W.D)
    wsp = torch.empty(max(int(wsb), 1), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def call():
        ra.attn_bwd_causal_rope(qg, kg, vg, o, lse, dg, cos, sin, kv_offset=W.kv_offset,
                                layout=W.layout, dq=dq, dk=dk, dv=dv, workspace=wsp)

    for _ in range(args.warmup):
        flush_l2(flush)
        call()
    torch.cuda.synchronize()
    if ra.ra_get_device_status() != 0:
        raise RuntimeError("device status error in backward warm-up")
    ts = []
    for _ in range(args.steps):
        flush_l2(flush)
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        e.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(e))
    if ra.ra_get_device_status() != 0:
        raise RuntimeError("device status error in backward")
    ms = statistics.mean(ts)
    flops = 2.5 * W.flops()
    return {"ms": ms, "flops": flops, "tflops": flops / (ms * 1e-3) / 1e12,
            "kernels": ra.ra_last_launch()}


def time_rope(ra, args, dev, stream):
    """Times the in-place rope_apply_qk over the continuous-batching batch
    (its 1.4 GB working set exceeds L2, so no flush is needed)."""
    rq, rk = ROPE.inputs()
    pos = ROPE.positions()
    T = ROPE.T
    if args.rope_tokens:
        T = args.rope_tokens
        rq, rk, pos = rq[:T], rk[:T], pos[:T]
    rpos = torch.from_numpy(pos).to(torch.int32).to(dev)
    rqg, rkg = rq.to(dev), rk.to(dev)
    rcos, rsin = ra.make_tables(ROPE.table_rows, ROPE.rot_dim, ROPE.base, device=dev)
    for _ in range(args.warmup):
        ra.rope_apply_qk(rqg, rkg, rpos, rcos, rsin, layout=ROPE.layout)
    torch.cuda.synchronize()
    rs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    re_ = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for s in range(args.steps):
        rs[s].record(stream)
        ra.rope_apply_qk(rqg, rkg, rpos, rcos, rsin, layout=ROPE.layout)
        re_[s].record(stream)
    torch.cuda.synchronize()
    if ra.ra_get_device_status() != 0:
        raise RuntimeError("device status error in rope_apply")
    ms = statistics.mean(a.elapsed_time(b) for a, b in zip(rs, re_))
    nbytes = ROPE.algorithmic_bytes() * T // ROPE.T
    return {"ms": ms, "bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9, "T": T}


def time_decode(ra, args, dev, stream, host_e2e=True):
    """Times the decoder step on the decode workload: rope_append_kv of the
    512 new tokens (Q rotated in place, rotated K and raw V written to the
    cache) and attn_decode over each request's whole context.  The cache is
    packed token-major ([rows][8][128], request b from row sum of the earlier
    lengths) and filled on the device from a seeded generator; its ~140 GB
    exceed L2, so no flush is needed."""
    lens = DEC.kv_lens()
    if args.decode_reqs:
        lens = lens[:args.decode_reqs]
    B = lens.shape[0]
    dt = wl.DTYPES[DEC.dtype]
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    rows = int(lens.sum())
    g = torch.Generator(device=dev)
    g.manual_seed(DEC.seed)
    kc = torch.randn((rows, DEC.Hkv, DEC.D), generator=g, device=dev, dtype=dt)
    vc = torch.randn((rows, DEC.Hkv, DEC.D), generator=g, device=dev, dtype=dt)
    cache = ra.KVCache(kc, vc, torch.from_numpy(starts).to(dev))
    q, kn, vn = DEC.new_tokens()
    q, kn, vn = q[:B], kn[:B], vn[:B]
    qg, kg, vg = q.to(dev), kn.to(dev), vn.to(dev)
    pos = torch.from_numpy(lens - 1).to(torch.int32).to(dev)
    kv_len = torch.from_numpy(lens).to(torch.int32).to(dev)
    max_len = int(lens.max())
    cos, sin = ra.make_tables(DEC.table_rows, DEC.rot_dim, DEC.base, device=dev)
    wsb = ra.attn_decode_workspace_size(dt, B, DEC.Hq, DEC.Hkv, DEC.Sq, DEC.D, max_len)
    wsp = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    out = torch.empty((B, DEC.Hq, DEC.Sq, DEC.D), dtype=dt, device=dev)
    lse = torch.empty((B, DEC.Hq, DEC.Sq), dtype=torch.float32, device=dev)
    q4 = qg.view(B, DEC.Sq, DEC.Hq, DEC.D).permute(0, 2, 1, 3)

    def append():
        ra.rope_append_kv(cache, qg, kg, vg, pos, cos, sin, layout=DEC.layout)

    def attend():
        ra.attn_decode(cache, q4, kv_len, max_len, out=out, lse=lse, workspace=wsp)

    for _ in range(args.warmup):
        append()
        attend()
    torch.cuda.synchronize()
    if ra.ra_get_device_status() != 0:
        raise RuntimeError("device status error in decode warm-up")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for s in range(args.steps):
        ev[s][0].record(stream)
        append()
        ev[s][1].record(stream)
        attend()
        ev[s][2].record(stream)
    torch.cuda.synchronize()
    if ra.ra_get_device_status() != 0:
        raise RuntimeError("device status error in decode")
    app_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    att_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    nbytes = DEC.algorithmic_bytes(lens)
    res = {"B": B, "rows": rows, "append_ms": app_ms, "attn_ms": att_ms,
           "step_ms": app_ms + att_ms, "bytes": nbytes, "gbs": nbytes / (att_ms * 1e-3) / 1e9,
           "splits": None if wsb == 0 else "split-KV with merge", "ws_bytes": wsb}
    if host_e2e:
        qh, kh, vh = q.pin_memory(), kn.pin_memory(), vn.pin_memory()
        oh = torch.empty(out.shape, dtype=dt).pin_memory()
        n = max(1, min(args.steps, 5))
        for it in range(1 + n):
            if it == 1:
                torch.cuda.synchronize()
                te = time.perf_counter()
            qg.copy_(qh, non_blocking=True)
            kg.copy_(kh, non_blocking=True)
            vg.copy_(vh, non_blocking=True)
            append()
            attend()
            oh.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        res["e2e_ms"] = (time.perf_counter() - te) / n * 1e3
        res["h2d"] = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
        res["d2h"] = oh.numel() * oh.element_size()
    del kc, vc, cache
    torch.cuda.empty_cache()
    return res


def decode_summary(d, hbm_peak, peak_kind):
    out = {"workload": DEC.name, "requests": d["B"], "cached_rows": d["rows"],
           "attn_decode_ms": d["attn_ms"], "rope_append_kv_ms": d["append_ms"],
           "step_ms": d["step_ms"], "algorithmic_bytes": d["bytes"], "value": d["gbs"],
           "unit": "GB/s",
           "roofline": {"bound": "hbm", "achieved": d["gbs"], "peak": hbm_peak, "unit": "GB/s",
                        "frac": d["gbs"] / hbm_peak,
                        "traffic": dram_traffic("attn_decode_tc", DECODE_KERNEL_SRC),
                        "peak_kind": f"{peak_kind} HBM copy",
                        "note": "attn_decode call (split kernel + merge) over its algorithmic "
                                "bytes"},
           "l2": "cache larger than L2"}
    if "e2e_ms" in d:
        out["e2e"] = {"ms_per_step": d["e2e_ms"], "h2d_bytes_per_step": d["h2d"],
                      "d2h_bytes_per_step": d["d2h"]}
    return out


def cold_ms(call, flush, stream, steps, warmup):
    """Median device time of one call with L2 flushed before it (CUDA events
    on the launching stream, the call queued behind a GPU-side sleep)."""
    for _ in range(warmup):
        call()
    ts = []
    for _ in range(steps):
        flush_l2(flush)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def time_small_configs(ra, args, dev, stream, tf_peak, hbm_peak, peak_kind):
    """The configurations small enough to fit in L2, each timed cold (L2
    flushed before every call, median of the timed calls): the bf16 GPT-J
    sweep (TFLOP/s against the bf16 peak, and the peak device memory one
    call allocates beyond its inputs against |O| + |LSE|), the decode RoPE
    batch (GB/s against the HBM copy) and the fp32 attention (device time)."""
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    steps = max(args.steps, 10)
    sweep = []
    for W in wl.SWEEP:
        q, k, v = [t.to(dev) for t in W.inputs()]
        cos, sin = ra.make_tables(max(W.Sk, W.kv_offset + W.Sq), W.r, W.base, device=dev)

        def call():
            return ra.attn_fwd_causal_rope(q, k, v, cos, sin, kv_offset=W.kv_offset,
                                           layout=W.layout)
        ms = cold_ms(call, flush, stream, steps, args.warmup)
        torch.cuda.synchronize()
        base_mem = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        o, lse = call()
        torch.cuda.synchronize()
        extra = torch.cuda.max_memory_allocated() - base_mem
        o_lse = o.numel() * o.element_size() + lse.numel() * lse.element_size()
        del o, lse
        tf = W.flops() / (ms * 1e-3) / 1e12
        sweep.append({"workload": W.name, "us": ms * 1e3, "TFLOP/s": tf,
                      "frac": tf / tf_peak, "peak_extra_bytes": int(extra),
                      "o_plus_lse_bytes": int(o_lse)})
    R = wl.DECODE_ROPE
    rq, rk = [t.to(dev) for t in R.inputs()]
    pos = torch.from_numpy(R.positions()).to(torch.int32).to(dev)
    cos, sin = ra.make_tables(R.table_rows, R.rot_dim, R.base, device=dev)
    ms = cold_ms(lambda: ra.rope_apply_qk(rq, rk, pos, cos, sin, layout=R.layout), flush,
                 stream, steps, args.warmup)
    gbs = R.algorithmic_bytes() / (ms * 1e-3) / 1e9
    decode_rope = {"workload": R.name, "us": ms * 1e3, "GB/s": gbs,
                   "algorithmic_bytes": R.algorithmic_bytes(),
                   "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak,
                                "unit": "GB/s", "frac": gbs / hbm_peak,
                                "peak_kind": f"{peak_kind} HBM copy"},
                   "l2": "flushed before every call"}
    F = wl.FP32_ATTN
    q, k, v = [t.to(dev) for t in F.inputs()]
    cos, sin = ra.make_tables(max(F.Sk, F.kv_offset + F.Sq), F.r, F.base, device=dev)
    ms = cold_ms(lambda: ra.attn_fwd_causal_rope(q, k, v, cos, sin, layout=F.layout,
                                                 softmax_scale=1.0 / 8), flush, stream, steps,
                 args.warmup)
    fp32 = {"workload": F.name, "us": ms * 1e3,
            "GFLOP/s": F.flops() / (ms * 1e-3) / 1e9, "l2": "flushed before every call"}
    if ra.ra_get_device_status() != 0:
        raise RuntimeError("device status error in the small configurations")
    # What any single launch costs under this protocol: a one-element
    # elementwise kernel (PyTorch's, not the library's) timed the same way.
    one = torch.zeros(1, device=dev)
    floor = {"us": cold_ms(lambda: one.add_(1.0), flush, stream, steps, args.warmup) * 1e3,
             "kernel": "one-element torch add_ (not a library kernel)",
             "l2": "flushed before every call"}
    return {"sweep": sweep, "decode_rope": decode_rope, "fp32_attn": fp32, "cold_floor": floor}


def warm_ms(call, stream, n):
    """Device time per call when calls are pipelined: n calls captured in one
    CUDA graph, one replay timed between two events (no host launch gaps, L2
    warm).  The library's one-time set-up runs before capture (warm-up)."""
    call()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for _ in range(n):
                call()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def run_sweep(ra, args, dev, stream, rank, tf_peak, hbm_peak):
    """One line per workload: attention TFLOP/s (L2 flushed per call, CUDA
    events, median) and rope GB/s; not the bench line."""
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for W in wl.ALL_ATTN:
        q, k, v = [t.to(dev) for t in W.inputs()]
        cos, sin = ra.make_tables(max(W.Sk, W.kv_offset + W.Sq), W.r, W.base, device=dev)
        scale = 1.0 / 8 if W is wl.FP32_ATTN else None
        call = lambda: ra.attn_fwd_causal_rope(q, k, v, cos, sin, kv_offset=W.kv_offset,
                                               layout=W.layout, softmax_scale=scale)
        for _ in range(args.warmup):
            call()
        ts = []
        for _ in range(args.steps):
            flush_l2(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ms = statistics.median(ts)
        tf = W.flops() / (ms * 1e-3) / 1e12
        warm = warm_ms(call, stream, 20)
        if rank == 0:
            print(json.dumps({"workload": W.name, "ms": ms, "TFLOP/s": tf,
                              "frac_of_bf16_peak": tf / tf_peak, "warm_ms": warm,
                              "warm_TFLOP/s": W.flops() / (warm * 1e-3) / 1e12}), flush=True)
    # P1's comparison on GB300: plain flash, rotate-then-flash, fused; device
    # time per call (graph-replayed) and peak extra memory of one call
    for W in wl.SWEEP:
        q, k, v = [t.to(dev) for t in W.inputs()]
        cos, sin = ra.make_tables(W.Sk, W.r, W.base, device=dev)

        def flash():
            return ra.attn_fwd_causal_rope(q, k, v, apply_rope=False)

        def unfused():
            qr = torch.empty_like(q)
            kr = torch.empty_like(k)
            for b in range(W.B):  # [H, S, D] of one batch viewed token-major as [S, H, D]
                ra.rope_apply_qk(q[b].transpose(0, 1), k[b].transpose(0, 1), pos, cos, sin,
                                 layout=W.layout, q_out=qr[b].transpose(0, 1),
                                 k_out=kr[b].transpose(0, 1))
            return ra.attn_fwd_causal_rope(qr, kr, v, apply_rope=False)

        def fused():
            return ra.attn_fwd_causal_rope(q, k, v, cos, sin, layout=W.layout)

        pos = torch.arange(W.Sq, dtype=torch.int32, device=dev)
        row = {"ablation": W.name}
        for name, fn in (("flash", flash), ("rope_then_flash", unfused), ("fused", fused)):
            fn()
            torch.cuda.synchronize()
            base_mem = torch.cuda.memory_allocated()
            torch.cuda.reset_peak_memory_stats()
            fn()
            torch.cuda.synchronize()
            extra = torch.cuda.max_memory_allocated() - base_mem
            row[name] = {"warm_ms": warm_ms(fn, stream, 20), "peak_extra_MB": extra / 2 ** 20}
        if rank == 0:
            print(json.dumps(row), flush=True)
    for R in wl.ALL_ROPE:
        rq, rk = [t.to(dev) for t in R.inputs()]
        pos = torch.from_numpy(R.positions()).to(torch.int32).to(dev)
        cos, sin = ra.make_tables(R.table_rows, R.rot_dim, R.base, device=dev)
        call = lambda: ra.rope_apply_qk(rq, rk, pos, cos, sin, layout=R.layout)
        for _ in range(args.warmup):
            call()
        ts = []
        for _ in range(args.steps):
            flush_l2(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ms = statistics.median(ts)
        gbs = R.algorithmic_bytes() / (ms * 1e-3) / 1e9
        warm = warm_ms(call, stream, 20)
        if rank == 0:
            print(json.dumps({"workload": R.name, "ms": ms, "GB/s": gbs,
                              "frac_of_hbm": gbs / hbm_peak, "l2": "flushed per call",
                              "warm_ms": warm}), flush=True)
    if ra.ra_get_device_status() != 0:
        raise RuntimeError("device status error in sweep")
    return 0


def run_ours(args, ws, rank, local):
    import rope_causal_attention_gb300 as ra
    from rope_causal_attention_gb300 import build as rbuild
    if rank == 0 or not os.path.exists(ra.library_path()):
        rbuild.build()
    if ws > 1:
        torch.distributed.barrier()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    hbm_peak, tf_peak, peak_kind = peaks()

    if args.sweep:
        return run_sweep(ra, args, dev, stream, rank, tf_peak, hbm_peak)
    if args.only == "bwd":
        W = attn_workload(args)
        bw = time_backward(ra, W, args, dev, stream)
        if rank == 0:
            print(json.dumps({"only": "bwd", "workload": W.name, "ms": bw["ms"],
                              "TFLOP/s": bw["tflops"], "frac": bw["tflops"] / tf_peak,
                              "kernels": bw["kernels"]}))
        return 0
    if args.only == "decode":
        d = time_decode(ra, args, dev, stream, host_e2e=False)
        if rank == 0:
            print(json.dumps({"only": "decode", **decode_summary(d, hbm_peak, peak_kind)}))
        return 0
    if args.only == "rope":
        r = time_rope(ra, args, dev, stream)
        if rank == 0:
            print(json.dumps({"only": "rope", "workload": ROPE.name, "tokens": r["T"],
                              "ms": r["ms"], "GB/s": r["gbs"], "frac": r["gbs"] / hbm_peak}))
        return 0
    W = attn_workload(args)
    a = time_attention(ra, W, args, dev, stream, ws, local, host_e2e=args.only == "all")
    per_gpu_tflops = a["flops"] / (a["ms"] * 1e-3) / 1e12
    if args.only == "attn":
        if rank == 0:
            print(json.dumps({"only": "attn", "workload": W.name, "ms": a["ms"],
                              "TFLOP/s": per_gpu_tflops, "frac": per_gpu_tflops / tf_peak,
                              "clocks": a["clocks"]}))
        return 0
    r = time_rope(ra, args, dev, stream)
    d = time_decode(ra, args, dev, stream)
    bw = time_backward(ra, W, args, dev, stream)
    small = time_small_configs(ra, args, dev, stream, tf_peak, hbm_peak, peak_kind)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        tf, dt, threads, desc = cpu_oracle_attention(args.cpu_rows)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": desc + f"; {dt:.1f} s"}
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": per_gpu_tflops * ws, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": a["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v, workloads.LONG_GQA)",
        "config": {"workload": W.name, "B": W.B, "Hq": W.Hq, "Hkv": W.Hkv, "Sq": W.Sq,
                   "Sk": W.Sk, "D": W.D, "kv_offset": W.kv_offset, "layout": "neox",
                   "base": W.base, "flop_per_step": a["flops"],
                   "l2": "flushed before every timed step (256 MiB write)",
                   "parallelism": f"replicas x{ws}"},
        "roofline": {"bound": "tensor", "achieved": per_gpu_tflops, "peak": tf_peak,
                     "unit": "TFLOP/s", "frac": per_gpu_tflops / tf_peak,
                     "traffic": dram_traffic("attn_tc_long_gqa", ATTN_KERNEL_SRC),
                     "peak_kind": f"{peak_kind} bf16 dense (burst)"},
        "rope_apply": {"workload": ROPE.name, "value": r["gbs"], "unit": "GB/s", "ms": r["ms"],
                       "algorithmic_bytes": r["bytes"],
                       "roofline": {"bound": "hbm", "achieved": r["gbs"], "peak": hbm_peak,
                                    "unit": "GB/s", "frac": r["gbs"] / hbm_peak,
                                    "traffic": dram_traffic("rope_apply_cb", ROPE_KERNEL_SRC),
                                    "peak_kind": f"{peak_kind} HBM copy"},
                       "l2": "working set 1.4 GB > L2"},
        "decode_step": decode_summary(d, hbm_peak, peak_kind),
        "backward": {"workload": W.name, "ms": bw["ms"], "value": bw["tflops"],
                     "unit": "TFLOP/s", "algorithmic_flops": bw["flops"],
                     "kernels": bw["kernels"],
                     "roofline": {"bound": "tensor", "achieved": bw["tflops"], "peak": tf_peak,
                                  "unit": "TFLOP/s", "frac": bw["tflops"] / tf_peak,
                                  "traffic": dram_traffic("attn_bwd_long_gqa", BWD_KERNEL_SRC),
                                  "traffic_scope": "DRAM bytes of one whole backward call "
                                                   "(row term, Q and K rotation, dK/dV, dQ)",
                                  "peak_kind": f"{peak_kind} bf16 dense (burst)",
                                  "note": "2.5x the forward's FLOPs (S, dP, dV, dK, dQ); the "
                                          "kernels recompute S and dP once more for dQ"},
                     "l2": "flushed before every timed call"},
        "sweep": small["sweep"],
        "decode_rope": small["decode_rope"],
        "fp32_attn": small["fp32_attn"],
        "cold_floor": small["cold_floor"],
        "cpu_baseline": cpu,
        "e2e": {"value": a["flops"] / a["e2e_s"] / 1e12 * ws, "unit": "TFLOP/s",
                "h2d_bytes_per_step": a["h2d"], "d2h_bytes_per_step": a["d2h"],
                "ms_per_step": a["e2e_s"] * 1e3, "link": a["link"]},
        "gpu_launches": args.steps,  # one attention kernel per timed step
        "clocks": a["clocks"],
        "wall_s_timed_region": a["wall"],
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-rows", type=int, default=4096)
    ap.add_argument("--ref-rows", type=int, default=2048)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-reqs", type=int, default=0,
                    help="profiling aid: decode only the first N requests of the decode batch")
    ap.add_argument("--only", choices=["all", "attn", "rope", "decode", "bwd"], default="all",
                    help="profiling aid: time one kernel only (no e2e, no CPU baseline)")
    ap.add_argument("--attn-sq", type=int, default=0,
                    help="profiling aid: shrink the attention workload to this many new "
                         "queries (the 4096-row cached prefix is kept)")
    ap.add_argument("--attn-workload", choices=[w.name for w in wl.ALL_ATTN], default=None,
                    help="profiling aid (with --only attn): time this attention workload "
                         "instead of the long-context one")
    ap.add_argument("--sweep", action="store_true",
                    help="report: time every attention workload (fp32, the GPT-J sweep, "
                         "long-context GQA) and both rope workloads, one JSON line each")
    ap.add_argument("--rope-tokens", type=int, default=0,
                    help="profiling aid: rotate only the first N tokens of the batch")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_env()
    if ws > 1:
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend)
    try:
        if args.impl == "reference":
            return run_reference(args, ws, rank)
        return run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
