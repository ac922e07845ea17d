"""Throughput of the compressed-KV attention layer on one GB300 (or N replicas).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one pass of the whole per-layer path over one batch:
  decode workloads  — for every layer: append the new token (raw window +
                      compressor), indexer top-k on ratio-4 layers, sparse
                      attention; one new token per sequence;
  prefill workload  — one 4096-token chunk: append, per-query top-k, chunk
                      attention with the raw-window commit.
Default workload: the 43-layer Flash schedule decoding 8 sequences at context
131,072 (ratio-4 and ratio-128 layers, both lanes, every step of the path).
`value` is whole-job tokens/s with every input resident in HBM, over K graph
replays timed as one region; `median_ms_per_step` is the median of at least
100 replays timed one by one. `e2e` adds the per-step host->device copy of the
step's inputs (pinned) and the device->host read of the last layer's output.
On one GPU the default line also carries, under `workloads`, the single c4a
layer decode (32 sequences at 65,536), the single c128a layer decode (one
sequence at 65,536) and the 4096-token prefill chunk at 28,672, each with its
own roofline, and under `boundary_step` the Flash stack decoding at 131,071,
where every compressed layer emits a row. `cpu_baseline` times the oracle on
every host core and on one core; the reference arm (--impl reference) times it
on every host core. Both time a bounded sample of the workload and scale it to
a step by a stated factor.
"""
import argparse
import json
import os

import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = ("c4a/c128a decode tok/s & HBM GB/s frac; 4096-chunk prefill tok/s (1×GB300)")
WORKLOADS = {"flash43": synth.FLASH_STACK, "c4a_decode": synth.C4A_DECODE,
             "c128a_decode": synth.C128A_DECODE, "prefill": synth.C4A_PREFILL,
             "tiny": synth.TINY, "flash_c4a_layer": synth.FLASH_C4A_LAYER}
WORKLOADS_BY_NAME = {w.name: w for w in WORKLOADS.values()}
SINGLE_THREAD_ENV = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
# ncu DRAM counters per call, recorded with the hash of the kernel sources they
# were taken on; a stale record (sources changed since) reports null
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")
CALL_KERNELS = {"index_topk": ("index_", "topk_"), "append": ("append_", "state_reset"),
                "attn": ("attn_", "ring_commit")}


def sources_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for d in ("compressed_kv_sparse_gb300/csrc", "include"):
        base = os.path.join(ROOT, d)
        for name in sorted(os.listdir(base)):
            if name.endswith((".cu", ".cuh", ".h")):
                with open(os.path.join(base, name), "rb") as f:
                    h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def recorded_traffic(workload: str, call: str):
    try:
        with open(TRAFFIC_PATH) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("sources_sha256") != sources_hash():
        return None
    if call.startswith("attn_r"):
        call = "attn"
    e = rec.get("entries", {}).get(workload, {}).get(call)
    return float(e["bytes_per_call"]) if e else None


def write_traffic(csv_path: str, workload: str, captured_on: str, calls: int):
    """Sum DRAM read + write bytes of one call's kernels from an ncu CSV
    (--metrics dram__bytes_read.sum,dram__bytes_write.sum) into the record."""
    import csv
    import re
    rows = list(csv.reader(open(csv_path)))
    hi = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    h = rows[hi]
    ki, mi, vi = h.index("Kernel Name"), h.index("Metric Name"), h.index("Metric Value")
    ui = h.index("Metric Unit") if "Metric Unit" in h else None
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    per_call = {}
    for r in rows[hi + 1:]:
        if len(r) <= vi or r[mi] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        # (the anonymous namespace prints as "(anonymous namespace)::" or
        # "<unnamed>::": strip it before the argument list, whose "(" it shares)
        name = re.sub(r"^.*?(unnamed>|anonymous namespace\))::", "", r[ki].replace("void ", ""))
        name = re.sub(r"\(.*", "", name)
        v = float(r[vi].replace(",", "")) * scale.get(r[ui] if ui is not None else "byte", 1)
        for call, prefixes in CALL_KERNELS.items():
            if name.startswith(prefixes):
                per_call[call] = per_call.get(call, 0.0) + v
    try:
        with open(TRAFFIC_PATH) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        rec = {}
    if rec.get("sources_sha256") != sources_hash():
        rec = {"sources_sha256": sources_hash(), "entries": {}}
    ent = rec["entries"].setdefault(WORKLOADS[workload].name, {})
    for call, v in per_call.items():
        ent[call] = {"bytes_per_call": v / calls, "captured_on": captured_on,
                     "kernels": list(CALL_KERNELS[call])}
    with open(TRAFFIC_PATH, "w") as f:
        json.dump(rec, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps(ent))


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------- GPU runner

class Runner:
    """Builds every layer's cache and inputs on the device and runs steps."""

    def __init__(self, wl: synth.Workload, device, rank: int = 0, qat: bool = False,
                 streams: int = 1, paged: bool = False):
        from compressed_kv_sparse_gb300 import lib
        self.lib, self.wl, self.dev = lib, wl, device
        # streams == 2 (decode): the indexer lane's append and the top-k of a
        # c4a layer run on a second stream beside the raw insert and the
        # attention lane's append
        self.streams = streams
        self.aux = torch.cuda.Stream(device=device) if streams == 2 else None
        self.decode = wl.mode == "decode"
        self.T = 1 if self.decode else wl.chunk
        self.p0 = wl.context
        seed_wl = wl if rank == 0 else synth.Workload(wl.name, wl.seed + 1000 * rank, wl.batch,
                                                      wl.layers, wl.context, wl.mode, wl.chunk,
                                                      wl.hidden)
        self.layers = []
        B = wl.batch
        end = self.p0 + self.T
        for il, s in enumerate(wl.layers):
            cap = end // s.ratio + 1 if s.ratio else 0
            table, n_blocks = None, 0
            if paged and s.ratio:
                # 256-position blocks in a random order of one shared pool
                rpb = 256 // s.ratio
                max_blocks = cap // rpb + 1
                cap, n_blocks = max_blocks * rpb, B * max_blocks
                perm = torch.randperm(n_blocks, generator=torch.Generator().manual_seed(il))
                table = perm.to(torch.int32).reshape(B, max_blocks).to(device)
            c = lib.LayerCache(ratio=s.ratio, head_dim=s.head_dim, n_rot=s.n_rot, batch=B,
                               comp_cap=cap, dtype=s.dtype, base=s.rope_base,
                               rope_max_pos=end + 1, index_dim=s.index_dim,
                               index_rot=s.index_rot, cap_raw=s.cap_raw,
                               qat=qat_flags(s.ratio) if qat else 0, device=device,
                               block_table=table, n_blocks=n_blocks)
            hist = synth.cache_history(seed_wl, il, self.p0, comp_cap=cap, device=device)
            c.load_state(hist, self.p0)
            del hist
            inp = synth.step_inputs(seed_wl, il, self.p0, self.T, device=device)
            inp = {k: v.contiguous() for k, v in inp.items()}
            L = {"s": s, "cache": c, "inp": inp}
            k = s.top_k
            if s.ratio == 4:
                L["topk"] = torch.empty((B, self.T, k) if not self.decode else (B, k),
                                        dtype=torch.int32, device=device)
                L["ws_idx"] = lib.workspace(c.workspace_bytes(lib.CALL_INDEX_TOPK, self.T,
                                                              s.index_heads, k), device)
            call = lib.CALL_ATTN_DECODE if self.decode else lib.CALL_ATTN_PREFILL
            L["ws_attn"] = lib.workspace(c.workspace_bytes(call, self.T, s.n_heads, k), device)
            if self.decode:
                L["q"] = inp["q"][:, 0].contiguous()
                L["out"] = torch.empty((B, s.n_heads, s.head_dim), dtype=c.torch_dtype,
                                       device=device)
            else:
                L["q"] = inp["q"]
                L["out"] = torch.empty((B, self.T, s.n_heads, s.head_dim), dtype=c.torch_dtype,
                                       device=device)
                L["chunk"] = torch.empty((B, self.T, s.head_dim), dtype=c.torch_dtype,
                                         device=device)
            self.layers.append(L)
        torch.cuda.synchronize(device)

    # the library calls of one layer's step, in order: (name, fn)
    def layer_calls(self, L):
        lib, s, c, inp = self.lib, L["s"], L["cache"], L["inp"]
        k, scale = s.top_k, lib.default_scale(s.head_dim)
        p0, T, end = self.p0, self.T, self.p0 + self.T

        def at(n, fn):          # the host position mirror each call expects
            def run():
                c.n_tokens = n
                fn()
            return run

        calls = []
        if self.decode:
            calls.append(("append", at(p0, lambda: lib.ds4a_compress_append(c, p0, 1, inp))))
            if s.ratio == 4:
                calls.append(("index_topk", at(end, lambda: lib.ds4a_index_topk(
                    c, p0, 1, inp["q_idx"], inp["w"], s.index_heads, k, L["topk"],
                    L["ws_idx"]))))
            calls.append((f"attn_r{s.ratio}", at(end, lambda: lib.ds4a_sparse_attn_decode(
                c, p0, L["q"], s.n_heads, L.get("topk"), k, scale, L["out"], L["ws_attn"]))))
        else:
            calls.append(("append", at(p0, lambda: lib.ds4a_compress_append(
                c, p0, T, inp, raw_chunk_out=L["chunk"]))))
            if s.ratio == 4:
                calls.append(("index_topk", at(end, lambda: lib.ds4a_index_topk(
                    c, p0, T, inp["q_idx"], inp["w"], s.index_heads, k, L["topk"],
                    L["ws_idx"]))))
            calls.append((f"attn_r{s.ratio}", at(end, lambda: lib.ds4a_sparse_attn_prefill_chunk(
                c, p0, T, L["q"], s.n_heads, L["chunk"], L.get("topk"), k, scale, L["out"],
                L["ws_attn"]))))
        return calls

    def layer_step(self, L):
        if self.streams == 2 and self.decode and L["s"].ratio == 4:
            self.layer_step_two_streams(L)
            return
        for _, fn in self.layer_calls(L):
            fn()

    def layer_step_two_streams(self, L):
        """c4a decode layer with the indexer pipeline on its own stream (vLLM's
        multi-stream partitioning): fork, [index-lane append -> top-k] beside
        [raw insert + attention-lane append], join, attention."""
        lib, s, c, inp = self.lib, L["s"], L["cache"], L["inp"]
        k, p0 = s.top_k, self.p0
        main = torch.cuda.current_stream()
        self.aux.wait_stream(main)
        c.n_tokens = p0
        with torch.cuda.stream(self.aux):
            lib.ds4a_compress_append_lanes(c, p0, 1, lib.LANE_INDEX, inp)
        lib.ds4a_compress_append_lanes(c, p0, 1, lib.LANE_RAW | lib.LANE_ATTN, inp)
        c.n_tokens = p0 + 1
        with torch.cuda.stream(self.aux):
            lib.ds4a_index_topk(c, p0, 1, inp["q_idx"], inp["w"], s.index_heads, k, L["topk"],
                                L["ws_idx"])
        main.wait_stream(self.aux)
        lib.ds4a_sparse_attn_decode(c, p0, L["q"], s.n_heads, L["topk"], k,
                                    lib.default_scale(s.head_dim), L["out"], L["ws_attn"])

    def step(self):
        for L in self.layers:
            self.layer_step(L)

    # every call of one kind, over all layers in order: (name, [fn, ...])
    def calls_by_kind(self):
        kinds = {}
        for L in self.layers:
            for name, fn in self.layer_calls(L):
                kinds.setdefault(name, []).append(fn)
        return kinds

    def tokens_per_step(self):
        return self.wl.batch * self.T

    # algorithmic bytes / FLOPs per call kind: the bytes a call must move at
    # least (rows it reads, inputs and outputs) and its useful multiply-adds
    def algorithmic(self):
        B, T = self.wl.batch, self.T
        out = {}
        for L in self.layers:
            s = L["s"]
            eb = 2 if s.dtype == "bf16" else 4
            p_last = self.p0 + T - 1
            if s.ratio == 4:
                vis = (p_last + 1) // 4
                if self.decode:
                    by = B * (vis * s.index_dim * eb + s.index_heads * (s.index_dim + 1) * eb +
                              s.top_k * 4)
                    fl = 2.0 * B * vis * s.index_heads * s.index_dim
                else:
                    pairs = sum((self.p0 + t + 1) // 4 for t in range(T))
                    by = B * (vis * s.index_dim * eb + T * s.index_heads * (s.index_dim + 1) * eb
                              + T * s.top_k * 4)
                    fl = 2.0 * B * pairs * s.index_heads * s.index_dim
                a = out.setdefault("index_topk", [0, 0.0, 0])
                a[0] += by
                a[1] += fl
                a[2] += 1
            # append: raw row in/out, lane candidates + scores in, state slots out
            lanes = [s.head_dim] if s.ratio else []
            if s.ratio == 4:
                lanes.append(s.index_dim)
            by = B * T * (2 * s.head_dim * eb + sum(2 * w * eb + 2 * w * 4 for w in lanes))
            a = out.setdefault("append", [0, 0.0, 0])
            a[0] += by
            a[2] += 1
            nw = min(p_last + 1, s.cap_raw)
            ncomp = s.top_k if s.ratio == 4 else (p_last + 1) // 128 if s.ratio == 128 else 0
            rows = nw + ncomp
            qo = 2 * s.n_heads * s.head_dim * eb
            if self.decode:
                by = B * (rows * s.head_dim * eb + qo + (s.top_k * 4 if s.ratio == 4 else 0))
            else:
                by = B * (T * rows * s.head_dim * eb + T * qo)
            fl = 4.0 * B * T * rows * s.n_heads * s.head_dim
            a = out.setdefault(f"attn_r{s.ratio}", [0, 0.0, 0])
            a[0] += by
            a[1] += fl
            a[2] += 1
        return out


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc = index, None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        else:
            self.lines = []

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            try:
                sm.append(float(f[0]))
                mx = max(mx, float(f[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def flush_l2(buf):
    buf.add_(1)


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's figure (every rank gets it); x itself on one rank."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_step_per_rank: int, step_s: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's step."""
    return world * tokens_per_step_per_rank / step_s


def qat_flags(ratio: int) -> int:
    """Step-8 flags of a layer: FP8 attention rows on compressed layers, FP4
    QAT of the indexer lane on ratio-4 layers."""
    from compressed_kv_sparse_gb300 import lib
    return (lib.QAT_FP8_ATTN if ratio else 0) | (lib.QAT_FP4_INDEX if ratio == 4 else 0)


def run_gpu(args, wl, rank, world, device):
    hbm, bf16, bf16s, peak_kind = peaks()
    lib_mod = __import__("compressed_kv_sparse_gb300.lib", fromlist=["lib"])
    R = Runner(wl, device, rank, qat=args.qat, streams=args.streams, paged=args.paged)
    step_bytes = sum(v[0] for v in R.algorithmic().values())
    flush = None
    if step_bytes < 512e6:      # working set below ~4x L2: flush between steps
        flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)

    def step():
        R.step()
        if flush is not None:
            flush_l2(flush)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)

    # graph of one step (launch overhead off the timed path)
    use_graph = not args.no_graph
    if use_graph:
        n0 = lib_mod.ds4a_launch_count()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device)
        s.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(s):
            R.step()           # one eager pass on the capture stream
        torch.cuda.current_stream(device).wait_stream(s)
        torch.cuda.synchronize(device)
        n0 = lib_mod.ds4a_launch_count()
        with torch.cuda.graph(g):
            R.step()
        launches_per_step = lib_mod.ds4a_launch_count() - n0
        run = lambda: (g.replay(), flush is not None and flush_l2(flush))
        for _ in range(2):
            run()
    else:
        n0 = lib_mod.ds4a_launch_count()
        R.step()
        launches_per_step = lib_mod.ds4a_launch_count() - n0
        run = step
    torch.cuda.synchronize(device)

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(device.index if device.index is not None else 0) as clk:
        e0.record()
        for _ in range(args.steps):
            run()
        e1.record()
        torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    ms = e0.elapsed_time(e1) / args.steps
    # the same replays timed one by one (median of at least 100), the L2
    # flush outside each pair of events
    rep_ms = []
    for _ in range(max(100, args.steps)):
        if flush is not None:
            flush_l2(flush)
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        r0.record()
        (g.replay() if use_graph else R.step())
        r1.record()
        rep_ms.append((r0, r1))
    torch.cuda.synchronize(device)
    rep_ms = sorted(a.elapsed_time(b) for a, b in rep_ms)
    median_ms = max_over_ranks(statistics.median(rep_ms), world, device)
    flush_ms = 0.0
    if flush is not None:        # subtract the L2 flush from the step time
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record()
        for _ in range(args.steps):
            flush_l2(flush)
        f1.record()
        torch.cuda.synchronize(device)
        flush_ms = f0.elapsed_time(f1) / args.steps
    ms_step = max_over_ranks(max(ms - flush_ms, 1e-6), world, device)
    value = job_throughput(world, R.tokens_per_step(), ms_step / 1e3)

    # per-call device time: for each call kind, one CUDA graph runs that call on
    # every layer that has it (layer order, as in a step); replays are timed
    # with CUDA events on the launching stream, with the L2 flush between
    # replays (when the step flushes) timed separately and subtracted
    per_call = {}
    torch.cuda.synchronize(device)
    reps = max(3, min(args.steps, 10))
    for name, fns in R.calls_by_kind().items():
        gk = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gk):
            for fn in fns:
                fn()
        for _ in range(2):
            gk.replay()
        torch.cuda.synchronize(device)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        for _ in range(reps):
            if flush is not None:
                flush_l2(flush)
            gk.replay()
        a1.record()
        torch.cuda.synchronize(device)
        per_call[name] = [(a0.elapsed_time(a1) - flush_ms * reps) / (reps * len(fns))]
        del gk
    alg = R.algorithmic()
    calls = {}
    for name, ts in per_call.items():
        n_per_step = alg[name][2]
        t_launch = max(ts[0], 1e-6) / 1e3           # seconds per call
        by = alg[name][0] / n_per_step
        fl = alg[name][1] / n_per_step
        calls[name] = {"ms_per_call": t_launch * 1e3, "calls_per_step": n_per_step,
                       "GB/s": by / t_launch / 1e9, "TFLOP/s": fl / t_launch / 1e12,
                       "bytes": by, "flop": fl}
    dom = max(calls, key=lambda n: calls[n]["ms_per_call"] * calls[n]["calls_per_step"])
    dc = calls[dom]
    tensor_bound = not R.decode
    if tensor_bound:
        roof = {"bound": "tensor", "achieved": dc["TFLOP/s"], "peak": bf16s, "unit": "TFLOP/s",
                "frac": dc["TFLOP/s"] / bf16s, "traffic": recorded_traffic(wl.name, dom),
                "kernel": dom, "peak_kind": f"{peak_kind} bf16 sustained"}
    else:
        roof = {"bound": "hbm", "achieved": dc["GB/s"], "peak": hbm, "unit": "GB/s",
                "frac": dc["GB/s"] / hbm, "traffic": recorded_traffic(wl.name, dom), "kernel": dom,
                "peak_kind": f"{peak_kind} hbm copy"}

    # end to end: pinned host inputs -> device, step, last output -> host
    host_in = []
    for L in R.layers:
        for name, t in L["inp"].items():
            if name.startswith(("ape", "gamma")):
                continue                       # weights stay resident
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            host_in.append((h, t))
    last = R.layers[-1]["out"]
    host_out = torch.empty(last.shape, dtype=last.dtype, pin_memory=True)
    h2d = sum(h.numel() * h.element_size() for h, _ in host_in)
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step():
        for h, t in host_in:
            t.copy_(h, non_blocking=True)
        if R.decode:
            for L in R.layers:
                L["q"].copy_(L["inp"]["q"][:, 0])
        run()
        host_out.copy_(last, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
        torch.cuda.synchronize(device)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / args.steps - flush_ms / 1e3, world,
                           device)
    e2e = {"value": job_throughput(world, R.tokens_per_step(), e2e_s), "unit": "tok/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    res = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
           "median_ms_per_step": median_ms, "timed_replays_for_median": len(rep_ms),
           "p10_p90_ms_per_step": [rep_ms[len(rep_ms) // 10], rep_ms[(9 * len(rep_ms)) // 10]],
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": wl.dtype, "data": "synthetic",
           "config": {"workload": wl.name, "mode": wl.mode, "batch_per_gpu": wl.batch,
                      "context": wl.context, "tokens_per_step_per_gpu": R.tokens_per_step(),
                      "positions": (f"decode at p = {wl.context}" if wl.mode == "decode" else
                                    f"chunk of {wl.chunk} at p = {wl.context}"),
                      "layers": len(wl.layers),
                      "ratios": {str(r): sum(1 for s in wl.layers if s.ratio == r)
                                 for r in (0, 4, 128)},
                      "l2": "flushed between steps" if flush is not None
                      else "inputs larger than L2 (algorithmic %.2f GB per step)" % (step_bytes / 1e9),
                      "cuda_graph": use_graph, "parallelism": f"replicas x{world}",
                      "step8_round_trips": "fp8 attention rows + fp4 indexer rows/queries"
                      if args.qat else "off",
                      "streams": args.streams,
                      "cache_layout": "paged, 256-position blocks" if args.paged else "contiguous",
                      "algorithmic_GB_per_step": step_bytes / 1e9,
                      "step_GB/s": step_bytes / (ms_step / 1e3) / 1e9},
           "roofline": roof, "calls": calls,
           "gpu_launches": int(launches_per_step) * args.steps,
           "clocks": clk.summary(), "e2e": e2e}
    return res, R


# ----------------------------------------------------------------- CPU oracle
# The CPU baseline and the reference arm time the oracle (test infrastructure)
# as it stands: plain numpy, one thread per process, on a bounded sample of the
# workload, once on every host core (one spawned process per core, each with
# its own units) and once on one core. The sample's time is scaled to a whole
# step by the stated factor.

def _one_seq(wl: synth.Workload, b: int) -> synth.Workload:
    """A one-sequence workload standing for sequence b (its own seeded draw)."""
    return synth.Workload(wl.name, wl.seed * 1000 + b, 1, wl.layers, wl.context, wl.mode,
                          wl.chunk, wl.hidden)


def _oracle_cache(s, hist, n_tokens):
    from oracle.layer import OracleCache
    f = lambda t: t.float().numpy()
    return OracleCache(ratio=s.ratio, head_dim=s.head_dim, n_rot=s.n_rot, cap_raw=s.cap_raw,
                       base=s.rope_base, dtype=s.dtype, n_tokens=n_tokens,
                       index_dim=s.index_dim, index_rot=s.index_rot,
                       **{k: f(v) for k, v in hist.items()})


def _build_unit(wl: synth.Workload, unit):
    """State for one unit of oracle work. Units: ("dec", ratio, il, b) one
    decode step of layer il for sequence b; ("app",) the prefill chunk's
    compressor append; ("qry", (t, ...)) the indexer top-k and attention of
    those chunk queries."""
    import numpy as np
    f = lambda t: t.float().numpy()
    if unit[0] == "dec":
        _, _, il, b = unit
        one = _one_seq(wl, b)
        s = wl.layers[il]
        cap = (wl.context + 1) // s.ratio + 1 if s.ratio else 0
        oc = _oracle_cache(s, synth.cache_history(one, il, wl.context, comp_cap=cap), wl.context)
        inp = {k: f(v) for k, v in synth.step_inputs(one, il, wl.context, 1).items()}
        state = {k: getattr(oc, k).copy() for k in ("attn_state_kv", "attn_state_score",
                                                     "index_state_kv", "index_state_score")
                 if getattr(oc, k) is not None}
        return {"oc": oc, "inp": inp, "state": state, "s": s}
    s = wl.layers[0]
    one = _one_seq(wl, 0)
    p0, T = wl.context, wl.chunk
    cap = (p0 + T) // 4 + 1
    oc = _oracle_cache(s, synth.cache_history(one, 0, p0, comp_cap=cap), p0)
    sd, key = one.seed, ("cpu-sample", p0, T)
    inp = {n: f(synth.normal((1, T, w), sd, *key, n, dtype=s.dtype))
           for n, w in (("raw_kv_in", s.head_dim), ("attn_cand", s.head_dim),
                        ("attn_score", s.head_dim), ("idx_cand", s.index_dim),
                        ("idx_score", s.index_dim))}
    inp.update({k: f(v) for k, v in synth.layer_weights(one, 0).items()})
    state = {k: getattr(oc, k).copy() for k in ("attn_state_kv", "attn_state_score",
                                                 "index_state_kv", "index_state_score")}
    if unit[0] == "app":
        return {"oc": oc, "inp": inp, "state": state, "s": s, "p0": p0}
    from oracle import layer as olayer
    ring = oc.raw_kv.copy()
    rows = olayer.compress_append(oc, p0, inp, chunk=True)
    ts = unit[1]
    n = len(ts)
    q = f(synth.normal((n, s.n_heads, s.head_dim), sd, *key, "q", dtype=s.dtype)).astype(np.float64)
    q_idx = f(synth.normal((n, s.index_heads, s.index_dim), sd, *key, "qidx", dtype=s.dtype))
    w = f(synth.normal((n, s.index_heads), sd, *key, "w", dtype=s.dtype))
    return {"oc": oc, "s": s, "p0": p0, "ring": ring, "rows": rows, "ts": ts, "q": q,
            "q_idx": q_idx, "w": w}


def _run_unit(unit, st):
    """The timed oracle work of one unit (state restored first where the work
    changes it: the same position is appended again on every repeat)."""
    from oracle import layer as olayer
    oc = st["oc"]
    if unit[0] == "dec":
        for k, v in st["state"].items():
            getattr(oc, k)[...] = v
        oc.n_tokens = st["p"]
        olayer.decode_step(oc, st["p"], st["inp"], st["s"].top_k)
        return
    if unit[0] == "app":
        for k, v in st["state"].items():
            getattr(oc, k)[...] = v
        oc.n_tokens = st["p0"]
        olayer.compress_append(oc, st["p0"], st["inp"], chunk=True)
        return
    from oracle.attention import attention_query, comp_row_ids
    from oracle.indexer import index_topk_query
    s, p0 = st["s"], st["p0"]
    for j, t in enumerate(st["ts"]):
        p = p0 + t
        tk = index_topk_query(st["q_idx"][j], st["w"][j], oc.index_comp_kv[0], p, oc.base,
                              oc.index_rot, oc.dtype, s.top_k)
        win = olayer._window_rows(oc, 0, p, p0, st["ring"], st["rows"])
        ids = comp_row_ids(oc.ratio, p, oc.n_comp, tk)
        attention_query(st["q"][j], p, win, oc.attn_comp_kv[0, ids], oc.base, oc.n_rot,
                        1.0 / s.head_dim ** 0.5, oc.dtype)


def _oracle_worker(conn, wl_name, units):
    """Child process: build every unit once, then on each command (a unit
    kind) run its units of that kind and reply with the start and end of the
    work on the host's monotonic clock."""
    wl = WORKLOADS_BY_NAME[wl_name]
    built = []
    for u in units:
        st = _build_unit(wl, u)
        if u[0] == "dec":
            st["p"] = wl.context
        built.append((u, st))
    conn.send("ready")
    while True:
        kind = conn.recv()
        if kind is None:
            break
        t0 = time.perf_counter()
        for u, st in built:
            if _unit_kind(u) == kind:
                _run_unit(u, st)
        conn.send((t0, time.perf_counter()))
    conn.close()


def _unit_kind(u):
    return ("dec", u[1]) if u[0] == "dec" else (u[0],)


def oracle_plan(wl: synth.Workload, cores: int):
    """Units of a bounded sample and how a step is built from them.

    Returns (units, phases, desc): phases is a list of (kind, factor): a step
    costs sum(factor * wall time of that kind's phase)."""
    if wl.mode == "decode":
        by = {}
        for il, s in enumerate(wl.layers):
            by.setdefault(s.ratio, []).append(il)
        units, phases, parts = [], [], []
        for ratio, ils in sorted(by.items()):
            n_l = len(ils)
            seqs = list(range(wl.batch)) if cores > 1 else [0]
            per = max(1, min(n_l, -(-cores // len(seqs)))) if cores > 1 else 1
            for il in ils[:per]:
                units += [("dec", ratio, il, b) for b in seqs]
            factor = n_l / per * (wl.batch / len(seqs))
            phases.append((("dec", ratio), factor))
            parts.append(f"ratio {ratio}: {per} of {n_l} layers x {len(seqs)} of {wl.batch} "
                         f"sequences (x{factor:g})")
        return units, phases, "decode step (append + top-k + attention) per (layer, sequence); "             + "; ".join(parts)
    T = wl.chunk
    n_q = max(4, 4 * cores)
    ts = [round(i * (T - 1) / (n_q - 1)) for i in range(n_q)]
    units = [("app",)] + [("qry", tuple(ts[i::cores])) for i in range(min(cores, n_q))]
    phases = [(("app",), float(wl.batch)), (("qry",), T / n_q * wl.batch)]
    return units, phases, (f"compressor append of the whole {T}-token chunk (x{wl.batch}), then "
                           f"{n_q} of {T} queries (indexer scan, top-k, attention; "
                           f"x{T / n_q * wl.batch:g})")


class OraclePool:
    """`cores` spawned worker processes, each holding its units' state."""

    def __init__(self, wl: synth.Workload, cores: int):
        import multiprocessing as mp
        self.units, self.phases, self.desc = oracle_plan(wl, cores)
        ctx = mp.get_context("spawn")
        n = min(cores, len(self.units))
        # deal the units of every kind round-robin over the workers
        share = [[] for _ in range(n)]
        for kind, _ in self.phases:
            ku = [u for u in self.units if _unit_kind(u) == kind]
            for i, u in enumerate(ku):
                share[i % n].append(u)
        self.conns, self.procs, self.share = [], [], share
        # one BLAS / OpenMP thread per worker: the children read these at start
        keep = {k: os.environ.get(k) for k in SINGLE_THREAD_ENV}
        os.environ.update({k: "1" for k in SINGLE_THREAD_ENV})
        try:
            for sh in share:
                a, b = ctx.Pipe()
                pr = ctx.Process(target=_oracle_worker, args=(b, wl.name, sh), daemon=True)
                pr.start()
                self.conns.append(a)
                self.procs.append(pr)
        finally:
            for k, v in keep.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        for c in self.conns:
            assert c.recv() == "ready"
        self.cores = n

    def step(self):
        """(seconds of sampled work on the wall clock, estimated seconds of one
        whole step)."""
        spent, est = 0.0, 0.0
        for kind, factor in self.phases:
            for c in self.conns:
                c.send(kind)
            ts = [c.recv() for c in self.conns]
            busy = [(t0, t1) for (t0, t1), sh in zip(ts, self.share)
                    if any(_unit_kind(u) == kind for u in sh)]
            wall = max(t1 for _, t1 in busy) - min(t0 for t0, _ in busy)
            spent += wall
            est += factor * wall
        return spent, est

    def close(self):
        for c in self.conns:
            try:
                c.send(None)
            except OSError:
                pass
        for pr in self.procs:
            pr.join(timeout=30)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _tokens(wl):
    return wl.batch * (1 if wl.mode == "decode" else wl.chunk)


def time_oracle(wl: synth.Workload, cores: int, budget_s: float, min_steps: int = 1):
    """Repeat the sampled step until budget_s of wall time; median estimate."""
    pool = OraclePool(wl, cores)
    try:
        pool.step()                       # warm-up
        spent, est = 0.0, []
        while spent < budget_s or len(est) < min_steps:
            sp, e = pool.step()
            spent += sp
            est.append(e)
        step_s = statistics.median(est)
        return {"value": _tokens(wl) / step_s, "unit": "tok/s", "cores": pool.cores,
                "kind": "oracle", "step_s_estimated": step_s,
                "sample": f"{pool.desc}; {len(est)} repeats, {spent:.1f} s of wall time"}
    finally:
        pool.close()


def cpu_baseline(wl: synth.Workload, budget_s: float = 8.0):
    """The oracle on every host core (headline) and on one core."""
    allc = time_oracle(wl, host_cores(), budget_s)
    one = time_oracle(wl, 1, budget_s / 2)
    allc["one_core"] = {k: one[k] for k in ("value", "unit", "cores", "sample")}
    return allc


def reference_arm(wl: synth.Workload, steps: int, warmup: int, world: int):
    pool = OraclePool(wl, host_cores())
    try:
        for _ in range(warmup):
            pool.step()
        spent, est = [], []
        for _ in range(steps):
            sp, e = pool.step()
            spent.append(sp)
            est.append(e)
    finally:
        pool.close()
    step_s = statistics.median(est)
    v = _tokens(wl) / step_s
    sampled = statistics.median(spent)
    return {"metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": world, "steps": steps,
            "warmup": warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
            "impl": "reference",
            "ms_per_step_is": "extrapolated from the timed sample (see extrapolation)",
            "extrapolation": {"timed_ms_per_step": sampled * 1e3,
                              "factor": step_s / sampled if sampled > 0 else None,
                              "sample": pool.desc},
            "config": {"workload": wl.name, "mode": wl.mode, "batch_per_gpu": wl.batch,
                       "context": wl.context},
            "cpu_baseline": {"value": v, "unit": "tok/s", "cores": pool.cores, "kind": "oracle",
                             "sample": pool.desc},
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def boundary(wl: synth.Workload) -> synth.Workload:
    """The same decode workload one token earlier: at p = 131,071 (3 mod 4,
    127 mod 128) every compressed layer's append emits a row, so the pooling,
    RMSNorm, rotation and insertion of both lanes run in the timed step."""
    return synth.Workload(wl.name + "_boundary", wl.seed, wl.batch, wl.layers, wl.context - 1,
                          wl.mode, wl.chunk, wl.hidden)


def summary(r: dict) -> dict:
    """The keys of another workload's line carried in the default line."""
    keys = ("value", "unit", "ms_per_step", "median_ms_per_step", "p10_p90_ms_per_step",
            "dtype", "roofline", "calls", "e2e", "clocks", "gpu_launches", "steps")
    out = {k: r[k] for k in keys if k in r}
    out["config"] = {k: r["config"][k] for k in ("workload", "mode", "batch_per_gpu", "context",
                                                  "positions", "tokens_per_step_per_gpu", "l2",
                                                  "algorithmic_GB_per_step", "step_GB/s")}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="flash43", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--streams", type=int, default=1, choices=[1, 2],
                    help="2: c4a decode layers run the indexer pipeline on a second stream")
    ap.add_argument("--paged", action="store_true",
                    help="compressed rows in 256-position blocks behind a block table")
    ap.add_argument("--qat", action="store_true",
                    help="compressor step 8 on: FP8 round trip of attention rows, FP4 QAT "
                         "round trip of indexer rows and queries")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="default workload only: skip the other workloads' keys "
                         "(c4a / c128a decode, prefill chunk, boundary step)")
    ap.add_argument("--write-traffic", metavar="NCU_CSV",
                    help="record per-call DRAM bytes of --workload from an ncu CSV and exit")
    ap.add_argument("--captured-on", default=None,
                    help="with --write-traffic: the workload the counters were taken on")
    ap.add_argument("--calls", type=int, default=1,
                    help="with --write-traffic: calls of each kind in the CSV")
    args = ap.parse_args()
    wl = WORKLOADS[args.workload]
    if args.write_traffic:
        write_traffic(args.write_traffic, args.workload, args.captured_on or wl.name, args.calls)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(reference_arm(wl, args.steps, args.warmup, world)))
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    res, R = run_gpu(args, wl, rank, world, device)
    del R
    if world == 1 and args.workload == "flash43" and not args.no_extras:
        torch.cuda.empty_cache()
        res["workloads"] = {}
        for name in ("c4a_decode", "c128a_decode", "prefill"):
            r, R = run_gpu(args, WORKLOADS[name], rank, world, device)
            del R
            torch.cuda.empty_cache()
            res["workloads"][name] = summary(r)
        r, R = run_gpu(args, boundary(wl), rank, world, device)
        del R
        torch.cuda.empty_cache()
        res["boundary_step"] = summary(r)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(wl)
        print(json.dumps(res))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
