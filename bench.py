"""Benchmark of the blockwise ring-attention hot path on GB300.

One step = the whole path over one batch of seeded synthetic input:
RoPE of Q and K (one rope_apply launch) and the fused Ring-Attention kernel
(ring_attn_fwd, P emulated ranks) on the rotated copies, all through the C ABI.
Default workload: long-context causal prefill, B=1, H=32, T=65536, d=128, bf16,
RoPE base 10000, P=16 zigzag ranks (the largest single-GPU workload).

Prints ONE JSON line (rank 0).  `value` is attention TFLOP/s counting 4*d FLOP
per visible (query, key) pair only, over the device-timed step with inputs
resident in HBM (inputs of 1.6 GB exceed the 129 MB L2, so no flush is
needed between steps).  `e2e` is the same metric through ring_attn_fwd with
host buffers: pinned host->device copies of Q, K, V and device->host copies of
out and lse inside the timed region.  `--impl reference` times the CPU oracle
on a bounded sample of the same workload.
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "attention TFLOP/s (visible pairs) and % of GB300 BF16 tensor peak; tokens/s"
DEFAULT_WORKLOAD = "zigzag_prefill_64k_rope"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--mode", default="fused", choices=["fused", "stepwise"])
    ap.add_argument("--partition", default=None, choices=["contiguous", "zigzag", "striped"],
                    help="override the workload's partition of the P ranks")
    ap.add_argument("--shard", default=None, choices=["heads"],
                    help="N > 1: split the workload's heads over the ranks (strong scaling) instead of one "
                         "replica of the whole workload per rank (weak scaling, the default)")
    ap.add_argument("--heads", type=int, default=None,
                    help="override the workload's head count (smaller cases for counter captures)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-groups", type=int, default=8, help="head / batch groups pipelined in the e2e leg")
    ap.add_argument("--e2e-split", default=None,
                    help="heads per group of the e2e leg, comma-separated (B = 1; overrides --e2e-groups); "
                         "default for B = 1 and H a multiple of 16: H/16, 3H/16, H/4, H/4, 3H/16, H/16")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches instead of CUDA graph replays")
    ap.add_argument("--seq", type=int, default=None,
                    help="override the workload's sequence length (smaller cases for counter captures)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-full", action="store_true",
                    help="time the oracle over the whole workload instead of a sample (small workloads)")
    ap.add_argument("--variant", default="ring", choices=["ring", "ulysses", "decode", "merge", "rope"],
                    help="ulysses: time ulysses_attn_fwd over P head-partitioned ranks (not the default line)")
    ap.add_argument("--direction", default="forward", choices=["forward", "backward"],
                    help="backward: time ring_attn_bwd instead (not the default bench line)")
    return ap.parse_args()


def visible_pairs(w, inp) -> int:
    """Exact count of visible (query, key) pairs over all (b, h)."""
    if w.pad_len is None and w.band is None:
        per = w.T * (w.T + 1) // 2 if w.causal else w.T * w.T
        return per * w.B * w.H
    total = 0
    T = w.T
    dev = inp.q.device
    i = torch.arange(T, device=dev).view(-1, 1)
    j = torch.arange(T, device=dev).view(1, -1)
    base = torch.ones((T, T), dtype=torch.bool, device=dev)
    if w.causal:
        base &= j <= i
    if inp.am is not None:
        base &= inp.am == 0
    for b in range(w.B):
        m = base
        if inp.kpm is not None:
            m = m & (inp.kpm[b] == 0).view(1, -1)
        total += int(m.sum().item())
    return total * w.H


KERNEL_SOURCES = ["blockwise_attention_gb300/csrc/attn_tc.cu", "blockwise_attention_gb300/csrc/tc_ptx.cuh",
                  "blockwise_attention_gb300/csrc/common.cuh",
                  "blockwise_attention_gb300/csrc/epilogue.cuh", "blockwise_attention_gb300/csrc/internal.h"]


def profiled_traffic(workload: str):
    """DRAM bytes of one attention launch from the committed ncu summary of this
    workload, or None when the kernel sources changed since it was captured."""
    import hashlib
    import re
    path = os.path.join(ROOT, "profiles", f"attn_tc_kernel_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    t = re.search(r"^traffic_bytes:\s*(\d+)", text, re.M)
    h = re.search(r"^source_sha256:\s*([0-9a-f]+)", text, re.M)
    if not t or not h:
        return None
    sha = hashlib.sha256()
    for src in KERNEL_SOURCES:
        with open(os.path.join(ROOT, src), "rb") as f:
            sha.update(f.read())
    return int(t.group(1)) if sha.hexdigest() == h.group(1) else None


# Dense bf16 tensor throughput of one SM per clock: one 128 x 128 x 16 MMA
# (kind::f16, cta_group::1) every 64 cycles, as measured on this part.
TENSOR_FLOP_PER_CLK_SM = 2 * 128 * 128 * 16 // 64
NUM_SMS = 152


def graphed(fn, dev, enabled=True):
    """fn captured into a CUDA graph (returned as a callable that replays it), or
    fn itself when capture is disabled or refused."""
    if not enabled:
        return fn, False
    try:
        cur = torch.cuda.current_stream(dev)
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(cur)
        with torch.cuda.stream(cap):
            fn()
        cur.wait_stream(cap)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap, capture_error_mode="relaxed"):
            fn()
        torch.cuda.synchronize()
        return g.replay, True
    except Exception as e:  # noqa: BLE001
        print(f"graph capture unavailable ({e}); timing eager launches", file=sys.stderr)
        return fn, False


def tensor_roofline(achieved, peaks, peak_src, clocks, timed_s):
    """Roofline object of a tensor-bound kernel.  It is graded against the
    measured burst bf16 peak (a cuBLAS GEMM timed best-of-10): the timed region
    lasts well under a second, while the measured sustained peak describes a
    GEMM looped for seconds under the power cap at a lower clock.  The
    clock-derived tensor peak at the sampled SM clock is given beside it."""
    burst = float(peaks["bf16_tflops"])
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    mhz = (clocks or {}).get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
    at_clock = TENSOR_FLOP_PER_CLK_SM * NUM_SMS * mhz * 1e6 / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": burst, "unit": "TFLOP/s", "frac": achieved / burst,
            "peak_source": f"{peak_src} bf16_tflops (burst; the timed region lasts {timed_s:.2f} s)",
            "frac_of_sustained_peak": achieved / sustained,
            "tensor_peak_at_clock": at_clock, "frac_of_peak_at_clock": achieved / at_clock,
            "peak_at_clock_source": f"{TENSOR_FLOP_PER_CLK_SM} FLOP/clk/SM x {NUM_SMS} SMs x median SM clock "
                                    f"{mhz:.0f} MHz"}


def e2e_groups(B: int, H: int, n_groups: int = 8, split=None):
    """Index tuples of the groups the e2e leg pipelines, one ring_attn_fwd call
    each.  B = 1: groups of heads, by default H/16, 3H/16, H/4, H/4, 3H/16, H/16
    when H is a multiple of 16 and eight groups are asked for (small first and
    last groups: the first group's inputs and the last group's outputs cross the
    host link while nothing else runs), else `split` (heads per group) or n_groups
    equal groups.  Otherwise groups of batch items, or the whole tensor."""
    if split is None and B == 1 and H % 16 == 0 and n_groups == 8:
        u = H // 16
        split = [u, 3 * u, 4 * u, 4 * u, 3 * u, u]
    if split and B == 1 and sum(split) == H and min(split) > 0:
        edges = [0]
        for x in split:
            edges.append(edges[-1] + x)
        return [(slice(None), slice(edges[i], edges[i + 1])) for i in range(len(split))]
    if B == 1 and H % n_groups == 0:
        return [(slice(None), slice(i * H // n_groups, (i + 1) * H // n_groups)) for i in range(n_groups)]
    if B % n_groups == 0:
        return [(slice(i * B // n_groups, (i + 1) * B // n_groups),) for i in range(n_groups)]
    return [(slice(None),)]


def shard_heads(H: int, world: int, rank: int):
    """Heads [h0, h1) of rank `rank` when the H heads of one workload are split
    over `world` ranks: contiguous, as even as possible (the first H % world ranks
    take one more).  Heads are independent problems, so no data moves between
    ranks."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank / world")
    base, extra = divmod(H, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of a per-rank scalar over all ranks (identity for one rank)."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.samples = []
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(self.dev).uuid)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                          "-lms", "200", "-i", uuid], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in self.samples:
            try:
                mhz.append(float(s[1].split()[0]))
                mx = float(s[2].split()[0])
                for n, v in zip(names, s[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


def oracle_cpu_baseline(w, inp_cpu_head, seconds, kpm=None, am=None):
    """Time the oracle, as it stands, on sampled query rows of one head (each
    row over its full key range, with the workload's exclusions), RoPE
    included.  kpm: (1, T) key-padding row of that head's batch item; am:
    (T, T).  Returns the JSON object for `cpu_baseline`."""
    import oracle
    q, k, v = inp_cpu_head            # (1, 1, T, d) float32 tensors on the CPU
    T, d = w.T, w.d
    threads = oracle.default_threads()
    rng = np.random.default_rng(0)

    def rope_head():
        if w.rope_base is None:
            return q, k
        return (oracle.rope(q, base=w.rope_base, round_to=w.dtype),
                oracle.rope(k, base=w.rope_base, round_to=w.dtype))

    vis = None
    if kpm is not None or am is not None:
        vis = np.ones((T, T), dtype=bool)
        if w.causal:
            vis &= np.tri(T, dtype=bool)
        if kpm is not None:
            vis &= (np.asarray(kpm).reshape(-1)[:T] == 0)[None, :]
        if am is not None:
            vis &= np.asarray(am) == 0

    def attend(qr, kr, nrows):
        rows = np.sort(rng.choice(T, size=nrows, replace=False)).astype(np.int64)
        oracle.attention(qr, kr, v, causal=w.causal, kpm=kpm, am=am, rows=rows, nthreads=threads)
        if vis is not None:
            return int(vis[rows].sum())
        return int((rows + 1).sum()) if w.causal else nrows * T

    # calibrate: RoPE of the head is a fixed cost, attention scales with the rows
    t0 = time.perf_counter()
    qr, kr = rope_head()
    t_rope = time.perf_counter() - t0
    t0 = time.perf_counter()
    p_cal = attend(qr, kr, threads)
    rate = p_cal / max(time.perf_counter() - t0, 1e-6)
    budget = max(seconds - t_rope, 0.25 * seconds)
    n = int(min(T, max(threads, threads * round(budget * rate / (T / 2) / threads))))
    # timed sample: RoPE of the head plus n rows
    t0 = time.perf_counter()
    qr, kr = rope_head()
    pairs = attend(qr, kr, n)
    dt = time.perf_counter() - t0
    flops = 4.0 * d * pairs
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} random query rows of one head (b=0, h=0) of {w.name}, each over its full "
                      f"key range with the workload's exclusions, RoPE of that head's Q and K included "
                      f"when the workload rotates; {pairs} visible pairs in {dt:.2f} s"}


def oracle_full_baseline(w, inp):
    """Time the oracle, as it stands, over the whole workload (every row of
    every head, RoPE included) on the host's cores."""
    import oracle
    threads = oracle.default_threads()
    q, k, v = inp.q.float().cpu(), inp.k.float().cpu(), inp.v.float().cpu()
    kpm = None if inp.kpm is None else inp.kpm.cpu()
    am = None if inp.am is None else inp.am.cpu()
    t0 = time.perf_counter()
    if w.rope_base is not None:
        q = torch.from_numpy(oracle.rope(q, base=w.rope_base, round_to=w.dtype))
        k = torch.from_numpy(oracle.rope(k, base=w.rope_base, round_to=w.dtype))
    oracle.attention(q, k, v, causal=w.causal, kpm=kpm, am=am, nthreads=threads)
    dt = time.perf_counter() - t0
    flops = 4.0 * w.d * visible_pairs(w, inp)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"the full workload {w.name}: all {w.B * w.H * w.T} rows, RoPE included when the "
                      f"workload rotates, in {dt:.2f} s"}


def reference_arm(args, w, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    kpm = am = None
    if w.B * w.H * w.T * w.d <= (1 << 26):
        # small workloads: the seeded inputs themselves, head (0, 0) with its masks
        from blockwise_attention_gb300.workloads import make_inputs
        inp = make_inputs(w, "cpu")
        qkv = [x[0:1, 0:1].float() for x in (inp.q, inp.k, inp.v)]
        kpm = None if inp.kpm is None else inp.kpm[0:1]
        am = inp.am
    else:
        # one head of the same distribution (the full tensors take minutes to draw here)
        g = torch.Generator().manual_seed(1000 + w.index)
        shape = (1, 1, w.T, w.d)
        qkv = []
        for _ in range(3):
            x = torch.randn(shape, generator=g) * w.std
            qkv.append(x.to(w.torch_dtype).float())
    times, last = [], None
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        last = oracle_cpu_baseline(w, qkv, seconds=max(2.0, args.cpu_seconds / 2), kpm=kpm, am=am)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    value = last["value"]
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d": w.d,
                                            "P": w.P, "partition": w.partition, "causal": w.causal,
                                            "rope_base": w.rope_base},
            "cpu_baseline": {k: last[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def native_arm(args, w, rank, world, local_rank):
    import blockwise_attention_gb300 as ba
    from blockwise_attention_gb300.workloads import make_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ba.load()
    inp = make_inputs(w, dev)
    rope = w.rope_base is not None
    pairs = visible_pairs(w, inp)
    flops = 4.0 * w.d * pairs
    stream = torch.cuda.current_stream(dev)

    qr = torch.empty_like(inp.q)
    kr = torch.empty_like(inp.k)
    out = torch.empty_like(inp.q)
    lse = torch.empty(inp.q.shape[:3], dtype=torch.float32, device=dev)
    ws_need = ba.ring_attn_fwd_workspace_size(w.B, w.H, w.T, w.d, inp.q.dtype, w.P, w.partition, args.mode,
                                              inp.kpm is not None or inp.am is not None, False)
    ws = torch.empty(max(ws_need, 1), dtype=torch.uint8, device=dev)

    def do_rope():
        ba.rope_apply(inp.q, x2=inp.k, base=w.rope_base, out=qr, out2=kr)

    def do_attn():
        q_in, k_in = (qr, kr) if rope else (inp.q, inp.k)
        ba.ring_attn_fwd(q_in, k_in, inp.v, P=w.P, partition=w.partition, mode=args.mode,
                         key_padding_mask=inp.kpm, attn_mask=inp.am, causal=w.causal, out=out, lse=lse,
                         workspace=ws)

    def step():
        if rope:
            do_rope()
        do_attn()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    rc = ba.sync_status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} after warm-up")

    # The step, and each of its two calls alone, captured once into CUDA graphs and
    # replayed: the launches of the small workloads would otherwise be timed as host
    # gaps between kernels (the 64K step is 21 ms of kernels either way).  Eager
    # launches if the capture is refused.
    graphs = {}
    if not args.no_graph:
        try:
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            with torch.cuda.stream(cap):
                step()
            stream.wait_stream(cap)
            for name, fn in (("step", step), ("attn", do_attn)) + ((("rope", do_rope),) if rope else ()):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap, capture_error_mode="relaxed"):
                    fn()
                graphs[name] = g
            torch.cuda.synchronize()
        except Exception as e:  # noqa: BLE001
            print(f"graph capture unavailable ({e}); timing eager launches", file=sys.stderr)
            graphs = {}

    def run(name, fn):
        if name in graphs:
            graphs[name].replay()
        else:
            fn()

    def timed(name, fn):
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        for _ in range(args.steps):
            run(name, fn)
        b_.record(stream)
        torch.cuda.synchronize()
        return a_.elapsed_time(b_) / args.steps

    for name, fn in (("step", step), ("attn", do_attn)) + ((("rope", do_rope),) if rope else ()):
        run(name, fn)   # each graph once before its timed loop
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.5)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        run("step", step)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop() if sampler else None
    total_ms = t_start.elapsed_time(t_end)
    # the dominant kernel and RoPE alone, each over the same number of steps
    attn_ms = [timed("attn", do_attn)]
    rope_ms = [timed("rope", do_rope)] if rope else [0.0]
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_step = total_ms / args.steps
    value = world * flops / (ms_step * 1e-3) / 1e12
    kernels_per_step = (1 if rope else 0) + (1 if args.mode == "fused" else w.P) + \
        (1 if (inp.kpm is not None or inp.am is not None) else 0)

    # end to end through the one-call API with host buffers
    e2e = None
    if not args.no_e2e:
        qh = inp.q.cpu().pin_memory()
        kh = inp.k.cpu().pin_memory()
        vh = inp.v.cpu().pin_memory()
        oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lh = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        qd, kd, vd = torch.empty_like(inp.q), torch.empty_like(inp.k), torch.empty_like(inp.v)
        ws_e = ba.ring_attn_fwd_workspace_size(w.B, w.H, w.T, w.d, inp.q.dtype, w.P, w.partition, args.mode,
                                               inp.kpm is not None or inp.am is not None, rope)
        # two compute streams, each with its own workspace: the next group's launch
        # fills the SMs as the current group's last work items drain
        wse = [torch.empty(max(ws_e, 1), dtype=torch.uint8, device=dev) for _ in range(2)]

        # Independent groups of heads (B == 1) or batch items are pipelined over four
        # streams: host->device copy of group g+1 and device->host copy of group g-1
        # run while group g computes, each group one ring_attn_fwd call, the groups
        # alternating between two compute streams.
        split = [int(x) for x in args.e2e_split.split(",")] if args.e2e_split else None
        sl = e2e_groups(w.B, w.H, args.e2e_groups, split)
        n_groups = len(sl)
        heads_per_group = [ix[1].stop - ix[1].start for ix in sl] if w.B == 1 and len(sl[0]) == 2 else None
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        s_comp = [stream, torch.cuda.Stream(dev)]
        ev_in = [torch.cuda.Event() for _ in range(n_groups)]
        ev_comp = [torch.cuda.Event() for _ in range(n_groups)]
        ev_out = [torch.cuda.Event() for _ in range(n_groups)]
        started = [False]

        def e2e_step():
            for i, ix in enumerate(sl):
                kpm_i = inp.kpm[ix[0]] if inp.kpm is not None else None
                with torch.cuda.stream(s_in):
                    if started[0]:
                        s_in.wait_event(ev_comp[i])      # previous step's compute read these inputs
                    qd[ix].copy_(qh[ix], non_blocking=True)
                    kd[ix].copy_(kh[ix], non_blocking=True)
                    vd[ix].copy_(vh[ix], non_blocking=True)
                    ev_in[i].record(s_in)
                cs = s_comp[i % 2]
                cs.wait_event(ev_in[i])
                if started[0]:
                    cs.wait_event(ev_out[i])             # previous step's copy-out read these outputs
                ba.ring_attn_fwd(qd[ix], kd[ix], vd[ix], P=w.P, partition=w.partition, mode=args.mode,
                                 key_padding_mask=kpm_i, attn_mask=inp.am, causal=w.causal, rope=rope,
                                 rope_base=w.rope_base or 10000.0, out=out[ix], lse=lse[ix], workspace=wse[i % 2],
                                 stream=cs)
                ev_comp[i].record(cs)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_comp[i])
                    oh[ix].copy_(out[ix], non_blocking=True)
                    lh[ix].copy_(lse[ix], non_blocking=True)
                    ev_out[i].record(s_out)
            started[0] = True

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_in)            # the first operation of a step is a copy on s_in
        for _ in range(args.steps):
            e2e_step()
        for cs in s_comp:
            s_out.wait_stream(cs)
        b.record(s_out)           # the last copy-out of the last step
        torch.cuda.synchronize()
        barrier()
        e_ms = a.elapsed_time(b) / args.steps
        e_ms = max_over_ranks(e_ms, world, dev)
        h2d = sum(x.numel() * x.element_size() for x in (qh, kh, vh))
        d2h = oh.numel() * oh.element_size() + lh.numel() * 4
        e2e = {"value": world * flops / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms, "pipeline_groups": n_groups}
        if heads_per_group:
            e2e["heads_per_group"] = heads_per_group
        del qh, kh, vh, qd, kd, vd, wse

    if ba.sync_status() != 0:
        raise RuntimeError("device status error after the timed region")
    if rank != 0:
        return

    peaks, peak_src = load_peaks()
    attn_avg = statistics.mean(attn_ms)
    achieved = flops / (attn_avg * 1e-3) / 1e12
    roof = tensor_roofline(achieved, peaks, peak_src, clocks, args.steps * ms_step / 1e3)
    roof.update({"traffic": profiled_traffic(w.name), "kernel": f"attn_tc_kernel<{w.d}>", "kernel_ms": attn_avg})
    cpu = None
    if not args.no_cpu and world == 1 or (not args.no_cpu and rank == 0 and world == 1):
        if args.cpu_full:
            cpu = oracle_full_baseline(w, inp)
        else:
            head = (inp.q[0:1, 0:1].float().cpu(), inp.k[0:1, 0:1].float().cpu(), inp.v[0:1, 0:1].float().cpu())
            cpu = oracle_cpu_baseline(w, head, args.cpu_seconds,
                                      kpm=None if inp.kpm is None else inp.kpm[0:1].cpu(),
                                      am=None if inp.am is None else inp.am.cpu())
    # --shard heads: the ranks together process one workload (value: its FLOPs over
    # the slowest rank's time); otherwise each rank processes a whole replica
    sharded = getattr(args, "shard", None) == "heads" and world > 1
    full = getattr(args, "full_workload", w)
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "strong" if sharded else "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": full.name if sharded else w.name, "B": w.B, "H": full.H if sharded else w.H,
                       "T": w.T, "d": w.d, "P": w.P,
                       "parallelism": f"heads split over {world} ranks" if sharded else f"{world} replica(s)",
                       "partition": w.partition, "causal": w.causal, "rope_base": w.rope_base,
                       "mode": args.mode, "visible_pairs": pairs, "flops_per_step": flops,
                       "launch": "CUDA graph replay" if graphs else "eager",
                       "l2": "inputs (Q, K, V: 1.6 GB) larger than the 129 MB L2; no flush"},
            "tokens_per_s": (1 if sharded else world) * w.B * w.T / (ms_step * 1e-3),
            "pct_of_bf16_peak": 100.0 * value / roof["peak"],
            "rope_ms": statistics.mean(rope_ms),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": kernels_per_step * args.steps}
    print(json.dumps(line), flush=True)


BWD_METRIC = "attention backward TFLOP/s (10*d FLOP per visible pair: QK^T, dout V^T, dV, dK, dQ)"


def backward_arm(args, w, rank, world, local_rank):
    """Time ring_attn_bwd (fused) on the workload; out and lse come from one
    forward before the timed region.  The kernels run on the CUDA cores in fp32,
    so the roofline is the fp32 FMA peak (152 SMs x 128 lanes x 2 FLOP x clock)."""
    import blockwise_attention_gb300 as ba
    from blockwise_attention_gb300.workloads import make_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ba.load()
    inp = make_inputs(w, dev)
    if w.rope_base is not None:
        q, k = ba.rope_apply(inp.q, x2=inp.k, base=w.rope_base)
    else:
        q, k = inp.q, inp.k
    out, lse = ba.ring_attn_fwd(q, k, inp.v, P=w.P, partition=w.partition, key_padding_mask=inp.kpm,
                                attn_mask=inp.am, causal=w.causal)
    g = torch.Generator(device="cpu").manual_seed(2000 + w.index)
    dout = torch.randn(inp.q.shape, generator=g).to(inp.q.dtype).to(dev)
    dq = torch.empty(inp.q.shape, dtype=torch.float32, device=dev)
    dk, dv = torch.empty_like(dq), torch.empty_like(dq)
    need = ba.load().ring_attn_bwd_workspace_size(w.B, w.H, w.T)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    pairs = visible_pairs(w, inp)
    flops = 10.0 * w.d * pairs
    stream = torch.cuda.current_stream(dev)

    def step():
        ba.ring_attn_bwd(q, k, inp.v, out, dout, lse, P=w.P, partition=w.partition, mode=args.mode,
                         key_padding_mask=inp.kpm, attn_mask=inp.am, causal=w.causal, dq=dq, dk=dk, dv=dv,
                         workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ba.sync_status() != 0:
        raise RuntimeError("device status error after warm-up")
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.5)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(a.elapsed_time(b) / args.steps, world, dev)
    if rank != 0:
        return
    value = world * flops / (ms * 1e-3) / 1e12
    sm_mhz = (clocks or {}).get("sm_mhz") or 2070.0
    tensor_path = w.torch_dtype == torch.bfloat16 and w.d in (64, 128)
    if tensor_path:
        peaks, src = load_peaks()
        roof = tensor_roofline(value, peaks, src, clocks, args.steps * ms / 1e3)
        roof.update({"traffic": None, "kernel": "bwd_dkdv_tc_kernel + bwd_dq_tc_kernel",
                     "executed_frac": 1.4 * value / roof["peak"],
                     "executed_note": "the kernels execute 14*d FLOP per pair (QK^T and dout V^T are formed in "
                                      "both) against the 10*d counted"})
    else:
        peak = 152 * 128 * 2 * sm_mhz * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": value, "peak": peak, "unit": "TFLOP/s", "frac": value / peak,
                "traffic": None, "kernel": "bwd_dkdv_kernel + bwd_dq_kernel",
                "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 FLOP x sampled SM clock; the kernels "
                               "execute 14*d FLOP per pair (scores and dout V^T in both)"}
    steps_per = 1 if args.mode == "fused" else w.P
    cpu = None
    if not args.no_cpu:
        import oracle
        oracle.build()
        n = min(w.T, 2048)
        sl = (slice(0, 1), slice(0, 1), slice(0, n))
        t0 = time.perf_counter()
        oracle.attention_bwd(q[sl].float().cpu(), k[sl].float().cpu(), inp.v[sl].float().cpu(),
                             dout[sl].float().cpu(), causal=w.causal)
        dt = time.perf_counter() - t0
        cpairs = n * (n + 1) // 2 if w.causal else n * n
        cpu = {"value": 10.0 * w.d * cpairs / dt / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": f"backward of the first {n} tokens of one head (b=0, h=0) of {w.name}, "
                         f"{cpairs} visible pairs in {dt:.2f} s (one thread per head)"}
    line = {"metric": BWD_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if tensor_path else "f32", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d": w.d, "P": w.P,
                       "partition": w.partition, "causal": w.causal, "mode": args.mode, "direction": "backward",
                       "visible_pairs": pairs, "flops_per_step": flops,
                       "l2": "inputs larger than the 129 MB L2; no flush"},
            "roofline": roof,
            "cpu_baseline": cpu, "e2e": None, "clocks": clocks,
            "gpu_launches": 3 * steps_per * args.steps}
    if not tensor_path:
        line["dtype"] = "f32"
    print(json.dumps(line), flush=True)


def ulysses_arm(args, w, rank, world, local_rank):
    """Time ulysses_attn_fwd on token shards (P, H, B, T/P, d): three exchanges,
    one attention launch, and the reverse exchange of out and lse.  `value` is
    attention TFLOP/s over visible pairs for the whole step; `roofline` is the
    exchange kernel against the measured HBM copy peak (it reads and writes each
    byte once)."""
    import blockwise_attention_gb300 as ba
    from blockwise_attention_gb300.workloads import make_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ba.load()
    inp = make_inputs(w, dev)
    P = w.P
    if w.H % P:
        raise SystemExit(f"ulysses needs P | H ({w.name}: H={w.H}, P={P})")

    def to_tok(x):
        B, H, T, d = x.shape
        return x.permute(1, 0, 2, 3).reshape(H, B, P, T // P, d).permute(2, 0, 1, 3, 4).contiguous()

    qt, kt, vt = to_tok(inp.q), to_tok(inp.k), to_tok(inp.v)
    out = torch.empty_like(qt)
    lse = torch.empty(qt.shape[:4], dtype=torch.float32, device=dev)
    need = ba.load().ulysses_attn_fwd_workspace_size(P, w.H, w.B, w.T, w.d, 1 if w.torch_dtype == torch.bfloat16
                                                      else 0, int(inp.kpm is not None or inp.am is not None))
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    head = torch.empty((P, w.H // P, w.B, w.T, w.d), dtype=qt.dtype, device=dev)
    pairs = visible_pairs(w, inp)
    flops = 4.0 * w.d * pairs
    stream = torch.cuda.current_stream(dev)

    def step():
        ba.ulysses_attn_fwd(qt, kt, vt, key_padding_mask=inp.kpm, attn_mask=inp.am, causal=w.causal, out=out,
                            lse=lse, workspace=ws)

    for _ in range(args.warmup):
        step()
        ba.ulysses_all_to_all(qt, P, "token_to_head", out=head)
    torch.cuda.synchronize()
    if ba.sync_status() != 0:
        raise RuntimeError("device status error after warm-up")
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.5)
    a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    for _ in range(args.steps):
        ba.ulysses_all_to_all(qt, P, "token_to_head", out=head)
    c.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(a.elapsed_time(b) / args.steps, world, dev)
    a2a_ms = b.elapsed_time(c) / args.steps
    if rank != 0:
        return
    peaks, src = load_peaks()
    a2a_bytes = 2.0 * qt.numel() * qt.element_size()
    achieved = a2a_bytes / (a2a_ms * 1e-3) / 1e9
    value = world * flops / (ms * 1e-3) / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if qt.dtype == torch.bfloat16 else "f32", "data": "synthetic",
            "config": {"workload": w.name, "variant": "ulysses", "B": w.B, "H": w.H, "T": w.T, "d": w.d, "P": P,
                       "causal": w.causal, "visible_pairs": pairs, "flops_per_step": flops,
                       "l2": "inputs larger than the 129 MB L2; no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": None, "kernel": "a2a_span_kernel (token->head)",
                         "algorithmic_bytes": a2a_bytes, "kernel_ms": a2a_ms,
                         "peak_source": f"{src} hbm_gbs (copy)"},
            "cpu_baseline": None, "e2e": None, "clocks": clocks, "gpu_launches": 7 * args.steps}
    print(json.dumps(line), flush=True)


def merge_arm(args, w, rank, world, local_rank):
    """Time attn_merge, the LSE merge of two fp32 partial attentions (the page's
    accumulate_out_and_lse), over every row of the workload: (B*H*T, d) fp32
    partials and (B*H*T) LSEs.  Bound by HBM: per row it reads both partials
    and both LSEs and writes one of each, (3d + 3) * 4 bytes."""
    import blockwise_attention_gb300 as ba

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ba.load()
    rows, d = w.B * w.H * w.T, w.d
    g = torch.Generator(device=dev).manual_seed(3000 + w.index)
    oa = torch.randn((rows, d), generator=g, device=dev)
    ob = torch.randn((rows, d), generator=g, device=dev)
    la = torch.randn((rows,), generator=g, device=dev) * 4
    lb = torch.randn((rows,), generator=g, device=dev) * 4
    stream = torch.cuda.current_stream(dev)

    def step():
        ba.attn_merge(oa, la, ob, lb)

    for _ in range(args.warmup):
        step()
    step, in_graph = graphed(step, dev, not args.no_graph)
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    if sampler:
        sampler.start()
        time.sleep(0.5)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(a.elapsed_time(b) / args.steps, world, dev)
    if rank != 0:
        return
    peaks, src = load_peaks()
    nbytes = float(rows) * (3 * d + 3) * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    line = {"metric": "LSE merge of partial attentions: HBM GB/s ((3d+3)*4 bytes per row)",
            "value": world * gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": f"merge_rows_of_{w.name}", "rows": rows, "d": d, "bytes_per_step": nbytes,
                       "launch": "CUDA graph replay" if in_graph else "eager",
                       "l2": f"partials ({2 * rows * d * 4 / 1e9:.2f} GB) far larger than the 129 MB L2; no flush"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": None, "kernel": "merge_kernel",
                         "algorithmic_bytes": nbytes, "kernel_ms": ms, "peak_source": f"{src} hbm_gbs (copy)"},
            "cpu_baseline": None, "e2e": None, "clocks": clocks, "gpu_launches": args.steps}
    print(json.dumps(line), flush=True)


def rope_arm(args, w, rank, world, local_rank):
    """Time rope_apply on the workload's Q and K (one launch for both), bf16 in
    and out.  Bound by HBM: 2 bytes read and 2 written per element and tensor."""
    import blockwise_attention_gb300 as ba
    from blockwise_attention_gb300.workloads import make_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ba.load()
    inp = make_inputs(w, dev)
    qr, kr = torch.empty_like(inp.q), torch.empty_like(inp.k)
    base = w.rope_base or 10000.0
    stream = torch.cuda.current_stream(dev)

    def step():
        ba.rope_apply(inp.q, x2=inp.k, base=base, out=qr, out2=kr)

    for _ in range(args.warmup):
        step()
    step, in_graph = graphed(step, dev, not args.no_graph)
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    if sampler:
        sampler.start()
        time.sleep(0.5)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(a.elapsed_time(b) / args.steps, world, dev)
    if rank != 0:
        return
    peaks, src = load_peaks()
    nbytes = 2.0 * inp.q.numel() * inp.q.element_size() * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    line = {"metric": "RoPE of Q and K: HBM GB/s (read + write of both tensors)",
            "value": world * gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": f"rope_of_{w.name}", "B": w.B, "H": w.H, "T": w.T, "d": w.d, "base": base,
                       "bytes_per_step": nbytes, "launch": "CUDA graph replay" if in_graph else "eager",
                       "l2": f"Q and K ({nbytes / 2e9:.2f} GB) larger than the 129 MB L2; no flush"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": None, "kernel": "rope_bf16_kernel",
                         "algorithmic_bytes": nbytes, "kernel_ms": ms, "peak_source": f"{src} hbm_gbs (copy)"},
            "cpu_baseline": None, "e2e": None, "clocks": clocks, "gpu_launches": args.steps}
    print(json.dumps(line), flush=True)


def decode_arm(args, rank, world, local_rank):
    """Time attn_decode_fwd on the decode workload (one query token per sequence,
    B=8, H=32, d=128, bf16, 64K-slot cache with ragged lengths).  Bound by HBM:
    `value` is the cache bytes read per second (every valid K and V byte once),
    against the measured HBM copy peak."""
    import blockwise_attention_gb300 as ba
    from blockwise_attention_gb300.workloads import DECODE, make_decode_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ba.load()
    inp = make_decode_inputs(dev)
    B, H, S, d = inp.k.shape
    out = torch.empty((B, H, 1, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, 1), dtype=torch.float32, device=dev)
    need = ba.load().attn_decode_workspace_size(B, H, S, d, 0)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    total_len = int(inp.lengths.sum().item())
    kv_bytes = 2.0 * total_len * H * d * 2
    io_bytes = kv_bytes + 2.0 * B * H * d * 2 + B * H * 4
    stream = torch.cuda.current_stream(dev)

    def step():
        ba.attn_decode_fwd(inp.q, inp.k, inp.v, lengths=inp.lengths, out=out, lse=lse, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ba.sync_status() != 0:
        raise RuntimeError("device status error after warm-up")
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.5)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(a.elapsed_time(b) / args.steps, world, dev)
    if rank != 0:
        return
    peaks, src = load_peaks()
    gbs = io_bytes / (ms * 1e-3) / 1e9
    line = {"metric": "decode attention: KV-cache bytes read per second (one query token per sequence)",
            "value": world * gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "decode_kv_64k", **{k: v for k, v in DECODE.items() if k != "seed"},
                       "valid_keys_total": total_len, "bytes_per_step": io_bytes,
                       "l2": "cache (8.6 GB) far larger than the 129 MB L2; no flush"},
            "tokens_per_s": world * B / (ms * 1e-3),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                         "kernel": "decode_split_kernel + decode_combine_kernel",
                         "peak_source": f"{src} hbm_gbs (copy)"},
            "cpu_baseline": None, "e2e": None, "clocks": clocks, "gpu_launches": 2 * args.steps}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    from blockwise_attention_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.partition:
        w = w.replace(partition=args.partition)
    if args.heads:
        w = w.replace(H=args.heads, name=f"{w.name}_h{args.heads}")
    if args.seq:
        w = w.replace(T=args.seq, name=f"{w.name}_t{args.seq}")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    args.full_workload = w
    if args.shard == "heads" and world > 1:
        if w.H % world:
            raise SystemExit(f"--shard heads: {w.H} heads do not split evenly over {world} ranks")
        h0, h1 = shard_heads(w.H, world, rank)
        # this rank's heads only (synthetic inputs of that shape, seeded per rank)
        w = w.replace(H=h1 - h0, index=w.index + 7919 * rank, name=f"{w.name}_heads{h0}-{h1}")
    if args.impl == "reference":
        reference_arm(args, w, rank, world)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    try:
        if args.direction == "backward":
            backward_arm(args, w, rank, world, local_rank)
        elif args.variant == "ulysses":
            ulysses_arm(args, w, rank, world, local_rank)
        elif args.variant == "decode":
            decode_arm(args, rank, world, local_rank)
        elif args.variant == "merge":
            merge_arm(args, w, rank, world, local_rank)
        elif args.variant == "rope":
            rope_arm(args, w, rank, world, local_rank)
        else:
            native_arm(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
