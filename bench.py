"""Benchmark of the load-balanced block-sparse attention forward path on GB300.

One step = one pass of the whole hot path over the LLM-heads workload
(B=1, H=32, S=8192, d=128, block=128, causal; 16 global heads Bernoulli(0.9)
below the diagonal, 16 local heads = window of 4 blocks + block-0 sink):
mask loads -> LPT plan over (b, h, q-block) items, one worker per SM ->
block-sparse attention forward (bf16 out + fp32 LSE).

Metric: effective TFLOP/s over computed dense blocks, 4 * block^2 * d FLOP per
dense block (diagonal blocks counted in full), reported with its fraction of the
measured bf16 dense tensor-core peak and the per-worker (per-SM) busy-time skew.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
With N > 1 (torchrun, one rank per GPU) every rank runs the same workload as an
independent replica (weak scaling; the path has no exchange step).
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "llm"
METRIC = "block-sparse attn fwd TFLOP/s on dense blocks, % of bf16 TC peak, SM skew"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) of one attention launch on this workload, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), valid only for the kernel source it was
# taken on: any other attn.cu reports null.
NCU_ATTN_TRAFFIC = {"attn_sha256_prefix": "d693011cd448583d", "bytes": 313.17e6}


def attn_traffic():
    """Profiled bytes per launch, or None when attn.cu changed since the capture."""
    import hashlib

    path = os.path.join(ROOT, "load_balancing_gb300", "csrc", "attn.cu")
    with open(path, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    return NCU_ATTN_TRAFFIC["bytes"] if sha.startswith(NCU_ATTN_TRAFFIC["attn_sha256_prefix"]) else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


MASK_TEXT = {
    "tiny": "8x8 Bernoulli(0.5) block mask per head, diagonal forced",
    "llm": "heads 0-15 Bernoulli(0.9) below the diagonal + diagonal, heads 16-31 window of 4 blocks + "
           "block-0 sink",
    "video": "16 frames x 1024 tokens; heads 0-11 same-frame blocks, heads 12-23 same in-frame offset, "
             "OR Bernoulli(rho_h), rho_h ~ U[0.05, 0.40]",
    "sharded": "full lower-triangular block mask; 8 contiguous / 8 striped KV shards",
    "imbalance": "per-head density lognormal(ln 0.1, 1) clipped to [1%, 60%], uniform block positions per "
                 "row, diagonal forced",
}


def workload_description(w):
    return (f"{w.name}: B={w.B} H={w.H} S={w.S} d={w.d} block={w.block} causal={int(w.causal)}; "
            f"{MASK_TEXT.get(w.name, w.kind)}; Q/K/V bf16 N(0,1)")


def bench_config(w, n_workers, n_dense, world=1):
    """The ``config`` object of the JSON line; both arms print the same one."""
    return {"workload": workload_description(w), "n_workers": n_workers, "worklist": "LPT",
            "plan_cost": "dense blocks per item (block_cost 1, item_cost 0); shard passes add "
                         "an item cost of 4 blocks, fitted from cta_timing",
            "dense_blocks": n_dense, "items": w.n_items,
            "l2": "flushed by a 256 MiB write before every timed GPU step (outside the events)",
            "step": "pipelined: batch i's attention runs on n_workers persistent CTAs (one per SM but one) "
                    "while the mask loads and LPT plan of batch i+1 run on the remaining SM, into the "
                    "second of two plan buffers; each timed step holds one attention and one loads + plan",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def attention_workers(n_sm):
    """Persistent attention CTAs of the timed step: one per SM but one, which runs the next
    batch's mask loads and plan meanwhile."""
    return max(1, n_sm - 1)


def dense_blocks(mask_np, causal):
    m = mask_np != 0
    if causal:
        m = m & np.tril(np.ones(m.shape[-2:], dtype=bool))
    return int(m.sum())


def diag_blocks(mask_np):
    n = min(mask_np.shape[-2:])
    return int((mask_np[..., np.arange(n), np.arange(n)] != 0).sum())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


class NvmlPoller:
    """SM clock and clock-event reasons read through NVML every millisecond while the
    timed region runs (read-only queries; nothing is set). The timed region of a default
    run lasts a few milliseconds, shorter than nvidia-smi's shortest sampling interval."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, device):
        import ctypes
        import threading

        self.ok = False
        self.samples, self.reasons = [], 0
        self._stop = threading.Event()
        self._thread = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            handle = ctypes.c_void_p()
            uuid = None
            try:
                import torch

                uuid = str(torch.cuda.get_device_properties(device).uuid)
            except Exception:
                pass
            found = False
            if uuid:
                key = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
                found = nv.nvmlDeviceGetHandleByUUID(key.encode(), ctypes.byref(handle)) == 0
            if not found:
                found = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device.index or 0), ctypes.byref(handle)) == 0
            if not found:
                return
            self._reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if nv.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0 else None
            self.nv, self.handle, self.ctypes = nv, handle, ctypes
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _run(self):
        c = self.ctypes
        mhz, rs = c.c_uint(), c.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.handle, 1, c.byref(mhz)) == 0:  # NVML_CLOCK_SM
                self.samples.append(float(mhz.value))
            if self._reason_fn(self.handle, c.byref(rs)) == 0:
                self.reasons |= int(rs.value)
            time.sleep(0.001)

    def start(self):
        import threading

        if self.ok:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def stop(self):
        if not self.ok or self._thread is None:
            return None
        self._stop.set()
        self._thread.join(timeout=5)
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for bit, n in self.REASONS.items() if self.reasons & bit),
                "samples": len(self.samples), "source": "NVML, every 1 ms during the timed steps"}


# ----------------------------------------------------------------------------- distributed
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle timing
def time_oracle(w, mask_np, q, k, v, heads, budget_s=None):
    """Oracle (fp64 CPU) on whole heads of the workload; returns (seconds, effective FLOP)."""
    from oracle import attention as OA

    flop_per_block = 4.0 * w.block * w.block * w.d
    t0 = time.perf_counter()
    flop = 0.0
    done = []
    for (b, h) in heads:
        qh = q[b:b + 1, h:h + 1].double().numpy()
        kh = k[b:b + 1, h:h + 1].double().numpy()
        vh = v[b:b + 1, h:h + 1].double().numpy()
        OA.attention_head(qh, kh, vh, mask_np[b:b + 1, h:h + 1], 0, 0, w.block, w.causal)
        flop += flop_per_block * dense_blocks(mask_np[b:b + 1, h:h + 1], w.causal)
        done.append((b, h))
        if budget_s is not None and time.perf_counter() - t0 > budget_s:
            break
    return time.perf_counter() - t0, flop, done


def cpu_baseline(w, mask_np):
    """Bounded sample of the oracle on the host cores: 2 global + 2 local heads."""
    import torch

    from load_balancing_gb300 import workloads as W

    cores = len(os.sched_getaffinity(0))
    q, k, v = W.make_qkv(W.custom("cpu_sample", 1, 4, w.S, w.d, w.block, w.causal, 0, w.qkv_seed), "cpu")
    heads_src = [0, 1, 16, 17]
    sub_mask = np.ascontiguousarray(mask_np[:, heads_src])
    secs, flop, done = time_oracle(w, sub_mask, q, k, v, [(0, i) for i in range(4)], budget_s=30.0)
    return {"value": flop / secs / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "torch_threads": torch.get_num_threads(),
            "sample": f"fp64 numpy oracle on {len(done)} whole heads (2 global, 2 local) of the {w.name} "
                      f"workload, {secs:.1f} s; dense-block FLOP / wall time"}


# ----------------------------------------------------------------------------- reference arm
def gpu_sm_count(default):
    """SM count of GPU 0 (the GPU arm's worker count), or ``default`` without a GPU."""
    try:
        import torch

        if torch.cuda.is_available():
            return torch.cuda.get_device_properties(0).multi_processor_count
    except Exception:
        pass
    return default


def run_reference(args):
    rank, world, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    import torch

    from load_balancing_gb300 import workloads as W
    from oracle import loads as OL
    from oracle import lpt as OP

    w = W.WORKLOADS[WORKLOAD]
    mask_np = W.make_mask(w)
    q, k, v = W.make_qkv(W.custom("ref_sample", 1, 2, w.S, w.d, w.block, w.causal, 0, w.qkv_seed), "cpu")
    cores = len(os.sched_getaffinity(0))
    sample_heads = [0, 16]  # one global and one local head per step
    sub_mask = np.ascontiguousarray(mask_np[:, sample_heads])
    m = args.workers  # the GPU arm's worker count: one per SM but one

    def step():
        t0 = time.perf_counter()
        row, _, _ = OL.block_mask_loads(mask_np)
        OP.lpt_plan(row.reshape(-1), m)
        _, flop, _ = time_oracle(w, sub_mask, q, k, v, [(0, 0), (0, 1)])
        return time.perf_counter() - t0, flop

    for _ in range(args.warmup):
        step()
    tot_t, tot_f = 0.0, 0.0
    for _ in range(args.steps):
        t, f = step()
        tot_t += t
        tot_f += f
    value = tot_f / tot_t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": bench_config(w, m, dense_blocks(mask_np, w.causal), world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "per step: oracle mask loads and textbook LPT over the full workload "
                                       f"({w.n_items} items, m={m}) plus fp64 attention of 2 whole heads "
                                       "(1 global, 1 local); FLOP = dense blocks of those heads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- GPU arm
def run_gpu(args):
    import torch

    from load_balancing_gb300 import dbsp
    from load_balancing_gb300 import path as P
    from load_balancing_gb300 import workloads as W

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dbsp.library()  # fail loudly now if the library is missing

    w = W.WORKLOADS[WORKLOAD]
    mask_np = W.make_mask(w)
    n_dense = dense_blocks(mask_np, w.causal)
    n_diag = diag_blocks(mask_np) if w.causal else 0
    flop_per_block = 4.0 * w.block * w.block * w.d
    flop = flop_per_block * n_dense
    flop_fa = flop - 0.5 * flop_per_block * n_diag  # diagonal blocks counted as half
    mask = torch.from_numpy(mask_np).to(dev)
    q, k, v = W.make_qkv(w, dev)
    n_sm = P.default_workers(dev)
    n_workers = attention_workers(n_sm)
    # the timed step: batch i's attention on n_workers SMs beside batch i+1's mask loads and
    # plan on the remaining one (two plan buffers, kept by PipelinedSteps)
    pipe = P.PipelinedSteps(w.B, w.H, w.nQ, w.nK, dev, causal=w.causal, n_workers=n_workers)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
    timing = torch.zeros(3 * n_workers, dtype=torch.int64, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)  # 256 MiB > L2
    s_attn = torch.cuda.Stream(dev, priority=-1)
    s_attn.wait_stream(torch.cuda.current_stream(dev))

    def loads_plan(pb, m, st):
        dbsp.dbsp_block_mask_loads(mask, pb.row_loads, pb.col_loads, pb.head_loads, stream=st)
        dbsp.dbsp_plan_lpt(pb.row_loads.view(-1), m, pb.worker_of, pb.worker_offsets, pb.worklist,
                           pb.worker_loads, stream=st)

    def attention(pb, m, st, cta_timing=None):
        dbsp.dbsp_block_sparse_attn_fwd(q, k, v, mask, w.block, w.causal, pb.worker_offsets, pb.worklist, m,
                                        out=out, lse=lse, cta_timing=cta_timing, stream=st)

    def pipelined(n, ev=None):
        for i in range(n):
            with torch.cuda.stream(s_attn):
                flush.zero_()  # L2 flush, outside the timed events
            pipe.step(q, k, v, mask, w.block, w.causal, next_mask=mask, out=out, lse=lse, cta_timing=timing,
                      stream=s_attn, events=ev[i] if ev else None)

    pipe.prime(mask, stream=s_attn)  # batch 0's plan
    pipelined(args.warmup)
    torch.cuda.synchronize(dev)
    status = dbsp.dbsp_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]

    clocks = ClockSampler(local)
    poller = NvmlPoller(dev)
    if rank == 0:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    poller.start()
    pipelined(args.steps, ev)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    nvml = poller.stop()
    barrier(world)
    clk = clocks.stop() if rank == 0 else None
    if clk is not None and nvml is not None:  # the in-region samples lead; nvidia-smi's around it
        clk = dict(nvml, nvidia_smi=clk)
    step_ms = [ev[i][0].elapsed_time(ev[i][3]) for i in range(args.steps)]
    attn_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    side_ms = [ev[i][0].elapsed_time(ev[i][2]) for i in range(args.steps)]  # loads + plan beside it
    total_s = sum(step_ms) / 1e3
    total_s = max_over_ranks(total_s, world, dev)
    t = timing.view(n_workers, 3).cpu().numpy()
    busy = (t[:, 1] - t[:, 0]).astype(np.float64)
    skew = float((busy.max() - busy.mean()) / busy.mean())
    blocks_per_worker = t[:, 2]
    status = dbsp.dbsp_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    # breakdown (not part of the value): the serial step, one CUDA graph of the three
    # launches on every SM (each kernel may start its prologue while the previous one
    # finishes), and its mask loads + plan alone
    plan_buf = P.alloc_plan(w.B, w.H, w.nQ, w.nK, n_sm, dev)
    timing_sm = torch.zeros(3 * n_sm, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    graph_lp = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        loads_plan(plan_buf, n_sm, side)
        attention(plan_buf, n_sm, side, timing_sm)
        side.synchronize()
        with torch.cuda.graph(graph, stream=side):
            loads_plan(plan_buf, n_sm, side)
            attention(plan_buf, n_sm, side, timing_sm)
        with torch.cuda.graph(graph_lp, stream=side):
            loads_plan(plan_buf, n_sm, side)
    stream.wait_stream(side)

    def graph_ms(g):
        for _ in range(3):
            flush.zero_()
            g.replay()
        ts = []
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            g.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        return [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]

    serial_ms = graph_ms(graph)
    plan_ms = graph_ms(graph_lp)
    # the same loads + plan graph replayed back to back between one pair of events (no
    # flush between the replays: the 131 KB mask stays in L2), per replay
    n_b2b = 100
    ev[0][0].record(stream)
    for _ in range(n_b2b):
        graph_lp.replay()
    ev[0][1].record(stream)
    torch.cuda.synchronize(dev)
    plan_b2b_us = 1e3 * ev[0][0].elapsed_time(ev[0][1]) / n_b2b
    status = dbsp.dbsp_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the serial step")

    # end to end through the public API, host (pinned) buffers in and out
    q_h, k_h, v_h = (x.cpu().pin_memory() for x in (q, k, v))
    mask_h = torch.from_numpy(mask_np).pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (q_h, k_h, v_h, mask_h))
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
    # Double-buffered over three streams, as a serving loop would run it: step i+1's inputs
    # go in while step i computes and step i's result comes out. Every step still copies
    # its own inputs in and its own result out; the inputs of a step (201 MB) are larger
    # than L2, so no flush is needed between steps.
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    bufs = [dict(q=q, k=k, v=v, mask=mask, out=out, lse=lse, plan=P.alloc_plan(w.B, w.H, w.nQ, w.nK, n_workers, dev))]
    bufs.append(dict(q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v),
                     mask=torch.empty_like(mask), out=torch.empty_like(out), lse=torch.empty_like(lse),
                     plan=P.alloc_plan(w.B, w.H, w.nQ, w.nK, n_workers, dev)))
    host_out = [(out_h, lse_h), (torch.empty_like(out_h).pin_memory(), torch.empty_like(lse_h).pin_memory())]

    def e2e_run(n_steps):
        ev_in = [torch.cuda.Event() for _ in range(n_steps)]
        ev_cmp = [torch.cuda.Event() for _ in range(n_steps)]
        ev_out = [torch.cuda.Event() for _ in range(n_steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream(dev)
        t0.record(cur)
        for st in (s_in, s_cmp, s_out):
            st.wait_event(t0)
        for i in range(n_steps):
            b = bufs[i % 2]
            if i >= 2:
                s_in.wait_event(ev_cmp[i - 2])  # the buffers' previous compute is done
            with torch.cuda.stream(s_in):
                for name, src in (("q", q_h), ("k", k_h), ("v", v_h), ("mask", mask_h)):
                    b[name].copy_(src, non_blocking=True)
            ev_in[i].record(s_in)
            s_cmp.wait_event(ev_in[i])
            if i >= 2:
                s_cmp.wait_event(ev_out[i - 2])  # its previous result has left
            p = P.plan(b["mask"], n_workers, out=b["plan"], stream=s_cmp)
            P.attention(b["q"], b["k"], b["v"], b["mask"], w.block, w.causal, p, out=b["out"], lse=b["lse"],
                        stream=s_cmp)
            ev_cmp[i].record(s_cmp)
            s_out.wait_event(ev_cmp[i])
            o_h, l_h = host_out[i % 2]
            with torch.cuda.stream(s_out):
                o_h.copy_(b["out"], non_blocking=True)
                l_h.copy_(b["lse"], non_blocking=True)
            ev_out[i].record(s_out)
        for st in (s_in, s_cmp, s_out):
            cur.wait_stream(st)
        t1.record(cur)
        t1.synchronize()
        return t0.elapsed_time(t1) / 1e3

    e2e_run(max(2, args.warmup))
    torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks(e2e_run(args.steps), world, dev)
    # the last step's result, read back, matches the device-timed path's output
    if not torch.equal(host_out[(args.steps - 1) % 2][0], bufs[(args.steps - 1) % 2]["out"].cpu()):
        raise RuntimeError("end-to-end result differs from its device copy")

    total_flop = sum_over_ranks(flop * args.steps, world, dev)
    value = total_flop / total_s / 1e12
    attn_avg_s = statistics.mean(attn_ms) / 1e3
    attn_tflops = flop / attn_avg_s / 1e12
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(w, n_workers, n_dense, world),
        "attn_tflops": attn_tflops,
        "attn_tflops_fa_convention": flop_fa / attn_avg_s / 1e12,
        "pct_of_bf16_peak": 100.0 * attn_tflops / peak,
        "sm_skew": skew,
        "blocks_per_worker": {"min": int(blocks_per_worker.min()), "max": int(blocks_per_worker.max()),
                              "mean": float(blocks_per_worker.mean())},
        "attn_us": 1e6 * attn_avg_s,
        "loads_plus_plan_beside_attn_us": 1e3 * statistics.mean(side_ms),
        "serial_step": {"value": flop / (statistics.mean(serial_ms) / 1e3) / 1e12, "unit": UNIT,
                        "ms_per_step": statistics.mean(serial_ms), "n_workers": n_sm,
                        "how": "one CUDA graph of the mask-loads, LPT-plan and attention launches on every SM"},
        "loads_plus_plan_us": 1e3 * statistics.mean(plan_ms),
        "loads_plus_plan_back_to_back_us": plan_b2b_us,
        "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": attn_tflops / peak, "traffic": attn_traffic(),
                     "traffic_unit": "bytes per launch (ncu dram read + write)",
                     "peak_source": f"{peak_src} bf16 dense (burst, cuBLAS)",
                     "kernel": "attn_fwd_kernel<128,128>"},
        "e2e": {"value": total_flop / e2e_s / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "pinned host inputs in and results out every step through the public API, "
                       "double-buffered on three streams (step i+1 copies in while step i's loads, plan "
                       "and attention run)"},
        "gpu_launches": 3 * args.steps,
        "wall_s_timed": wall,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, mask_np)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------- suite (all workloads)
L2_BYTES = 129 * 1000 * 1000  # GB300 L2


def _time_ms(fn, stream, flush, reps):
    import torch

    ts = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def static_worklist(n_items, m, kind, device):
    """Round-robin (item i -> worker i mod m) or contiguous (equal slices) worklists."""
    import torch

    ids = np.arange(n_items)
    owner = ids % m if kind == "round_robin" else (ids * m) // max(1, n_items)
    order = np.argsort(owner, kind="stable")
    offsets = np.zeros(m + 1, dtype=np.int32)
    np.add.at(offsets, owner + 1, 1)
    offsets = np.cumsum(offsets).astype(np.int32)
    return (torch.from_numpy(offsets).to(device), torch.from_numpy(order.astype(np.int32)).to(device))


def run_suite(args):
    """One JSON line per workload: each kernel of the path timed on its own."""
    import torch

    from load_balancing_gb300 import dbsp
    from load_balancing_gb300 import path as P
    from load_balancing_gb300 import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dbsp.library()
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    peaks, peak_src = load_peaks()
    reps = max(3, args.steps)
    names = args.workloads.split(",") if args.workloads else W.ORDER
    for name in [x for x in names if x in W.WORKLOADS]:
        w = W.WORKLOADS[name]
        mask_np = W.make_mask(w)
        n_dense = dense_blocks(mask_np, w.causal)
        flop = 4.0 * w.block * w.block * w.d * n_dense
        mask = torch.from_numpy(mask_np).to(dev)
        q, k, v = W.make_qkv(w, dev)
        m = P.default_workers(dev)
        pb = P.alloc_plan(w.B, w.H, w.nQ, w.nK, m, dev)
        out = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
        timing = torch.zeros(3 * m, dtype=torch.int64, device=dev)
        line = {"suite": True, "workload": workload_description(w), "dense_blocks": n_dense,
                "items": w.n_items, "n_workers": m}
        # a1: mask loads
        loads = lambda: dbsp.dbsp_block_mask_loads(mask, pb.row_loads, pb.col_loads, pb.head_loads, stream=stream)
        t = _time_ms(loads, stream, flush, reps)
        nbytes = mask_np.size + 4 * (w.B * w.H * (w.nQ + w.nK + 1))
        line["mask_loads"] = {"us": 1e3 * t, "GB/s": nbytes / t / 1e6, "bytes": nbytes,
                              "frac_of_hbm": nbytes / t / 1e6 / float(peaks["hbm_gbs"])}
        # back to back: R launches captured in one CUDA graph (no host in the loop), cycling
        # through enough copies of the mask (together more than twice the 129 MB L2) that
        # each launch reads its mask from HBM; per-launch time without the event overhead
        copies = int(min(16, max(2, -(-2 * L2_BYTES // mask_np.size))))
        masks = [mask.clone() for _ in range(copies)]
        R = 4 * copies
        side = torch.cuda.Stream(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            dbsp.dbsp_block_mask_loads(masks[0], pb.row_loads, pb.col_loads, pb.head_loads, stream=side)
            side.synchronize()
            with torch.cuda.graph(graph, stream=side):
                for i in range(R):
                    dbsp.dbsp_block_mask_loads(masks[i % copies], pb.row_loads, pb.col_loads, pb.head_loads,
                                               stream=side)
        tb = _time_ms(graph.replay, stream, flush, 5) / R
        line["mask_loads"]["back_to_back"] = {
            "us": 1e3 * tb, "GB/s": nbytes / tb / 1e6, "frac_of_hbm": nbytes / tb / 1e6 / float(peaks["hbm_gbs"]),
            "launches": R, "mask_copies": copies, "from_hbm": bool(copies * mask_np.size > 2 * L2_BYTES),
            "how": "CUDA graph of the launches"}
        del graph
        del masks
        # a2: LPT plan
        plan = lambda: dbsp.dbsp_plan_lpt(pb.row_loads.view(-1), m, pb.worker_of, pb.worker_offsets, pb.worklist,
                                          pb.worker_loads, stream=stream)
        line["lpt_plan"] = {"us": 1e3 * _time_ms(plan, stream, flush, reps)}
        # a3/a4: attention under three worklists
        obs = []  # per CTA: (units, dense blocks, busy us), over all three worklists
        for kind in ("lpt", "round_robin", "contiguous"):
            if kind == "lpt":
                off, wl = pb.worker_offsets, pb.worklist
            else:
                off, wl = static_worklist(w.n_items, m, kind, dev)
            fn = lambda: dbsp.dbsp_block_sparse_attn_fwd(q, k, v, mask, w.block, w.causal, off, wl, m, out=out,
                                                         lse=lse, cta_timing=timing, stream=stream)
            t = _time_ms(fn, stream, flush, reps)
            tt = timing.view(m, 3).cpu().numpy()
            busy = (tt[:, 1] - tt[:, 0]).astype(np.float64)
            line[f"attn_{kind}"] = {"us": 1e3 * t, "TFLOP/s": flop / t / 1e9,
                                   "frac_of_bf16_peak": flop / t / 1e9 / float(peaks["bf16_tflops"]),
                                   "sm_skew": float((busy.max() - busy.mean()) / busy.mean()),
                                   "blocks_max_over_mean": float(tt[:, 2].max() / max(1e-9, tt[:, 2].mean()))}
            units = np.diff(off.cpu().numpy()).astype(np.float64)
            obs.append(np.stack([units, tt[:, 2].astype(np.float64), busy / 1e3], 1))
        # f3: planning cost fitted from cta_timing. busy ~ a * items + b * blocks per CTA, by
        # least squares over the CTAs of all three worklists (under LPT alone items and
        # blocks per CTA move together and the fit is ill-conditioned); then the A/B of an
        # LPT plan on block_cost * row_load + item_cost with item_cost / block_cost = a / b
        X = np.concatenate(obs)
        coef = np.linalg.lstsq(X[:, :2], X[:, 2], rcond=None)[0]
        c0 = float(coef[0] / coef[1]) if coef[1] > 0 else 0.0
        bc, ic = P.PLAN_BLOCK_COST_SCALE, int(round(max(0.0, c0) * P.PLAN_BLOCK_COST_SCALE))
        line["cost_fit"] = {"us_per_item": float(coef[0]), "us_per_block": float(coef[1]), "item_in_blocks": c0,
                            "ctas": int(X.shape[0])}
        # A/B: LPT on block_cost * row_load + item_cost at a few item costs (in blocks),
        # the fitted one included; the first entry is the pages' plan on dense blocks
        line["cost_ab"] = {}
        costs = [(1, 0), (1, 2), (1, P.ITEM_COST_BLOCKS), (1, 8), (bc, ic)]
        for bc2, ic2 in dict.fromkeys(costs):
            pc = P.plan(mask, m, block_cost=bc2, item_cost=ic2)
            fn = lambda: dbsp.dbsp_block_sparse_attn_fwd(q, k, v, mask, w.block, w.causal, pc.worker_offsets,
                                                         pc.worklist, m, out=out, lse=lse, cta_timing=timing,
                                                         stream=stream)
            t = _time_ms(fn, stream, flush, max(7, reps))
            tt = timing.view(m, 3).cpu().numpy()
            busy = (tt[:, 1] - tt[:, 0]).astype(np.float64)
            line["cost_ab"][f"{bc2}:{ic2}"] = {"us": 1e3 * t, "TFLOP/s": flop / t / 1e9,
                                              "sm_skew": float((busy.max() - busy.mean()) / busy.mean())}
        # head-level LPT over a few "virtual GPUs" (db-SP blog, scenario 1): makespan
        # against the lower bound max(ceil(total / m), largest head)
        hl = pb.head_loads.view(-1).contiguous()
        total, largest = int(hl.sum().item()), int(hl.max().item())
        line["head_lpt"] = {}
        for mv in (2, 4, 8):
            hp = P.alloc_plan(1, 1, hl.numel(), 1, mv, dev)
            dbsp.dbsp_plan_lpt(hl, mv, hp.worker_of, hp.worker_offsets, hp.worklist, hp.worker_loads, stream=stream)
            makespan = int(hp.worker_loads.max().item())
            bound = max(-(-total // mv), largest)
            line["head_lpt"][str(mv)] = {"makespan": makespan, "lower_bound": bound, "ratio": makespan / bound}
        # a5: merge of KV-shard partials (sharded workload), shards contiguous, striped
        # or planned by LPT over the KV blocks' column loads (db-SP blog, scenario 2)
        if "n_shards" in w.extra:
            n_sh = w.extra["n_shards"]
            for layout in ("contiguous", "striped", "lpt"):
                if layout == "lpt":
                    sp = P.plan_kv_shards(mask, n_sh, stream=stream)
                    t_sp = _time_ms(lambda: P.plan_kv_shards(mask, n_sh, stream=stream), stream, flush, reps)
                    shards = P.shard_masks_from_plan(mask, sp)
                else:
                    t_sp = None
                    shards = torch.from_numpy(W.shard_masks(mask_np, n_sh, layout)).to(dev)
                o_p = torch.empty((n_sh, w.B, w.H, w.S, w.d), dtype=torch.float32, device=dev)
                m_p = torch.empty((n_sh, w.B, w.H, w.S), dtype=torch.float32, device=dev)
                l_p = torch.empty_like(m_p)
                plans = [P.plan(shards[s], m, block_cost=P.SHARD_BLOCK_COST, item_cost=P.SHARD_ITEM_COST)
                         for s in range(n_sh)]

                def partials():
                    for s in range(n_sh):
                        P.attention_partial(q, k, v, shards[s], w.block, w.causal, plans[s], o_p[s], m_p[s],
                                            l_p[s], stream=stream)

                t_part = _time_ms(partials, stream, flush, reps)
                merge = lambda: dbsp.dbsp_merge_partials(o_p.view(n_sh, -1, w.d), m_p.view(n_sh, -1),
                                                         l_p.view(n_sh, -1), out.view(-1, w.d), lse.view(-1),
                                                         stream=stream)
                t = _time_ms(merge, stream, flush, reps)
                rows = w.B * w.H * w.S
                # an empty partial's O is never read: count the live ones
                live = int(((l_p > 0) & torch.isfinite(m_p)).sum().item())
                nbytes = live * 4 * w.d + n_sh * rows * 8 + rows * (2 * w.d + 4)
                shard_load = np.array([int(pl.head_loads.sum().item()) for pl in plans], dtype=np.float64)
                line[f"merge_{layout}"] = {"us": 1e3 * t, "GB/s": nbytes / t / 1e6, "bytes": nbytes,
                                           "frac_of_hbm": nbytes / t / 1e6 / float(peaks["hbm_gbs"]),
                                           "partials_us": 1e3 * t_part,
                                           "partials_TFLOP/s": flop / t_part / 1e9,
                                           "shard_loads": shard_load.astype(int).tolist(),
                                           "shard_max_over_mean": float(shard_load.max() / shard_load.mean())}
                if t_sp is not None:
                    line[f"merge_{layout}"]["shard_plan_us"] = 1e3 * t_sp
                # A/B of the shard passes' planning cost (block_cost:item_cost)
                ab = {}
                for bc2, ic2 in dict.fromkeys([(1, 0), (8, 1), (P.SHARD_BLOCK_COST, P.SHARD_ITEM_COST)]):
                    plans = [P.plan(shards[s], m, block_cost=bc2, item_cost=ic2) for s in range(n_sh)]
                    ab[f"{bc2}:{ic2}"] = {"partials_us": 1e3 * _time_ms(partials, stream, flush, max(5, reps))}
                line[f"merge_{layout}"]["cost_ab"] = ab
        line["peaks"] = {"bf16_tflops": peaks["bf16_tflops"], "hbm_gbs": peaks["hbm_gbs"], "source": peak_src}
        status = dbsp.dbsp_device_status()
        line["device_status"] = status
        print(json.dumps(line), flush=True)
        del q, k, v, out, lse, mask
        torch.cuda.empty_cache()
    if not args.workloads or "long_causal" in names:
        split_study(dev, stream, flush, reps, peaks)
    if not args.workloads or "bonus" in names:
        bonus_study(dev, stream, flush, reps)
    return 0


def bonus_study(dev, stream, flush, reps):
    """Plan reuse across consecutive masks (db-SP blog, scenario 2, third bullet): the
    next step's mask flips 2 % of the blocks; its plan takes the previous plan as home
    with a stay bonus. Reported per bonus: the fraction of items kept on their worker,
    the makespan over the lower bound max(ceil(total / m), largest item), plan time."""
    import torch

    from load_balancing_gb300 import path as P
    from load_balancing_gb300 import workloads as W

    m = P.default_workers(dev)
    for name in ("llm", "video"):
        w = W.WORKLOADS[name]
        mask0_np = W.make_mask(w)
        mask1_np = W.perturb_mask(mask0_np, 0.02, 1, w.causal)
        mask0 = torch.from_numpy(mask0_np).to(dev)
        mask1 = torch.from_numpy(mask1_np).to(dev)
        p0 = P.plan(mask0, m, stream=stream)
        home = p0.worker_of.clone()
        loads1 = (mask1_np != 0).sum(-1).reshape(-1)
        bound = max(-(-int(loads1.sum()) // m), int(loads1.max()))
        line = {"suite": True, "study": "stay bonus", "workload": name, "flipped_fraction": 0.02,
                "n_workers": m, "lower_bound": bound, "bonus": {}}
        for bonus in (0, 1, 2, 4, 8, 16, 32, 1 << 20):
            p1 = P.plan(mask1, m, home=home, stay_bonus=bonus, stream=stream)
            stay = float((p1.worker_of == home).float().mean().item())
            makespan = int(p1.worker_loads.max().item())
            t = _time_ms(lambda: P.plan(mask1, m, home=home, stay_bonus=bonus, out=p1, stream=stream), stream,
                         flush, reps)
            line["bonus"][str(bonus)] = {"stay": stay, "makespan_over_bound": makespan / bound, "plan_us": 1e3 * t}
        print(json.dumps(line), flush=True)


def split_study(dev, stream, flush, reps, peaks):
    """Heavy items split along their KV blocks (db-SP blog, closing remark) on rows as
    heavy as the mean load per SM: two fully causal heads of 16,384 tokens. Whole-item
    LPT against split LPT (automatic piece load), plan + attention (+ merge) timed."""
    import torch

    from load_balancing_gb300 import dbsp
    from load_balancing_gb300 import path as P
    from load_balancing_gb300 import workloads as W

    w = W.custom("long_causal", 1, 2, 16384, 128, 128, True, 6, 106, "causal_full")
    mask_np = W.make_mask(w)
    n_dense = dense_blocks(mask_np, w.causal)
    flop = 4.0 * w.block * w.block * w.d * n_dense
    mask = torch.from_numpy(mask_np).to(dev)
    q, k, v = W.make_qkv(w, dev)
    m = P.default_workers(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
    timing = torch.zeros(3 * m, dtype=torch.int64, device=dev)
    line = {"suite": True, "workload": f"long_causal: B=1 H=2 S=16384 d=128 block=128 causal=1; full causal mask; "
                                      f"Q/K/V bf16 N(0,1)", "dense_blocks": n_dense, "items": w.n_items,
            "n_workers": m, "largest_item": int((mask_np != 0).sum(-1).max()), "mean_per_worker": n_dense / m}
    pb = P.plan(mask, m, stream=stream)

    def skew():
        tt = timing.view(m, 3).cpu().numpy()
        busy = (tt[:, 1] - tt[:, 0]).astype(np.float64)
        return float((busy.max() - busy.mean()) / busy.mean())

    attn = lambda: dbsp.dbsp_block_sparse_attn_fwd(q, k, v, mask, w.block, w.causal, pb.worker_offsets,
                                                   pb.worklist, m, out=out, lse=lse, cta_timing=timing,
                                                   stream=stream)
    t = _time_ms(attn, stream, flush, reps)
    line["whole_lpt"] = {"attn_us": 1e3 * t, "TFLOP/s": flop / t / 1e9, "sm_skew": skew(),
                         "plan_us": 1e3 * _time_ms(lambda: P.plan(mask, m, out=pb, stream=stream), stream, flush,
                                                   reps)}
    def per_unit_cost(offsets):
        # busy time against the number of units and blocks per CTA (least squares):
        # busy ~ a * units + b * blocks
        tt = timing.view(m, 3).cpu().numpy().astype(np.float64)
        busy = (tt[:, 1] - tt[:, 0]) / 1e3
        units = np.diff(offsets.cpu().numpy()).astype(np.float64)
        coef = np.linalg.lstsq(np.stack([units, tt[:, 2]], 1), busy, rcond=None)[0]
        return {"us_per_unit": float(coef[0]), "us_per_block": float(coef[1])}

    line["whole_lpt"]["fit"] = per_unit_cost(pb.worker_offsets)
    mean_t = -(-n_dense // m)
    line["split_lpt"] = {}
    for label, t_max in (("half_mean", 0), ("mean", mean_t)):
        sp = P.plan_split(mask, m, w.block, w.d, max_piece_load=t_max, stream=stream)
        attn_s = lambda: P.attention_split(q, k, v, mask, w.block, w.causal, sp, out=out, lse=lse,
                                           cta_timing=timing, stream=stream)
        t_s = _time_ms(attn_s, stream, flush, reps)
        sk = skew()
        fit = per_unit_cost(sp.worker_offsets)
        counts = sp.counts.cpu().numpy().tolist()
        t_plan = _time_ms(lambda: P.plan_split(mask, m, w.block, w.d, max_piece_load=t_max, out=sp,
                                               stream=stream), stream, flush, reps)
        line["split_lpt"][label] = {"attn_plus_merge_us": 1e3 * t_s, "TFLOP/s": flop / t_s / 1e9, "sm_skew": sk,
                                    "plan_us": 1e3 * t_plan, "units": counts[0], "split_items": counts[2],
                                    "pieces": counts[3], "piece_load": counts[4], "fit": fit,
                                    "planned_max_over_mean": float(sp.worker_loads.max().item() /
                                                                   sp.worker_loads.float().mean().item()),
                                    "frac_of_bf16_peak": flop / t_s / 1e9 / float(peaks["bf16_tflops"])}
    line["whole_lpt"]["planned_max_over_mean"] = float(pb.worker_loads.max().item() /
                                                       pb.worker_loads.float().mean().item())
    line["whole_lpt"]["frac_of_bf16_peak"] = flop / t / 1e9 / float(peaks["bf16_tflops"])
    line["device_status"] = dbsp.dbsp_device_status()
    print(json.dumps(line), flush=True)


def run_kernels_once(args):
    """One launch each of the mask-loads, LPT-plan and merge kernels (a profiler target).

    Mask loads on the imbalance workload's mask (41.9 MB), the plan over the LLM-heads
    workload's 2,048 row loads, and the merge of 8 fp32 partials of 131,072 rows x 128
    (20 % of them empty, m = -inf, l = 0).
    """
    import torch

    from load_balancing_gb300 import dbsp
    from load_balancing_gb300 import path as P
    from load_balancing_gb300 import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wi = W.WORKLOADS["imbalance"]
    mask = torch.from_numpy(W.make_mask(wi)).to(dev)
    row = torch.empty((wi.B, wi.H, wi.nQ), dtype=torch.int32, device=dev)
    col = torch.empty((wi.B, wi.H, wi.nK), dtype=torch.int32, device=dev)
    head = torch.empty((wi.B, wi.H), dtype=torch.int32, device=dev)
    wl = W.WORKLOADS["llm"]
    lrow = torch.from_numpy(W.make_mask(wl)).to(dev).ne(0).sum(-1, dtype=torch.int32).reshape(-1).contiguous()
    m = P.default_workers(dev)
    n = lrow.numel()
    wo = torch.empty(n, dtype=torch.int32, device=dev)
    off = torch.empty(m + 1, dtype=torch.int32, device=dev)
    wlst = torch.empty(n, dtype=torch.int32, device=dev)
    wload = torch.empty(m, dtype=torch.int64, device=dev)
    rows, d, ns = 131072, 128, 8
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    o = torch.randn((ns, rows, d), generator=g, device=dev)
    mm = torch.randn((ns, rows), generator=g, device=dev) * 4
    ll = torch.rand((ns, rows), generator=g, device=dev) * 50 + 0.5
    empty = torch.rand((ns, rows), generator=g, device=dev) < 0.2
    mm[empty] = -float("inf")
    ll[empty] = 0
    out = torch.empty((rows, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty(rows, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    ni = row.numel()
    iwo = torch.empty(ni, dtype=torch.int32, device=dev)
    iwl = torch.empty(ni, dtype=torch.int32, device=dev)
    dbsp.dbsp_block_mask_loads(mask, row, col, head)
    dbsp.dbsp_plan_lpt(lrow, m, wo, off, wlst, wload)
    dbsp.dbsp_plan_lpt(row.view(-1), m, iwo, off, iwl, wload)  # the imbalance workload's 40,960 items
    dbsp.dbsp_merge_partials(o, mm, ll, out, lse)
    torch.cuda.synchronize()
    status = dbsp.dbsp_device_status()
    print(json.dumps({"profile_kernels": ["mask_loads", "lpt_plan (llm)", "lpt_plan (imbalance)", "merge_partials"],
                      "device_status": status}))
    return 0 if status == 0 else 1


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["dbsp", "reference"], default="dbsp")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workers", type=int, default=0,
                    help="LPT workers of the reference arm (default: the GPU arm's, SM count - 1)")
    ap.add_argument("--suite", action="store_true", help="one line per workload, every kernel timed alone")
    ap.add_argument("--workloads", default="", help="comma-separated workload names for --suite")
    ap.add_argument("--profile-kernels", action="store_true",
                    help="launch the mask-loads, plan and merge kernels once each (for a profiler)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl != "reference":
        args.warmup = 3
    if args.impl == "reference":
        if args.workers <= 0:
            args.workers = attention_workers(gpu_sm_count(152))
        return run_reference(args)
    if args.suite:
        return run_suite(args)
    if args.profile_kernels:
        return run_kernels_once(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
