"""Benchmark of one MLA decode step (absorb -> latent attention with split-KV
-> combine -> out-projection) on synthetic inputs of the DeepSeek-V2 layer
shape: B=32 sequences, H=128 heads, 4096 cached tokens each, 576-d bf16
latent cache in 64-token pages.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload v2_layer|tiny|long_ctx|ragged|fp8_batch]

Prints one JSON line.  The L2 is flushed (a 256 MiB write) before every timed
step; the step itself is timed with CUDA events on the launching stream.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import mla_inputs as mi  # noqa: E402

E2E_STEPS = 32  # steps recorded in one graph by the end-to-end leg
METRIC = "MLA decode tokens/s and latent-cache HBM GB/s (% of ~8 TB/s roofline), 1 B300"
FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="v2_layer", choices=sorted(mi.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="host time of the reference arm's warm-up and timed steps together")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6400.0, 1800.0, "fallback"


# Sources of the decode kernel; their hash is recorded beside the ncu DRAM
# traffic in profiles/, so a stale figure (kernel changed since the capture)
# is reported as null.
DECODE_SOURCES = ("mla_latent_kv_66_b300/csrc/decode_tc.cu", "mla_latent_kv_66_b300/csrc/tc.cuh",
                  "mla_latent_kv_66_b300/csrc/common.cuh")
CLOCK_WINDOW_S = 1.5  # the step repeated under the clock sampler before the timed steps


def decode_source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM read + write bytes of one decode launch on this workload, from the
    committed ncu summary (profiles/decode_tc_<workload>.md, lines
    `traffic_bytes_per_launch: N` and `decode_source_hash: H`); None when
    there is no capture or the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"decode_tc_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        line = line.strip().strip("`")
        for key in ("traffic_bytes_per_launch", "decode_source_hash"):
            if line.startswith(key + ":"):
                vals[key] = line.split(":", 1)[1].strip()
    if vals.get("decode_source_hash") != decode_source_hash() or "traffic_bytes_per_launch" not in vals:
        return None
    return float(vals["traffic_bytes_per_launch"])


def host_cpu():
    model = None
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    return os.cpu_count(), model


def cache_bytes_per_token(kv_dtype):
    return 576 * 2 if kv_dtype == "bf16" else 576 + 4


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            self.proc.wait()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = max(mx, float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- ours
def setup_gpu(w, device):
    import torch
    import mla_latent_kv_66_b300 as mla
    from mla_latent_kv_66_b300 import _lib as L

    inp = mi.make_inputs(w, with_kv=False)
    table, lens = inp["page_table"], inp["seq_lens"]
    npg = inp["num_pages"]
    p = L.make_params(w.B, w.H, table.shape[1], npg, w.kv_dtype, w.out_dtype)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)

    if w.kv_dtype.startswith("e4m3"):
        ckv = torch.zeros(npg, 64, 512, dtype=torch.uint8, device=device)
        kpe = torch.zeros(npg, 64, 64, dtype=torch.uint8, device=device)
        sc = torch.ones(npg, 64, dtype=torch.float32, device=device)
    else:
        ckv = torch.zeros(npg, 64, 512, dtype=torch.bfloat16, device=device)
        kpe = torch.zeros(npg, 64, 64, dtype=torch.bfloat16, device=device)
        sc = None
    for b in range(w.B):  # write the cache with the library's append kernel
        n = int(lens[b])
        t = np.arange(n)
        slots = torch.from_numpy((table[b, t // 64].astype(np.int64) * 64 + t % 64).astype(np.int32)).to(device)
        mla.mla_cache_append(p, bf(mi.kv_rows(w, b, n)), slots,
                             torch.from_numpy(t.astype(np.int32)).to(device), 3, ckv, kpe, sc)
    lens_d = torch.from_numpy(lens).to(device)
    table_d = torch.from_numpy(table).to(device)
    step = mla.MLADecodeStep(w.B, w.H, table.shape[1], npg, w.kv_dtype, w.out_dtype, w.splits, device,
                             q_len=w.q_len)
    # rows of the step: the sequences, or q_len rows per sequence (the page
    # table and lengths the calls see; the query is rotated at each
    # row's length minus one)
    rows_table, rows_lens = step.expand_rows(table_d, lens_d)
    q_pe = torch.empty(w.B * w.q_len, w.H, 64, dtype=torch.bfloat16, device=device)
    mla.mla_rope_q(step.p, bf(inp["q_pe_raw"].reshape(-1, w.H, 64)), rows_lens, q_pe)
    state = dict(inp=inp, p=p, ckv=ckv, kpe=kpe, sc=sc, lens=lens_d, table=table_d,
                 rows_table=rows_table, rows_lens=rows_lens, q_nope=bf(inp["q_nope"]), q_pe=q_pe,
                 w_uk=bf(inp["w_uk"]), w_uv=bf(inp["w_uv"]))
    torch.cuda.synchronize()
    return state, step


def max_over_ranks(vals, world, device=None):
    """Element-wise maximum over the ranks of per-rank timings: the slowest
    replica sets the job's time.  One all-reduce; no-op for one process."""
    vals = [float(v) for v in vals]
    if world <= 1:
        return vals
    import torch
    import torch.distributed as dist
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tokens_per_s(world, tokens_per_step, ms):
    """Whole-job throughput of `world` replicas that each decode
    `tokens_per_step` tokens per step of `ms` milliseconds (the max over ranks)."""
    return world * tokens_per_step / (ms / 1000.0)


def pin_to_gpu_cpus(dev):
    """Run this process on the CPUs next to GPU `dev` (NVML's CPU affinity of
    the device with the same UUID), so that the pinned host buffers of the
    end-to-end leg sit on the GPU's NUMA node.  Reads the GPU's topology only;
    does nothing where NVML or the UUID is unavailable."""
    try:
        import pynvml
        import torch
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
        pynvml.nvmlInit()
        try:
            h = pynvml.nvmlDeviceGetHandleByUUID(uuid)
            masks = pynvml.nvmlDeviceGetCpuAffinity(h, (os.cpu_count() + 63) // 64)
            cpus = {64 * i + b for i, m in enumerate(masks) for b in range(64) if (m >> b) & 1}
            cpus &= set(range(os.cpu_count()))
            if cpus:
                os.sched_setaffinity(0, cpus)
        finally:
            pynvml.nvmlShutdown()
    except Exception:
        pass


def run_ours(args, w, rank, world):
    import torch
    import torch.distributed as dist
    import mla_latent_kv_66_b300 as mla
    from mla_latent_kv_66_b300 import _lib as L

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    pin_to_gpu_cpus(dev)
    st, step = setup_gpu(w, dev)
    p, G = step.p, step.num_splits
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    args_step = (st["q_nope"], st["q_pe"], st["w_uk"], st["w_uv"], st["ckv"], st["kpe"], st["sc"],
                 st["table"], st["lens"])

    def one(ev=None):
        L.mla_absorb_q(p, st["q_nope"], st["w_uk"], step.q_lat)
        if ev:
            # the decode launch (host side: four tensor-map encodings and the
            # launch) is queued before the event fires: a GPU spin of about
            # 0.5 ms covers it on slow hosts too
            torch.cuda._sleep(1_000_000)
            ev[0].record()
        L.mla_decode(p, step.q_lat, st["q_pe"], st["ckv"], st["kpe"], st["sc"], st["rows_table"], st["rows_lens"],
                     G, step.workspace, step.o_lat, step.lse)
        if ev:
            ev[1].record()
        L.mla_combine_out_proj(p, step.workspace, G, st["rows_lens"], step.o_lat, st["w_uv"], step.out, step.lse)

    # the step as a CUDA graph (its launches recorded once)
    step.capture(*args_step)
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with ClockSampler(dev.index) as clk:
        # the same step repeated for CLOCK_WINDOW_S under the sampler, so the
        # clock record holds enough samples under this load even when K is small
        t_end = time.perf_counter() + CLOCK_WINDOW_S
        while time.perf_counter() < t_end:
            for _ in range(50):
                flush.zero_()
                step.replay()
            torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        wall0 = time.perf_counter()
        for i in range(K):
            flush.zero_()
            evs[i][0].record()
            step.replay()
            evs[i][1].record()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        wall = time.perf_counter() - wall0
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)

    # the decode kernel alone (roofline): events around mla_decode in an eager step
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        one()
    dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(min(K, 200))]
    for b_, c_ in dev_ev:
        flush.zero_()
        one((b_, c_))
    torch.cuda.synchronize()
    dms = statistics.mean(b_.elapsed_time(c_) for b_, c_ in dev_ev)
    ms, dms = max_over_ranks([ms, dms], world, dev)

    # end to end: every step's per-token inputs (q_nope, rotated q_pe, page
    # table, lengths) packed in one pinned host buffer and copied in with one
    # host-to-device copy, the step, and its output copied back to pinned host
    # memory.  Steps alternate between two buffer sets so that one set's
    # copies overlap the other's compute (a set's inputs are rewritten only
    # after its previous step has read them, its output buffer only after it
    # has been copied out); E2E_STEPS such steps are recorded as one CUDA graph
    # (copies on their own streams), so the host issues one launch per
    # E2E_STEPS steps.  No L2 flush inside: the cache (151 MB for v2_layer) is
    # larger than the L2.
    inp = st["inp"]
    names = ("q_nope", "q_pe", "table", "lens")
    offs, total = {}, 0
    for k in names:
        offs[k] = total
        total += (st[k].numel() * st[k].element_size() + 255) // 256 * 256

    def view(buf, k):
        n = st[k].numel() * st[k].element_size()
        return buf[offs[k]: offs[k] + n].view(st[k].dtype).view(st[k].shape)

    table_np = inp["page_table"]
    sets = []
    for k in range(2):
        host_pack = torch.empty(total, dtype=torch.uint8).pin_memory()
        dev_pack = torch.empty(total, dtype=torch.uint8, device=dev)
        for nm in names:
            view(host_pack, nm).copy_(st[nm].cpu())
        devb = {nm: view(dev_pack, nm) for nm in names}
        stp = mla.MLADecodeStep(w.B, w.H, table_np.shape[1], inp["num_pages"], w.kv_dtype, w.out_dtype, w.splits,
                                dev, q_len=w.q_len)
        sargs = (devb["q_nope"], devb["q_pe"], st["w_uk"], st["w_uv"], st["ckv"], st["kpe"], st["sc"], devb["table"],
                 devb["lens"])
        dev_pack.copy_(host_pack)
        stp(*sargs)  # first-call set-up outside the capture
        out_h = torch.empty(stp.out.shape, dtype=stp.out.dtype).pin_memory()
        sets.append(dict(host=host_pack, dev=dev_pack, step=stp, args=sargs, out_h=out_h))
    torch.cuda.synchronize()
    h2d = sum(st[k].numel() * st[k].element_size() for k in names)
    d2h = sets[0]["out_h"].numel() * sets[0]["out_h"].element_size()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap = torch.cuda.current_stream()
        ev_done, ev_d2h = [], []
        for i in range(E2E_STEPS):
            k = sets[i % 2]
            if i >= 2:
                s_in.wait_event(ev_done[i - 2])  # the set's previous step has read its inputs
            else:
                s_in.wait_stream(cap)
            with torch.cuda.stream(s_in):
                k["dev"].copy_(k["host"], non_blocking=True)
            e_in = torch.cuda.Event()
            e_in.record(s_in)
            cap.wait_event(e_in)
            if i >= 2:
                cap.wait_event(ev_d2h[i - 2])  # the set's previous output has been copied out
            k["step"](*k["args"])
            ev_done.append(torch.cuda.Event())
            ev_done[-1].record(cap)
            s_out.wait_event(ev_done[-1])
            with torch.cuda.stream(s_out):
                k["out_h"].copy_(k["step"].out, non_blocking=True)
            ev_d2h.append(torch.cuda.Event())
            ev_d2h[-1].record(s_out)
        cap.wait_stream(s_in)
        cap.wait_stream(s_out)
    reps = max(1, min(K, 500) // E2E_STEPS)
    for _ in range(max(3, args.warmup // E2E_STEPS + 1)):  # copies and steps warmed up too
        graph.replay()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start.record()
    for _ in range(reps):
        graph.replay()
    t_end.record()
    torch.cuda.synchronize()
    e2e, = max_over_ranks([t_start.elapsed_time(t_end) / (reps * E2E_STEPS)], world, dev)
    status = step.status()
    return dict(ms=ms, dec_ms=dms, e2e_ms=e2e, h2d=h2d, d2h=d2h, wall=wall, clocks=clk.summary(),
                status=status, G=G, tokens=int(inp["seq_lens"].sum()))


# --------------------------------------------------------------------------- oracle (CPU)
def blas_threads():
    """Threads the oracle's numpy BLAS calls use (its only parallel part)."""
    try:
        from threadpoolctl import threadpool_info
        n = max([i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"] or [0])
        if n:
            return n
    except ImportError:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return len(os.sched_getaffinity(0))


class OracleSample:
    """The fp64 oracle run on a bounded sample of the same workload: whole
    sequences, all H heads each, in a seeded order.  Inputs are drawn once;
    each sequence's cache is written when first reached (not timed)."""

    def __init__(self, w, seed=0):
        from oracle import mla_oracle as O
        self.O, self.w = O, w
        self.base = mi.make_inputs(w, with_kv=False)
        self.order = [int(b) for b in np.random.default_rng(seed).permutation(w.B)]
        self.pos, self.h, self.cur = 0, 0, None
        self.seqs = []

    def _load(self):
        O, w = self.O, self.w
        b = self.order[self.pos % len(self.order)]
        n = int(self.base["seq_lens"][b])
        table = np.arange((n + 63) // 64, dtype=np.int32)[None, :]
        fmt = "e4m3" if w.kv_dtype.startswith("e4m3") else "bf16"  # the oracle's cache format
        sub = {"workload": mi.Workload("sample", B=1, H=w.H, L=n, seed=w.seed, kv_dtype=fmt),
               "seq_lens": np.array([n], np.int32), "page_table": table, "num_pages": table.shape[1],
               "q_nope": self.base["q_nope"][[b]], "q_pe_raw": self.base["q_pe_raw"][[b]],
               "w_uk": self.base["w_uk"], "w_uv": self.base["w_uv"], "kv_raw": {0: mi.kv_rows(w, b, n)}}
        cache = O.build_cache(sub, fmt)
        if w.q_len > 1:
            qpe = O.rope_q_multi_bf16(sub["q_pe_raw"], sub["seq_lens"], w.q_len)
        else:
            qpe = O.rope_q_bf16(sub["q_pe_raw"], sub["seq_lens"])
        self.cur = (sub, cache, qpe)
        self.seqs.append((b, n))

    def run(self, budget_s):
        """Decode (sequence, head) pairs for about budget_s seconds (at least
        one pair); returns (pairs, seconds)."""
        pairs, spent = 0, 0.0
        while pairs == 0 or spent < budget_s:
            if self.cur is None:
                self._load()
            sub, cache, qpe = self.cur
            t0 = time.perf_counter()
            if self.w.q_len > 1:  # one (sequence, head) pair: all of its query tokens
                self.O.decode_multi_reference(cache, sub, qpe, self.w.q_len,
                                              [(0, i, self.h) for i in range(self.w.q_len)])
            else:
                self.O.decode_reference(cache, sub, qpe, [(0, self.h)])
            spent += time.perf_counter() - t0
            pairs += 1
            self.h += 1
            if self.h == self.w.H:
                self.h, self.pos, self.cur = 0, self.pos + 1, None
        return pairs, spent

    def describe(self, pairs, spent):
        b, n = self.seqs[0]
        return (f"{pairs} (sequence, head) pairs over {len(self.seqs)} sequence(s) (first: b={b}, L={n}), "
                f"non-absorbed fp64 oracle, {spent:.1f} s")


def cpu_oracle_sample(w, budget_s=15.0, seed=0):
    """Decoded tokens/s of the oracle (one token = all H heads of one
    sequence) over about budget_s seconds; returns (value, threads, text)."""
    s = OracleSample(w, seed)
    pairs, spent = s.run(budget_s)
    return (pairs * w.q_len / w.H) / spent, blas_threads(), s.describe(pairs, spent)


def run_reference(args, w):
    """The oracle as the reference arm: every step is a bounded sample of the
    workload, sized so that warm-up plus timed steps take about --ref-seconds."""
    s = OracleSample(w, 0)
    per_step = min(20.0, max(0.02, args.ref_seconds / (args.steps + max(3, args.warmup))))
    for _ in range(max(3, args.warmup)):
        s.run(per_step)
    pairs, spent = 0, 0.0
    for _ in range(args.steps):
        p, t = s.run(per_step)
        pairs, spent = pairs + p, spent + t
    return (pairs * w.q_len / w.H) / spent, blas_threads(), s.describe(pairs, spent), 1000.0 * spent / args.steps


# --------------------------------------------------------------------------- main
def main():
    args = parse()
    w = mi.WORKLOADS[args.workload]
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "L": w.L or "log-uniform[%d,%d]" % w.ragged, "q_len": w.q_len,
           "kv_lora_rank": 512, "rope_dim": 64, "page_size": 64, "kv_dtype": w.kv_dtype,
           "pages": w.pages, "l2": "flushed before every timed step (256 MiB write)",
           "step": "CUDA graph: q absorption, decode, split-KV combine fused into the out-projection",
           "e2e": "pinned host inputs and output copied every step; steps alternate two buffer sets (copies "
                  "overlap the other set's compute), %d steps per CUDA graph; " % E2E_STEPS +
                  "no L2 flush (cache larger than the L2)",
           "parallelism": "replicas" if world > 1 else "single-gpu"}
    if args.impl == "reference":
        if rank != 0:
            return
        v, cores, desc, ms = run_reference(args, w)
        print(json.dumps({"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
                          "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": ms, "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                          "config": cfg,
                          "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                           "sample": desc, "nproc": host_cpu()[0], "cpu_model": host_cpu()[1]},
                          "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    cpus = os.sched_getaffinity(0)
    r = run_ours(args, w, rank, world)
    os.sched_setaffinity(0, cpus)  # the CPU baseline runs on every core again
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    hbm, tflops, src = peaks()
    tokens_per_step = w.B * w.q_len
    value = job_tokens_per_s(world, tokens_per_step, r["ms"])
    cache_bytes = r["tokens"] * cache_bytes_per_token(w.kv_dtype)
    achieved = cache_bytes / (r["dec_ms"] / 1000.0) / 1e9
    if w.kv_dtype == "bf16":
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm}
    else:
        # E4M3 cache: 2*H*(576+512) flops per cached token over 580 bytes, above
        # the ridge, so the bound is the tensor rate: bf16 when the codes are
        # expanded, E4M3 (the measured bf16 rate x 2, the nominal ratio) when
        # the 8-bit tensor cores multiply them
        mma8 = w.kv_dtype in ("e4m3_mma", "e4m3_mma1")
        pk = tflops * 2 if mma8 else tflops
        flops = r["tokens"] * 2.0 * w.H * (576 + 512)
        tf = flops / (r["dec_ms"] / 1000.0) / 1e12
        roofline = {"bound": "tensor", "achieved": tf, "peak": pk, "unit": "TFLOP/s", "frac": tf / pk,
                    "cache_gbs": achieved, "cache_frac_of_hbm": achieved / hbm}
        if mma8:
            src = src + " (e4m3 = 2 x bf16, nominal ratio)"
    roofline.update({"traffic": ncu_traffic(w.name), "kernel": "mla_decode", "peak_source": src,
                     "decode_ms": r["dec_ms"], "decode_source_hash": decode_source_hash()})
    cpu = None
    if not args.no_cpu_baseline:
        v, cores, desc = cpu_oracle_sample(w)
        nproc, model = host_cpu()
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc,
               "nproc": nproc, "cpu_model": model}
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"bf16": "bf16", "e4m3": "e4m3-cache/bf16"}.get(w.kv_dtype, "e4m3-cache/e4m3-mma"),
        "data": "synthetic (seeded, DeepSeek-V2 MLA shapes; random-init weights)", "config": cfg,
        "cache_gbs": achieved, "cache_bytes_per_step": cache_bytes,
        "cached_tokens_per_s": r["tokens"] / (r["dec_ms"] / 1000.0),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": job_tokens_per_s(world, tokens_per_step, r["e2e_ms"]), "unit": "tokens/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        # per step: absorption, (E4M3 tensor-core path: query quantisation),
        # decode, combine + out-projection; several query tokens: the row expansion
        "gpu_launches": (3 + (w.kv_dtype in ("e4m3_mma", "e4m3_mma1")) + (w.q_len > 1)) * args.steps,
        "clocks": r["clocks"], "status": r["status"], "num_splits": r["G"], "wall_s_timed": r["wall"],
    }
    print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
