#!/usr/bin/env python
"""LRKV decode benchmark on GB300.

One step = one decode step of one layer for a batch of requests, through the
C ABI: lrkv_decode_step appends each request's new row (shared + private
projections) at position T-1 and attends over the T cached rows (factored
scores, one online softmax, shared + private value reductions, expansion by
B_V^T).  Inputs are seeded synthetic tensors of the workload's shape,
resident in HBM when the timed region starts.

Prints one JSON line (rank 0).  The headline is the decode_T4096 workload;
the same line carries, under "configs", the long-context, ragged-paged and
prefill workloads measured the same way (step time, the dominant kernel's
roofline over >= 500 launches, end-to-end throughput from host buffers).
``--impl reference`` times the float64 CPU oracle on the same workload and
sample as the line's cpu_baseline.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LRKV decode tokens/s and achieved HBM GB/s (% of roofline) at 1 GB300"
PREFILL_METRIC = "LRKV prefill tokens/s"
L2_BYTES = 129 * 10 ** 6
NORTH_STAR_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

WORKLOADS = {
    "decode_T4096": "B=16 requests, d=2048, H=16, d_h=128, r=48, history T=4096 (current row "
                    "included), bf16 cache, fp32 accumulation, contiguous 64-token pages",
    "decode_T32768": "B=4, d=4096, H=32, d_h=128, r=32, T=32768, bf16 cache, fp32 accumulation",
    "ragged_paged": "B=64, lengths uniform on [256, 8192], 64-token pages shuffled in one pool, "
                    "H=16, d_h=128, r=56, d=2048 for the append, bf16",
    "decode_T4096_fp8": "decode_T4096 over an 8-bit cache: the four pools hold E4M3 codes (one "
                        "scale per pool), q, bases and output bf16, f16 tensor-core inputs, fp32 "
                        "accumulation",
    "decode_T4096_rope": "decode_T4096 with the exact rotary embedding (section 8): the cache keeps "
                         "unrotated projections, every key is scored at its distance from the query, "
                         "q~.(S_K D_j) + (C_j W_h).R_K with q~ = q D_i and (q D_(i-j)) B_K[h] = C_j W_h "
                         "(d_h*r multiply-adds per key and head, on tensor cores), then attention "
                         "with those scores; cos/sin table built once",
    "decode_T4096_norm": "decode_T4096 with joint key RMSNorm (section 8): a bf16 reciprocal per "
                         "head and token multiplies each score; the step appends the rows, stores "
                         "their reciprocals (lrkv_key_norms) and decodes",
    "decode_T4096_g2": "decode_T4096 with one shared basis per group of heads (section 3): G=2 "
                       "groups of 8 consecutive heads, each token caches 2 shared rows of d_h=128 "
                       "and r=32 private ranks per head (payload ratio 3/8 of multi-head "
                       "attention, against 7/16 for one basis with r=48), bf16",
    "prefill_2048": "B=8 fresh 2048-token prompts, d=2048, H=16, d_h=128, r=48, bf16: append "
                    "projection X.[W_S_K|W_S_V|U_K|U_V] then causal LRKV attention of every row",
}
# measured beside the headline in the same run (one entry each under "configs")
EXTRA_CONFIGS = "decode_T32768,ragged_paged,prefill_2048"
# the cache is drawn on the device for these (host drawing of 0.6-1.1 GB
# would dominate the run); every other workload uses the host generator
DEVICE_DRAWN = ("decode_T32768", "ragged_paged")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="decode_T4096", choices=sorted(WORKLOADS))
    ap.add_argument("--extra-configs", default=EXTRA_CONFIGS,
                    help="comma-separated workloads measured beside the headline ('none' for none)")
    ap.add_argument("--extra-steps", type=int, default=300,
                    help="timed steps of each extra workload")
    ap.add_argument("--roofline-launches", type=int, default=512,
                    help="launches the dominant kernel is timed over (outside the timed steps)")
    ap.add_argument("--cpu-workers", type=int, default=0,
                    help="host processes for the oracle timing (0: one per core)")
    ap.add_argument("--cpu-pairs", type=int, default=1024,
                    help="(request, head) pairs of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def rank_barrier(world):
    """Barrier across the ranks of a multi-process run (no-op on one)."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    """The largest of every rank's x (a duration): the job takes as long as
    its slowest rank.  device: where the process group's backend reduces
    (cuda for nccl, cpu for gloo)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks(key="hbm_gbs", fallback=FALLBACK_HBM_GBS):
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p[key]), "measured"
    except Exception:
        return fallback, "fallback"


def workload_shape(name):
    import lrkv_inputs as I
    c = dict(I.CONFIGS[name])
    c.setdefault("d", 2048)
    return c


def decode_lengths(name):
    """Sequence lengths of a decode workload (host only, no pools drawn)."""
    import numpy as np
    import lrkv_inputs as I
    c = I.CONFIGS[name]
    if name == "ragged_paged":
        return I.ragged_lengths(c["B"], c["lo"], c["hi"], c["seed"])
    return np.full(c["B"], c["T"], np.int32)


def cache_copies(cache_bytes):
    """Copies of the cache the timed steps rotate over: at least two, and
    enough that the working set is four times L2, so every step reads its
    cache from HBM (the previous step's rows are never the next step's)."""
    return max(2, math.ceil(4 * L2_BYTES / cache_bytes))


def describe(name, world):
    """The line's ``config`` object for a workload (both arms print the same)."""
    c = workload_shape(name)
    base = {"workload": f"{name}: {WORKLOADS[name]}", "B": c["B"], "d": c["d"], "H": c["H"],
            "d_h": c["d_h"], "r": c["r"], "parallelism": f"replicas x{world} (requests are independent)"}
    if name == "prefill_2048":
        base.update({"seq_len": c["T"], "rows": c["B"] * c["T"],
                     "l2": "no flush: one step's working set (~0.35 GB) exceeds L2",
                     "step": "lrkv_prefill (projection and placement of every row, then causal "
                             "attention of every row)"})
        return base
    lens = decode_lengths(name)
    G = c.get("groups", 1)
    eb = 1 if c["dtype"] == "fp8" else 2
    norm, rope = bool(c.get("norm")), bool(c.get("rope"))
    cached = int(lens.astype("int64").sum())
    pages = int(sum((int(L) + 63) // 64 for L in lens)) + (3 if name == "ragged_paged" else 0)
    cache_bytes = pages * 64 * (2 * (G * c["d_h"] + c["H"] * c["r"]) * eb + (2 * c["H"] if norm else 0))
    n = cache_copies(cache_bytes)
    base.update({"groups": G, "seq_len": int(lens.max()), "cached_rows": cached,
                 "l2": f"inputs larger than L2: the cache is rotated over {n} copies "
                       f"({n * cache_bytes / 1e6:.0f} MB working set vs 129 MB L2); no flush",
                 "step": ("lrkv_append (B new rows) + lrkv_decode_rope (B queries)" if rope else
                          "lrkv_decode_step (append of the B new rows" +
                          (", their reciprocal key norms" if norm else "") + ", decode of the B queries)")})
    if name in DEVICE_DRAWN:
        base["inputs"] = ("lengths, page table, queries and bases from the host generator; cache "
                          "pools N(0,1) bf16 drawn on the device by torch's seeded generator")
    return base


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        rows = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            rows = [r for r in out.strip().splitlines() if r.strip()]
        after = False
        if not rows:  # timed region shorter than one sampling period
            try:
                out = subprocess.run(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                      "--format=csv,noheader,nounits"], capture_output=True,
                                     text=True, timeout=10).stdout
                rows = [r for r in out.strip().splitlines() if r.strip()]
                after = True
            except Exception:
                rows = []
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "sampled_after_region": after}


class NvmlClockSampler:
    """SM clock and clock-event reasons of this process's GPU, read through the
    driver's NVML library (ctypes; read-only queries) by a host thread every
    ~0.2 ms.  The thread starts before the timed region; begin() and end()
    mark the region on the host clock and only the samples between the marks
    count, so that even a region of a few steps gets samples under load.
    ``available`` is False where NVML cannot be loaded; the caller then uses
    ClockSampler."""
    # clock-event reason bits (NVML's documented values)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index):
        import ctypes
        import threading
        import torch
        self.ct, self.threading = ctypes, threading
        self.available = False
        self.samples, self.max_mhz = [], None  # (host time, MHz, reason bits)
        self.t0 = self.t1 = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(cuda_index)
            bus = None
            if hasattr(props, "pci_bus_id"):
                bus = (f"{getattr(props, 'pci_domain_id', 0):08x}:{props.pci_bus_id:02x}:"
                       f"{getattr(props, 'pci_device_id', 0):02x}.0").encode()
            if bus is None or lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(h)) != 0:
                if lib.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(h)) != 0:
                    return
            self.lib, self.h = lib, h
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # 1: SM clock
                self.max_mhz = float(mx.value)
            self.available = True
        except Exception:
            self.available = False

    def _run(self):
        ct = self.ct
        mhz, bits = ct.c_uint(), ct.c_ulonglong()
        while not self.stop_flag.is_set():
            t = time.perf_counter()
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz)) == 0:
                b = 0
                if self.reasons_fn is not None and self.reasons_fn(self.h, ct.byref(bits)) == 0:
                    b = bits.value
                self.samples.append((t, float(mhz.value), b))
            time.sleep(0.0002)

    def start(self):
        self.stop_flag = self.threading.Event()
        self.thread = self.threading.Thread(target=self._run, daemon=True)
        self.thread.start()
        time.sleep(0.01)  # the thread is polling before the region begins

    def begin(self):
        self.t0 = time.perf_counter()

    def end(self):
        self.t1 = time.perf_counter()

    def stop(self):
        self.stop_flag.set()
        self.thread.join(timeout=5)
        t0 = self.t0 if self.t0 is not None else -math.inf
        t1 = self.t1 if self.t1 is not None else math.inf
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        bits = 0
        for x in inside:
            bits |= x[2]
        reasons = sorted(n for b, n in self.REASONS.items() if bits & b)
        return {"sm_mhz": statistics.median(x[1] for x in inside) if inside else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(inside),
                "sampled_after_region": False, "source": "nvml, in-process, ~0.2 ms period"}


def clock_sampler(cuda_index):
    """The in-process NVML sampler where NVML loads, else nvidia-smi."""
    s = NvmlClockSampler(cuda_index)
    return s if s.available else ClockSampler(cuda_index)


# ----------------------------------------------------------------------------
# committed ncu summaries
# ----------------------------------------------------------------------------
DECODE_SPLIT_SOURCES = ("decode_fast.cu", "decode_kernels.cuh", "lrkv_common.cuh")
PREFILL_SOURCES = ("prefill_tc.cu", "append_tc.cu", "tc_common.cuh", "tc_pair.cuh", "append_kernels.cuh",
                   "lrkv_common.cuh")
ROPE_SCORE_SOURCES = ("decode_fast.cu", "decode_kernels.cuh", "lrkv_common.cuh", "tc_common.cuh")


def kernel_source_hash(files=DECODE_SPLIT_SOURCES):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "rank_kv_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def summary_sections(path):
    """The '- key: value' figures of an ncu summary, per kernel: a section
    starts at a '- kernel: `name`' line and runs to the next one.  Figures
    before the first such line (the capture's source hash) belong to the
    file."""
    head, sections, cur = {}, {}, None
    for line in open(path):
        t = line.strip()
        if not (t.startswith("- ") and ":" in t):
            continue
        k, v = t[2:].split(":", 1)
        k, v = k.strip(), v.strip().split("  (")[0].strip().strip("`")
        if k == "kernel":
            cur = sections.setdefault(v, {})
        elif cur is None:
            head[k] = v
        else:
            cur[k] = v
    return head, sections


def profiled_traffic(summary, kernel, files):
    """DRAM bytes per launch of ``kernel`` from the committed ncu summary
    profiles/<summary>.md (read from that kernel's own section), or None if
    the file or section is absent or the capture was taken on a different
    kernel source."""
    path = os.path.join(ROOT, "profiles", f"{summary}.md")
    if not os.path.exists(path):
        return None
    head, sections = summary_sections(path)
    sec = sections.get(kernel)
    if sec is None:
        return None
    if head.get("kernel_source_sha256_16") != kernel_source_hash(files):
        return None
    try:
        return float(sec["dram_bytes_per_full_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------
# our arm: one decode workload
# ----------------------------------------------------------------------------
def profile_pass(lib, fn, n):
    """Run fn(i) n times with the library's per-kernel event pairs on and
    return {kind: (mean ms per launch, launches)}."""
    import ctypes
    import torch
    assert lib.lrkv_profile_enable(1) == 0
    for i in range(n):
        fn(i)
    torch.cuda.synchronize()
    out = {}
    for which in (0, 1, 2):
        tot, nl = ctypes.c_double(), ctypes.c_int32()
        assert lib.lrkv_profile_read(which, ctypes.byref(tot), ctypes.byref(nl)) == 0
        out[which] = (tot.value / nl.value if nl.value else None, nl.value)
    lib.lrkv_profile_enable(0)
    return out


def decode_leg(lib, name, dev, world, local_rank, K, W, R, Ke, headline):
    """Step timing, the split kernel's roofline and the end-to-end rate of
    one decode workload; returns the line's fields for it."""
    import ctypes
    import numpy as np
    import torch
    import lrkv_inputs as I
    import rank_kv_attention_gb300 as L
    from rank_kv_attention_gb300.api import PagedCache

    c = workload_shape(name)
    case = I.config_decode_case(name, device=dev if name in DEVICE_DRAWN else None)
    Bn, H, d_h, r, d = case.B, case.H, case.d_h, case.r, c["d"]
    G = case.groups
    w = I.make_weights(d, H, d_h, r, "bf16", seed=1, groups=G)
    x_new = I.make_append_case([1] * Bn, case.seq_lens - 1, d, seed=2).X

    def to_dev(a, kind="bf16"):
        if isinstance(a, torch.Tensor):
            return a.to(dev)
        if kind == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        if kind == "fp8":
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).view(torch.float8_e4m3fn).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    eb = 1 if case.dtype == "fp8" else 2   # bytes per cache element
    norm, rope = bool(c.get("norm")), bool(c.get("rope"))
    base = PagedCache(*(to_dev(t, case.dtype) for t in (case.S_K, case.S_V, case.R_K, case.R_V)),
                      tuple(case.scale))
    if norm:   # joint key norms of every cached row, written once before timing
        base.N_K = torch.empty((case.num_pages, case.page_size, case.H), dtype=torch.bfloat16,
                               device=dev)
        base.norm_eps = 1e-6
        allpos = np.concatenate([np.arange(Lr) for Lr in case.seq_lens]).astype(np.int32)
        allsid = np.concatenate([np.full(Lr, b) for b, Lr in enumerate(case.seq_lens)]).astype(np.int32)
        L.key_norms(to_dev(allpos, "i32"), to_dev(allsid, "i32"), to_dev(case.B_K), base,
                    to_dev(case.page_table, "i32"))
    cache_bytes = sum(t.numel() * eb for t in (base.S_K, base.S_V, base.R_K, base.R_V)) + \
        (base.N_K.numel() * 2 if norm else 0)
    n_copies = cache_copies(cache_bytes)
    caches = [base] + [PagedCache(*(t.clone() for t in (base.S_K, base.S_V, base.R_K, base.R_V)),
                                  base.scale, base.N_K.clone() if norm else None, base.norm_eps)
                       for _ in range(n_copies - 1)]
    q = to_dev(case.q)
    BK, BV = to_dev(case.B_K), to_dev(case.B_V)
    Wsk, Wsv, Uk, Uv = (to_dev(a) for a in (w.W_S_K, w.W_S_V, w.U_K, w.U_V))
    X = to_dev(x_new)
    pos = to_dev(case.seq_lens - 1, "i32")
    sid = to_dev(np.arange(Bn), "i32")
    seq_lens = to_dev(case.seq_lens, "i32")
    pt = to_dev(case.page_table, "i32")
    max_seq = int(case.seq_lens.max())
    out = torch.empty_like(q)
    ws = L.workspace(max(L.decode_step_workspace_bytes(Bn, H, d_h, r, max_seq),
                         L.decode_rope_workspace_bytes(Bn, H, d_h, r, max_seq) if rope else 0), dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    descs = [cc.desc() for cc in caches]

    def make_calls(X_, q_, pos_, sid_, sl_, out_):
        calls = []
        for dsc in descs:
            a = (P(X_), P(pos_), P(sid_), Bn, d, P(Wsk), P(Wsv), P(Uk), P(Uv), ctypes.byref(dsc),
                 P(pt), Bn, pt.shape[1], P(status), sp)
            dd = (P(q_), ctypes.byref(dsc), P(BK), P(BV), P(sl_), P(pt), Bn, pt.shape[1], max_seq,
                  P(out_), P(ws), ws.numel(), P(status), sp)
            fs = (P(X_), d, P(Wsk), P(Wsv), P(Uk), P(Uv), P(q_), ctypes.byref(dsc), P(BK), P(BV),
                  P(sl_), P(pt), Bn, pt.shape[1], max_seq, P(out_), P(ws), ws.numel(), P(status), sp)
            kn = (P(pos_), P(sid_), Bn, P(BK), ctypes.byref(dsc), P(pt), Bn, pt.shape[1], P(status), sp)
            calls.append((a, dd, fs, kn))
        return calls

    if rope:   # the cos/sin table is built once, outside every timed region
        table = L.rope_table(d_h, max_seq, device=dev)
        rope_args = (P(table.buf), table.max_pos)

        def dec_rope(q_, dsc, BK_, BV_, sl_, pt_, B_, mp_, msl_, out_, ws_, wsn_, st_, s_):
            return lib.lrkv_decode_rope(q_, dsc, BK_, BV_, sl_, pt_, B_, mp_, msl_, *rope_args,
                                        out_, ws_, wsn_, st_, s_)
    calls = make_calls(X, q, pos, sid, seq_lens, out)
    f_app, f_dec, f_step = lib.lrkv_append, (dec_rope if rope else lib.lrkv_decode), lib.lrkv_decode_step

    def step(i):
        # one decode step: append the B new rows (with their key norms when
        # the cache keeps them) and decode the B queries -- one
        # lrkv_decode_step call; the rotary path calls lrkv_append, then
        # lrkv_decode_rope
        a, dd, fs, _ = calls[i % n_copies]
        if rope:
            rc, rc2 = f_app(*a), f_dec(*dd)
        else:
            rc, rc2 = f_step(*fs), 0
        if rc or rc2:
            raise RuntimeError(f"lrkv call failed: {rc} {rc2}")

    def separate(i):
        # the same step as separate calls: lrkv_append, [lrkv_key_norms,] lrkv_decode
        a, dd, _, kn = calls[i % n_copies]
        rc = f_app(*a)
        rc3 = lib.lrkv_key_norms(*kn) if norm else 0
        rc2 = f_dec(*dd)
        if rc or rc2 or rc3:
            raise RuntimeError(f"lrkv call failed: {rc} {rc3} {rc2}")

    barrier = lambda: rank_barrier(world)
    ranks_max = lambda x: max_over_ranks(x, world, dev)

    # ---- device-resident timed region (step throughput): exactly K steps
    for i in range(max(W, 3)):
        step(i)
    torch.cuda.synchronize()
    barrier()
    clocks = clock_sampler(local_rank)
    if isinstance(clocks, ClockSampler):  # nvidia-smi needs a moment to start sampling
        clocks.start()
        time.sleep(0.25)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nvml = not isinstance(clocks, ClockSampler)
    if nvml:
        clocks.start()
        clocks.begin()
    e0.record(stream)
    for i in range(K):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    if nvml:
        clocks.end()
    clk = clocks.stop()
    barrier()
    total_ms = ranks_max(e0.elapsed_time(e1))

    # ---- live breakdown: the calls of a step on their own
    def timed(fn, n):
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for i in range(n):
            fn(i)
        a1.record(stream)
        torch.cuda.synchronize()
        return a0.elapsed_time(a1) / n
    nb = max(K, R)
    append_ms = timed(lambda i: f_app(*calls[i % n_copies][0]), nb)
    decode_ms = timed(lambda i: f_dec(*calls[i % n_copies][1]), nb)
    separate_ms = None if rope else timed(separate, nb)

    # ---- the dominant kernel's own duration over R launches: the library
    # brackets each launch with CUDA events on its stream (outside the timed
    # steps above, so those events do not perturb the step timing)
    prof = profile_pass(lib, step, R)
    split_ms, n_split = prof[0]
    scores_ms, n_scores = prof[2]
    st = int(status.item())
    if st:
        raise RuntimeError(f"device status {st}")

    # ---- end to end through the C ABI with host buffers
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    d2h = hout.numel() * hout.element_size()
    if not rope:
        # a step graph (lrkv_step_graph_create, one per rotated cache copy)
        # replays lrkv_decode_step_host: X, q and the lengths in pinned host
        # memory are copied in, the step runs and out is copied back, with one
        # launch; the host then waits for the result
        hX, hq, hsl = (t.cpu().contiguous().pin_memory() for t in (X, q, seq_lens))
        ws_h = L.workspace(L.decode_step_host_workspace_bytes(Bn, H, d_h, r, d, max_seq), dev)
        graphs = []
        for dsc in descs:
            hg = ctypes.c_void_p()
            rc = lib.lrkv_step_graph_create(ctypes.byref(hg), P(hX), d, P(Wsk), P(Wsv), P(Uk), P(Uv),
                                            P(hq), ctypes.byref(dsc), P(BK), P(BV), P(hsl), P(pt), Bn,
                                            pt.shape[1], max_seq, P(hout), P(ws_h), ws_h.numel(),
                                            P(status))
            if rc:
                raise RuntimeError(f"lrkv_step_graph_create failed: {rc}")
            graphs.append(hg)
        h2d = sum(t.numel() * t.element_size() for t in (hX, hq, hsl))
        e2e_note = ("lrkv_step_graph_launch (lrkv_decode_step_host as a graph): pinned host X, q "
                    "and lengths copied in by a copy kernel through their device-mapped "
                    "addresses, the step, out written back to pinned host memory by the decode's "
                    "last kernel, then the host synchronises; every step")

        def e2e_step(i):
            rc = lib.lrkv_step_graph_launch(graphs[i % n_copies], sp)
            if rc:
                raise RuntimeError(f"lrkv_step_graph_launch failed: {rc}")
            stream.synchronize()   # the host reads this step's result
    else:
        # the rotary path: the step's inputs (new rows, queries, lengths,
        # positions, ids) live in one pinned host staging buffer and move with
        # one copy; the C-ABI calls take device views of its device twin
        # (256-byte aligned)
        parts = (X, q, seq_lens, pos, sid)
        offs, o = [], 0
        for t in parts:
            offs.append(o)
            o += (t.numel() * t.element_size() + 255) // 256 * 256
        hbuf = torch.empty(o, dtype=torch.uint8).pin_memory()
        dbuf = torch.empty(o, dtype=torch.uint8, device=dev)
        views = []
        for t, a in zip(parts, offs):
            nbytes = t.numel() * t.element_size()
            hbuf[a:a + nbytes].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
            views.append(dbuf[a:a + nbytes].view(t.dtype).view(t.shape))
        dX, dq, dsl, dpos, dsid = views
        dout = torch.empty_like(out)
        calls = make_calls(dX, dq, dpos, dsid, dsl, dout)
        h2d = hbuf.numel()   # the staging buffer as copied (payload rounded up to 256 B per input)
        e2e_note = ("pinned host inputs (one staging buffer) copied in, result copied out and "
                    "synchronised every step")

        def e2e_step(i):
            dbuf.copy_(hbuf, non_blocking=True)
            step(i)
            hout.copy_(dout, non_blocking=True)
            stream.synchronize()   # the host reads this step's result

    for i in range(5):
        e2e_step(i)
    barrier()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for i in range(Ke):
        e2e_step(i)
    g1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = ranks_max(g0.elapsed_time(g1))
    if not rope:
        for hg in graphs:
            lib.lrkv_step_graph_destroy(hg)

    # ---- numbers
    ms_step = total_ms / K
    value = world * Bn * K / (total_ms / 1e3)
    seq_total = int(case.seq_lens.astype(np.int64).sum())
    split_bytes = seq_total * (2 * (G * d_h + H * r) * eb + (2 * H if norm else 0))  # cache rows read once
    step_bytes = (split_bytes + 2 * H * d_h * r * 2 + 2 * Bn * H * d_h * 2   # + bases, q, out
                  + (2 * G * d_h + 2 * H * r) * d * 2 + Bn * d * 2)         # + append W, X
    peak, peak_kind = measured_peaks()
    bf16_peak, bf16_kind = measured_peaks("bf16_tflops", FALLBACK_BF16_TFLOPS)
    if rope:
        # the rotary score kernel reads S_K and R_K once and writes one fp32
        # score per row and head: an HBM-bound pass (about 104 flops per byte,
        # below the tensor/HBM ridge of ~290); its contractions per key and
        # head, 2 (d_h r + r + d_h) flops, are reported beside it
        score_bytes = seq_total * ((d_h + H * r) * eb + 4 * H)
        gsplit_bytes = seq_total * ((d_h + H * r) * eb + 4 * H)   # S_V, R_V and the scores
        rope_flops = seq_total * H * 2 * (d_h * r + r + d_h)
        ach = score_bytes / (scores_ms / 1e3) / 1e9
        roof = {"kernel": "rotary score kernel (tcgen05: C_j W_h private products and the rotated "
                          "shared term; S_K and R_K read once, one fp32 score per row and head written)",
                "bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "peak_source": f"{peak_kind} HBM copy bandwidth",
                "frac_of_8TBs": round(ach / NORTH_STAR_HBM_GBS, 4),
                "algorithmic_bytes_per_launch": score_bytes,
                "avg_launch_ms": round(scores_ms, 5), "launches_timed": n_scores,
                "flops_per_launch": rope_flops,
                "tflops": round(rope_flops / (scores_ms / 1e3) / 1e12, 1),
                "tensor_frac_of_bf16_peak": round(rope_flops / (scores_ms / 1e3) / 1e12 / bf16_peak, 4),
                "given_score_split": {"avg_launch_ms": round(split_ms, 5),
                                      "algorithmic_bytes_per_launch": gsplit_bytes,
                                      "hbm_gbs": round(gsplit_bytes / (split_ms / 1e3) / 1e9, 1),
                                      "frac_of_hbm": round(gsplit_bytes / (split_ms / 1e3) / 1e9 / peak, 4)},
                "traffic": profiled_traffic(f"rope_scores_{name}", "rope_scores_tc_kernel",
                                            ROPE_SCORE_SOURCES)}
    else:
        achieved = split_bytes / (split_ms / 1e3) / 1e9
        roof = {"kernel": "decode split (factored scores, online softmax, value reductions; its "
                          "last phase merges each request's segments and expands by B_V)",
                "bound": "hbm", "achieved": round(achieved, 1),
                "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "peak_source": f"{peak_kind} HBM copy bandwidth",
                "frac_of_8TBs": round(achieved / NORTH_STAR_HBM_GBS, 4),
                "algorithmic_bytes_per_launch": split_bytes,
                "avg_launch_ms": round(split_ms, 5), "launches_timed": n_split,
                "traffic": profiled_traffic(f"decode_split_{name}", "decode_split_fast_kernel",
                                            DECODE_SPLIT_SOURCES)}
    res = {
        "value": round(value, 1), "unit": "tokens/s", "ms_per_step": round(ms_step, 5),
        "dtype": "e4m3 cache, f16 mma inputs" if eb == 1 else "bf16",
        "config": describe(name, world),
        "roofline": roof,
        "step_effective_gbs": round(step_bytes / (ms_step / 1e3) / 1e9, 1),
        "step_frac_of_hbm": round(step_bytes / (ms_step / 1e3) / 1e9 / peak, 4),
        "breakdown_ms": {"split_kernel": round(split_ms, 5),
                         "rotary_score_kernel": None if scores_ms is None else round(scores_ms, 5),
                         "lrkv_append_alone": round(append_ms, 5),
                         "lrkv_decode_alone": round(decode_ms, 5),
                         "lrkv_append_then_lrkv_decode": None if separate_ms is None else round(separate_ms, 5)},
        "e2e": {"value": round(world * Bn * Ke / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke,
                "note": e2e_note},
        # per step: append, [key norms,] prologue, [rotary scores,] split (the
        # split kernel's last phase merges the segments; no combine launch)
        "gpu_launches": (3 + int(norm) + int(rope)) * K,
        "clocks": clk,
    }
    del caches, base
    return res


# ----------------------------------------------------------------------------
# our arm: prefill
# ----------------------------------------------------------------------------
def prefill_leg(lib, name, dev, world, local_rank, K, W, R, Ke):
    """Step timing (one lrkv_prefill over the batch), the attention and
    projection kernels' rooflines and the end-to-end rate of the prefill
    workload."""
    import ctypes
    import numpy as np
    import torch
    import lrkv_inputs as I
    import rank_kv_attention_gb300 as L
    from rank_kv_attention_gb300 import _abi
    from rank_kv_attention_gb300.api import PagedCache

    c = I.CONFIGS[name]
    Bq, d, H, d_h, r, T = c["B"], c["d"], c["H"], c["d_h"], c["r"], c["T"]
    n = Bq * T
    ac = I.make_append_case([T] * Bq, [0] * Bq, d, dtype="bf16", seed=c["seed"], shuffle=True)
    w = I.make_weights(d, H, d_h, r, "bf16", seed=c["seed"])
    rng = np.random.default_rng(99)
    Q = I.f32_to_bf16_bits(rng.standard_normal((n, H, d_h)).astype(np.float32))

    def to_dev(a, kind="bf16"):
        if kind == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    cache = PagedCache.empty(ac.num_pages, 64, H, d_h, r, torch.bfloat16, dev)
    X, Qd = to_dev(ac.X), to_dev(Q)
    Wt = [to_dev(a) for a in (w.W_S_K, w.W_S_V, w.U_K, w.U_V, w.B_K, w.B_V)]
    cu = to_dev(np.arange(0, n + 1, T), "i32")
    sp = to_dev(np.zeros(Bq), "i32")
    pt = to_dev(ac.page_table, "i32")
    out = torch.empty_like(Qd)
    ws = L.workspace(L.prefill_workspace_bytes(Bq, n, H, d_h, r, T), dev)
    stream = torch.cuda.current_stream(dev)

    def step(i=0):
        L.prefill(X, Qd, cu, sp, T, *Wt, cache, pt, out=out, ws=ws, stream=stream)

    for _ in range(max(W, 3)):
        step()
    torch.cuda.synchronize()
    rank_barrier(world)
    clocks = clock_sampler(local_rank)
    if isinstance(clocks, ClockSampler):  # nvidia-smi needs a moment to start sampling
        clocks.start()
        time.sleep(0.25)
    torch.cuda.synchronize()
    rank_barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nvml = not isinstance(clocks, ClockSampler)
    if nvml:
        clocks.start()
        clocks.begin()
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    if nvml:
        clocks.end()
    clk = clocks.stop()
    rank_barrier(world)
    total_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    prof = profile_pass(lib, step, R)
    attn_ms, n_attn = prof[0]
    proj_ms, n_proj = prof[1]

    # ---- end to end with host buffers: the step's rows X and queries Q from
    # pinned host memory, the output back to pinned host memory, the host
    # synchronising every step
    hX, hQ = X.cpu().pin_memory(), Qd.cpu().pin_memory()
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e_step():
        X.copy_(hX, non_blocking=True)
        Qd.copy_(hQ, non_blocking=True)
        step()
        hout.copy_(out, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    rank_barrier(world)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(Ke):
        e2e_step()
    g1.record(stream)
    torch.cuda.synchronize()
    rank_barrier(world)
    e2e_ms = max_over_ranks(g0.elapsed_time(g1), world, dev) / Ke
    h2d = hX.numel() * hX.element_size() + hQ.numel() * hQ.element_size()
    d2h = hout.numel() * hout.element_size()
    tiled = lib.lrkv_prefill_kernel_kind(ctypes.byref(cache.desc())) == _abi.LRKV_PREFILL_TILED

    ms = total_ms / K
    Ntot = 2 * d_h + 2 * H * r
    proj_flops = 2 * n * d * Ntot
    peak, kind = measured_peaks("bf16_tflops", FALLBACK_BF16_TFLOPS)
    # attention: per (row, head) with v visible keys, scores and values cost
    # 2 v (d_h + r) each; p = q B_K[h] and the B_V[h] expansion 2 d_h r each
    visible = Bq * T * (T + 1) // 2
    attn_flops = H * (4 * visible * (d_h + r) + 4 * n * d_h * r)
    attn_tf = attn_flops / (attn_ms / 1e3) / 1e12
    proj_tf = proj_flops / (proj_ms / 1e3) / 1e12
    res = {
        "value": round(world * n / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 5),
        "dtype": "bf16", "config": describe(name, world),
        "roofline": {"kernel": "prefill_tc_kernel (causal attention, tcgen05)", "bound": "tensor",
                     "achieved": round(attn_tf, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(attn_tf / peak, 4), "peak_source": f"{kind} bf16 GEMM (burst)",
                     "flops_per_launch": attn_flops, "avg_launch_ms": round(attn_ms, 5),
                     "launches_timed": n_attn,
                     "traffic": profiled_traffic(f"prefill_attention_{name}", "prefill_tc_kernel",
                                                 PREFILL_SOURCES)},
        "projection": {"kernel": "append_tc_kernel (X.[W_S_K|W_S_V|U_K|U_V], tcgen05)",
                       "bound": "tensor", "achieved": round(proj_tf, 1), "peak": peak,
                       "unit": "TFLOP/s", "frac": round(proj_tf / peak, 4),
                       "flops_per_launch": proj_flops, "avg_launch_ms": round(proj_ms, 5),
                       "launches_timed": n_proj,
                       "traffic": profiled_traffic(f"prefill_attention_{name}", "append_tc_kernel",
                                                   PREFILL_SOURCES)},
        "breakdown_ms": {"projection": round(proj_ms, 5), "attention": round(attn_ms, 5)},
        "e2e": {"value": round(world * n / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke,
                "note": "pinned host X and Q copied in, lrkv_prefill, out copied back and "
                        "synchronised every step"},
        # per step: row metadata, the projection, the attention (tiled path)
        "gpu_launches": 3 * K if tiled else None,
        "clocks": clk,
    }
    return res


def run_ours(args, rank, world, local_rank):
    import torch
    import rank_kv_attention_gb300 as L

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    lib = L.lib()
    K, W, R = args.steps, args.warmup, max(1, args.roofline_launches)
    Ke = args.e2e_steps or max(50, min(K, 2000))
    name = args.config
    if name == "prefill_2048":
        head = prefill_leg(lib, name, dev, world, local_rank, K, W, R, args.e2e_steps or max(3, min(K, 50)))
    else:
        head = decode_leg(lib, name, dev, world, local_rank, K, W, R, Ke, True)
    res = {"metric": PREFILL_METRIC if name == "prefill_2048" else METRIC, "value": head["value"],
           "unit": head["unit"], "n_gpus": world, "steps": K, "warmup": W,
           "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic"}
    res.update({k: v for k, v in head.items() if k not in res})
    extras = [x for x in (args.extra_configs or "").split(",") if x and x not in (name, "none")]
    if extras:
        res["configs"] = {}
        for x in extras:
            torch.cuda.empty_cache()
            if x == "prefill_2048":
                leg = prefill_leg(lib, x, dev, world, local_rank, max(3, args.extra_steps // 6), 5,
                                  R, 20)
            else:
                leg = decode_leg(lib, x, dev, world, local_rank, args.extra_steps, 10, R, 200, False)
            res["configs"][x] = {"metric": PREFILL_METRIC if x == "prefill_2048" else METRIC, **leg}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = (cpu_baseline_prefill(name, args.cpu_workers) if name == "prefill_2048"
                               else cpu_baseline(name, args.cpu_pairs, args.cpu_workers))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return res


# ----------------------------------------------------------------------------
# the oracle on host cores (cpu_baseline and the reference arm)
# ----------------------------------------------------------------------------
def oracle_decode_sample(name, n_pairs, workers=0):
    """The float64 oracle on ``n_pairs`` seeded (request, head) pairs of a
    decode workload, on all host cores: the one sample both the line's
    cpu_baseline and the reference arm report."""
    from oracle.cpu_timing import time_oracle_decode
    t = time_oracle_decode(name, n_pairs, workers=workers or None)
    return {"value": round(t["pairs"] / t["heads"] / t["wall_s"], 3), "unit": "tokens/s",
            "cores": t["cores"], "nproc": os.cpu_count(), "kind": "oracle",
            "sample": f"{t['pairs']} seeded random (request, head) pairs of the {name} workload "
                      f"({t['pairs'] / t['heads']:.0f} request-steps), float64 oracle "
                      f"(gather, materialise K_h/V_h, textbook softmax), {t['cores']} single-"
                      f"threaded processes (spawned and warmed before timing), "
                      f"{t['cpu_s']:.1f} s CPU, {t['wall_s']:.2f} s wall",
            "wall_s": t["wall_s"]}


def cpu_baseline(name, n_pairs, workers=0):
    """The oracle on all host cores (the reported value), and once more on one
    core over a proportionally smaller sample."""
    from oracle.cpu_timing import time_oracle_decode
    out = oracle_decode_sample(name, n_pairs, workers)
    n1 = max(4, n_pairs // max(1, out["cores"]))
    t1 = time_oracle_decode(name, n1, workers=1, seed=1)
    out.pop("wall_s")
    out["single_core"] = {"value": round(t1["pairs"] / t1["heads"] / t1["wall_s"], 3),
                          "unit": "tokens/s", "cores": 1,
                          "sample": f"{t1['pairs']} random (request, head) pairs, one process"}
    return out


def cpu_baseline_prefill(name, workers=0, k_rows=8):
    from oracle.cpu_timing import time_oracle_prefill
    t = time_oracle_prefill(name, k_rows, workers=workers or None)
    return {"value": round(t["tokens_per_s"], 3), "unit": "tokens/s", "cores": t["cores"],
            "nproc": os.cpu_count(), "kind": "oracle",
            "sample": f"{t['cores']} requests of the {name} workload, one per single-threaded "
                      f"process: the float64 projection of the request's rows, then causal "
                      f"attention of {k_rows} sampled rows (all heads), scaled to the full "
                      f"request; {t['wall_s']:.1f} s wall"}


def run_reference(args, rank, world):
    """The float64 oracle timed on host cores, on the same workload, config
    and sample as our line's cpu_baseline (rank 0 alone; other ranks exit)."""
    if rank != 0:
        return None
    c = workload_shape(args.config)
    if args.config == "prefill_2048":   # the prefill line's metric, on host cores
        cb = cpu_baseline_prefill(args.config, args.cpu_workers)
        v = cb["value"]
        metric, ms = PREFILL_METRIC, c["B"] * c["T"] / v * 1e3
    else:
        cb = oracle_decode_sample(args.config, args.cpu_pairs, args.cpu_workers)
        v = cb["value"]
        metric, ms = METRIC, c["B"] / v * 1e3
        cb.pop("wall_s")
    return {
        "impl": "reference", "metric": metric, "value": v, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": describe(args.config, world),
        "cpu_baseline": cb,
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
