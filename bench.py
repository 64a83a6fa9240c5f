#!/usr/bin/env python
"""fp8 paged decode attention benchmark (libfp8kv on GB300).

One step = one decode step of one attention layer: fp8kv_quant_append of
every sequence's newest K/V row into the paged E4M3 cache, then
fp8kv_paged_decode over the whole cache (all steps of the hot path).  The
default workload is the Llama-3.1-8B serving batch (32 q / 8 kv heads,
head_dim 128, batch 8, contexts uniform in 18000..22000, block_size 16,
shuffled physical blocks).

Printed (rank 0, one JSON line): whole-step algorithmic GB/s and us/step, the
roofline of the decode call against the measured HBM peak, an end-to-end
number through host (pinned) buffers, SM clocks sampled during the timed
region, and the CPU oracle timed on the host cores.

Timing: W warm-up steps, then K timed steps back to back between one pair of
CUDA events on the stream the library launches on; barrier + synchronize
around the region; max over ranks.  The inputs are larger than L2: a workload
that streams less than 1.5x the L2 size per step gets several copies of its
cache ("layers", as the attention layers of one model have), and step i reads
layer i mod n, so that a layer's pages have left L2 before it comes round
again.  Where the copies would not fit in 8 GB (the windowed workloads, which
read a small part of a large cache) every step is timed alone after an L2
flush (a device write larger than L2, then a read of another buffer larger
than L2, so that L2 holds no dirty lines), outside the events.  With --gpus N > 1 (torchrun) every rank runs an independent replica
(the path does not exchange data between GPUs).

--impl reference times the CPU oracle (the only other implementation of this
path) on the host cores, one bounded sample of the same workload per step.
"""
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from fp8_kv_cache_fp8kv_gb300 import accounting, workload  # noqa: E402

METRIC = "fp8 paged decode attention: achieved HBM GB/s and % of GB300 peak; µs/decode step"
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 256 << 20


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["fp8kv", "reference"], default="fp8kv")
    p.add_argument("--config", default="llama31_8b_b8_20k", choices=list(workload.CONFIGS))
    p.add_argument("--window", type=int, default=None, help="default: the workload's first window")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--no-per-config", action="store_true",
                   help="time only --config (the default run also times the 128K needle workload as its own record)")
    p.add_argument("--sweep-layout", choices=list(SWEEP_LAYOUTS), default="llama",
                   help="head layout of the --sweep layer")
    p.add_argument("--sweep", action="store_true",
                   help="instead of the step: decode time against context length, fp8 cache and bf16 cache")
    p.add_argument("--copy-probe", action="store_true",
                   help="instead of the step: build and run the copy-pipeline probe (csrc/probe/copy_probe.cu), "
                        "the page-streaming rates the decode kernel's design rests on")
    p.add_argument("--prefill", type=str, default=None, metavar="CHUNKS",
                   help="instead of the step: chunked prefill over the fp8 cache of --config, the last CHUNK "
                        "tokens of every sequence as queries, for each comma-separated CHUNK")
    a = p.parse_args(argv)
    a.warmup = max(3, a.warmup)
    a.steps = max(1, a.steps)
    return a


# ---------------------------------------------------------------- distributed

def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, ws


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x, ws):
    """Maximum of a float over ranks (every rank gets it)."""
    if ws <= 1:
        return float(x)
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- measurement helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBps", "hbm"):
            if key in d:
                return float(d[key]), "measured (MEASURED_PEAKS.json)"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback (no MEASURED_PEAKS.json)"


FALLBACK_BF16_TFLOPS = 1900.0


def measured_tensor_peak():
    """Dense bf16 tensor TFLOP/s as a burst (the f16 MMA has the same nominal rate)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("bf16_tflops", "bf16_TFLOPs", "bf16"):
            if key in d:
                return float(d[key]), "measured (MEASURED_PEAKS.json)"
    except (OSError, ValueError):
        pass
    return FALLBACK_BF16_TFLOPS, "fallback (no MEASURED_PEAKS.json)"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 100 ms in a thread."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 5:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        scope = "during timed region"
        if not inside:
            near = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            inside = [p for _, p in near]
            scope = "nearest samples (timed region shorter than the 100 ms sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "scope": "nvidia-smi unavailable"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "scope": scope}


def traffic_for(kernel_key):
    """DRAM bytes per launch recorded from an ncu capture of this kernel, if the
    kernel source is unchanged since (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    ent = d.get(kernel_key)
    if not ent:
        return None
    if ent.get("source_sha256") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_kv_cache_fp8kv_gb300", "csrc")
    for name in ("paged_decode.cu", "partition.cuh", "walk.cuh", "ptx.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


class L2Policy:
    """An L2 flush between timed calls when a call streams less than 1.5x the
    L2 size (else nothing to flush: inputs larger than L2): a device buffer
    larger than L2 is written, then another one read, so that the next call
    starts with none of its inputs in L2 and no dirty lines to write back."""

    def __init__(self, step_read_bytes, device):
        self.l2 = int(torch.cuda.get_device_properties(device).L2_cache_size)
        self.read = int(step_read_bytes)
        self.buf = self.rbuf = None
        if self.read <= 3 * self.l2 // 2:
            n = max(FLUSH_BYTES, 2 * self.l2)
            self.buf = torch.empty(n, dtype=torch.uint8, device=device)
            self.rbuf = torch.ones(n, dtype=torch.uint8, device=device)

    def __call__(self):
        if self.buf is not None:
            self.buf.zero_()
            self.rbuf.sum(dtype=torch.int64)

    def describe(self):
        if self.buf is None:
            return ("inputs larger than L2: %.0f MB read per step vs %.0f MB L2, no flush"
                    % (self.read / 1e6, self.l2 / 1e6))
        return ("flushed before every timed step (%.0f MiB device write, then a %.0f MiB read, vs %.0f MB L2; "
                "outside the events)" % (self.buf.numel() / 2 ** 20, self.rbuf.numel() / 2 ** 20, self.l2 / 1e6))


class NoFlush:
    buf = None

    def __call__(self):
        pass


LAYER_BUDGET_BYTES = 8 << 30   # device memory the extra layer caches may take


def layer_plan(read_bytes, cache_bytes, device):
    """How a decode workload keeps its inputs out of L2 between timed steps:
    (layers, flush).  More than 1.5x L2 read per step: one layer, no flush.
    Otherwise n = ceil(3 x L2 / read) copies of the cache, read in turn (the
    other n - 1 layers stream at least 2x L2 between two visits of a layer),
    when they fit in LAYER_BUDGET_BYTES; else one layer and an L2 flush before
    every timed step."""
    l2 = int(torch.cuda.get_device_properties(device).L2_cache_size)
    if read_bytes > 3 * l2 // 2:
        return 1, NoFlush()
    n = -(-3 * l2 // max(1, int(read_bytes)))
    if n * cache_bytes <= LAYER_BUDGET_BYTES:
        return n, NoFlush()
    return 1, L2Policy(read_bytes, device)


def describe_layers(layers, flush, read_bytes, cache_bytes, device):
    l2 = int(torch.cuda.get_device_properties(device).L2_cache_size)
    if flush.buf is not None:
        return flush.describe()
    if layers == 1:
        return "inputs larger than L2: %.0f MB read per step vs %.0f MB L2, no flush" % (read_bytes / 1e6, l2 / 1e6)
    return ("inputs larger than L2: %d copies of the %.0f MB cache (layers), step i reads layer i mod %d; "
            "%.0f MB read per step, %.0f MB by the other layers between two visits of one, vs %.0f MB L2"
            % (layers, cache_bytes / 1e6, layers, read_bytes / 1e6, (layers - 1) * read_bytes / 1e6, l2 / 1e6))


# ---------------------------------------------------------------- the CUDA path

class DecodeStep:
    """Device state of one workload and one decode step through the C ABI.
    With layers > 1 the cache is copied that many times (the KV caches of
    consecutive attention layers) and each call goes to the next layer."""

    def __init__(self, w, window, device, layers=1):
        from fp8_kv_cache_fp8kv_gb300 import binding as fk
        self.fk = fk
        fk.load(build_if_missing=True)
        s = w.shape
        self.w, self.window, self.dev = w, window, device
        shape = (w.num_blocks, s.num_kv_heads, workload.BLOCK_SIZE, s.head_dim)
        k_cache = torch.zeros(shape, dtype=torch.uint8, device=device)
        v_cache = torch.zeros(shape, dtype=torch.uint8, device=device)
        fk.fp8kv_quant_append(w.k.to(device), w.v.to(device), w.slot_mapping.to(device),
                              k_cache, v_cache, w.k_scale, w.v_scale)
        self.caches = [(k_cache, v_cache)] + [(k_cache.clone(), v_cache.clone()) for _ in range(layers - 1)]
        self.k_cache, self.v_cache = k_cache, v_cache
        self.cache_bytes = 2 * k_cache.numel()
        rows = w.new_token_rows()
        self.h_q = w.q.contiguous()
        self.h_k_new = w.k[rows].contiguous()
        self.h_v_new = w.v[rows].contiguous()
        self.h_slots = w.slot_mapping[rows].contiguous()
        # the inputs that change every step (q, the new K/V rows, the lengths)
        # share one device buffer, so that a step's host-to-device transfer is
        # one copy (the e2e measurement); each is a 256-byte-aligned view
        parts = [self.h_q, self.h_k_new, self.h_v_new, w.seq_lens.contiguous()]
        offs, total = [], 0
        for t in parts:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        self.h_inputs = torch.zeros(total, dtype=torch.uint8)
        for t, o in zip(parts, offs):
            n = t.numel() * t.element_size()
            self.h_inputs[o:o + n] = t.view(torch.uint8).reshape(-1)
        self.inputs = self.h_inputs.to(device)

        def view(i):
            t = parts[i]
            n = t.numel() * t.element_size()
            return self.inputs[offs[i]:offs[i] + n].view(t.dtype).view(t.shape)

        self.q, self.k_new, self.v_new, self.seq_lens = view(0), view(1), view(2), view(3)
        self.slots = self.h_slots.to(device)
        self.block_tables = w.block_tables.to(device)
        self.out = torch.empty_like(self.q)
        self.ws = fk.alloc_workspace(w.q.shape[0], s.num_q_heads, s.num_kv_heads, s.head_dim,
                                     w.max_seq_len, 16, window, device=device)
        torch.cuda.synchronize()

        self._append, self._decode, self._step = [], [], []
        self._decode_engine = {fk.ENGINE_TENSOR_CORES: [], fk.ENGINE_CUDA_CORES: []}
        for kc, vc in self.caches:
            self._append.append(fk.prepare_quant_append(self.k_new, self.v_new, self.slots, kc, vc,
                                                        w.k_scale, w.v_scale))
            self._decode.append(fk.prepare_paged_decode(self.q, kc, vc, self.block_tables, self.seq_lens,
                                                        w.max_seq_len, w.k_scale, w.v_scale, w.sm_scale, window,
                                                        self.out, self.ws))
            for e in self._decode_engine:
                self._decode_engine[e].append(
                    fk.prepare_paged_decode(self.q, kc, vc, self.block_tables, self.seq_lens, w.max_seq_len,
                                            w.k_scale, w.v_scale, w.sm_scale, window, self.out, self.ws, engine=e))
            self._step.append(fk.prepare_decode_step(self.q, self.k_new, self.v_new, kc, vc, self.block_tables,
                                                     self.seq_lens, w.max_seq_len, w.k_scale, w.v_scale,
                                                     w.sm_scale, window, self.out, self.ws))
        self.layer = 0

    @property
    def layers(self):
        return len(self.caches)

    def _next(self):
        i = self.layer
        self.layer = (i + 1) % len(self.caches)
        return i

    def append(self):
        self._append[self._next()]()

    def decode(self):
        self._decode[self._next()]()

    def decode_engine(self, engine):
        self._decode_engine[engine][self._next()]()

    def step(self):
        """The decode step: every sequence's newest row appended, then attended."""
        self._step[self._next()]()


PER_CONFIG = ("llama33_70b_needle_128k",)   # also timed, as their own records, in a default run


def time_steps(st, K, flush, stream):
    """The timed region: K decode steps, returned as total milliseconds and a
    description.  Inputs larger than L2 (directly, or through the rotation
    over layer caches): the K steps run back to back between one pair of CUDA
    events.  Otherwise an L2 flush before every step, outside per-step
    events."""
    if flush.buf is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            st.step()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1), "one CUDA-event pair around the K back-to-back steps"
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        st.step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(K)), "CUDA events around each step (L2 flushed before each)"


def isolated_step_us(st, K, flush, stream):
    """Median step time with CUDA events recorded around every single step
    (an event between two steps keeps the next step from starting while the
    previous one drains)."""
    evs = []
    for _ in range(K):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        st.step()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3


def measure_config(args, rank, ws, config, window=None, extras=True):
    """One workload's record: the decode step timed K times (see time_steps),
    its roofline, SM clocks during the timed region and, unless disabled, the
    end-to-end number through host buffers."""
    dev = torch.device("cuda", torch.cuda.current_device())
    w = workload.make_workload(config, seed=args.seed)
    s = w.shape
    window = s.windows[0] if window is None else window
    lens = w.seq_lens.tolist()
    B = len(lens)
    dec_bytes = accounting.decode_bytes(lens, s.num_q_heads, s.num_kv_heads, s.head_dim, window)
    app_bytes = accounting.append_bytes(B, s.num_kv_heads, s.head_dim)
    step_bytes = dec_bytes + app_bytes
    cache_bytes = 2 * w.num_blocks * s.num_kv_heads * workload.BLOCK_SIZE * s.head_dim
    layers, flush = layer_plan(dec_bytes, cache_bytes, dev)
    st = DecodeStep(w, window, dev, layers=layers)
    stream = torch.cuda.current_stream()

    clocks = ClockSampler(torch.cuda.current_device()) if not args.no_clocks else None
    if clocks:
        clocks.start()
    for _ in range(max(args.warmup, st.layers)):
        st.step()
    torch.cuda.synchronize()
    assert st.fk.fp8kv_read_error(st.ws) == 0

    K = args.steps
    barrier(ws)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    total_ms, timing = time_steps(st, K, flush, stream)
    barrier(ws)
    t_wall1 = time.time()
    total_ms = reduce_max(total_ms, ws)
    clk = clocks.summary(t_wall0, t_wall1) if clocks else None
    iso_us = reduce_max(isolated_step_us(st, K, flush, stream), ws)
    assert st.fk.fp8kv_read_error(st.ws) == 0
    rec = {}
    if extras:
        # for reference: the unfused pair (decode call alone, append call alone)
        dec_ms, app_ms = [], []
        for i in range(K):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            st.decode()
            e1.record(stream)
            dec_ms.append((e0, e1))
            flush()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            st.append()
            a1.record(stream)
            app_ms.append((a0, a1))
        torch.cuda.synchronize()
        rec["paged_decode_us"] = round(reduce_max(statistics.fmean(a.elapsed_time(b) for a, b in dec_ms), ws) * 1e3, 3)
        rec["quant_append_us"] = round(statistics.fmean(a.elapsed_time(b) for a, b in app_ms) * 1e3, 3)
        # the two contraction engines of the decode call, each call timed alone
        eng_us = {}
        for name, eng in (("tensor_cores", st.fk.ENGINE_TENSOR_CORES), ("cuda_cores", st.fk.ENGINE_CUDA_CORES)):
            for _ in range(3):
                st.decode_engine(eng)
            evs = []
            for i in range(K):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                st.decode_engine(eng)
                e1.record(stream)
                evs.append((e0, e1))
            torch.cuda.synchronize()
            assert st.fk.fp8kv_read_error(st.ws) == 0
            eng_us[name + "_us"] = round(reduce_max(statistics.fmean(a.elapsed_time(b) for a, b in evs), ws) * 1e3, 3)
        rec["paged_decode_engines"] = eng_us
    if clocks:
        clocks.stop()

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(st, args, ws, step_bytes, flush)

    ms_per_step = total_ms / K
    peak, peak_src = measured_peaks()
    # roofline of the step call itself (decode kernel with the fused append,
    # then the split merge), timed inside the timed region above
    achieved = step_bytes / (ms_per_step * 1e-3) / 1e9
    key = "decode_step/%s/w%d" % (config, window)
    traffic = traffic_for(key)
    out = {
        "value": round(ws * achieved, 2), "unit": "GB/s", "ms_per_step": round(ms_per_step, 6),
        "us_per_step": round(ms_per_step * 1e3, 3), "us_per_step_isolated": round(iso_us, 3),
        "timing": timing,
        "config": {"workload": config, "batch": B, "num_q_heads": s.num_q_heads,
                   "num_kv_heads": s.num_kv_heads, "head_dim": s.head_dim, "block_size": 16,
                   "seq_lens": "uniform %d..%d" % (s.len_lo, s.len_hi), "total_tokens": int(sum(lens)),
                   "window": window, "kv_cache": "e4m3, per-tensor k/v scales",
                   "step": "fp8kv_decode_step: append B new tokens + paged decode, one call",
                   "l2": describe_layers(layers, flush, dec_bytes, cache_bytes, dev),
                   "parallelism": "replicas" if ws > 1 else "1 gpu",
                   "input_sha256": w.digest()[:16]},
        "step_bytes": step_bytes,
        "roofline": {"kernel": "fp8kv_decode_step call: split-context decode kernel (per-warp cp.async "
                               "streaming, append fused in) + split-merge kernel",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": step_bytes},
        "gpu_launches": 2 * K,  # decode kernel + split-merge kernel per step
        "clocks": clk,
    }
    out.update(rec)
    if e2e is not None:
        out["e2e"] = e2e
    out["_w"] = (w, window, dec_bytes + app_bytes)
    del st
    torch.cuda.empty_cache()
    return out


def run_fp8kv(args, rank, ws):
    main = measure_config(args, rank, ws, args.config, args.window)
    w, window, step_bytes = main.pop("_w")
    line = {"metric": METRIC, "value": main.pop("value"), "unit": main.pop("unit"), "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup}
    line.update(main)
    line.update({"higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                 "data": "synthetic (seeded N(0,1) bf16, per-tensor amax/448 E4M3 scales, shuffled 16-token pages)"})
    if args.config == "llama31_8b_b8_20k" and args.window is None and not args.no_per_config:
        line["per_config"] = {}
        for cfg in PER_CONFIG:
            rec = measure_config(args, rank, ws, cfg, None, extras=False)
            rec.pop("_w")
            line["per_config"][cfg] = rec
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, window, step_bytes)
    return line


def measure_e2e(st, args, ws, step_bytes, flush):
    """The same step through the C ABI from host buffers: fp8kv_decode_step_host
    copies the step's packed inputs (q, the new K/V rows, the sequence
    lengths) from pinned host memory to the device and runs the step, whose
    kernels write out directly into the pinned host output buffer (the device
    addresses it under unified addressing); the host then waits for the
    stream.  Each step is timed with the host clock, from the launch to the
    end of the wait.

    Two launch paths: the C call itself every step ("direct"), and the same
    call captured once into a CUDA graph that is replayed every step, as a
    decode loop issues a fixed step ("graph").  The copies and kernels are
    the same; the graph saves the per-call host work and launch gaps."""
    h_in = st.h_inputs.pin_memory()
    h_out = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
    st.step()   # the device step's output, which every host-staged step must reproduce
    torch.cuda.synchronize()
    ref_out = st.out.cpu()
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_out.numel() * h_out.element_size()
    w = st.w
    side = torch.cuda.Stream()

    def prepared(stream, layer):
        kc, vc = st.caches[layer]
        return st.fk.prepare_decode_step_host(h_in, st.inputs, h_out, st.q, st.k_new, st.v_new, kc, vc,
                                              st.block_tables, st.seq_lens, w.max_seq_len, w.k_scale,
                                              w.v_scale, w.sm_scale, st.window, st.out, st.ws, stream=stream)

    n = st.layers
    calls = [prepared(side, i) for i in range(n)]
    for i in range(max(args.warmup, n)):
        calls[i % n]()
        side.synchronize()
    graphs = []
    for i in range(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            prepared(side, i)()
        graphs.append(g)
    torch.cuda.synchronize()
    nxt = [0]

    def direct():
        calls[nxt[0]]()
        nxt[0] = (nxt[0] + 1) % n

    def run_graph():
        graphs[nxt[0]].replay()
        nxt[0] = (nxt[0] + 1) % n

    def timed(one, stream):
        for _ in range(max(args.warmup, n)):
            one()
            stream.synchronize()
        times = []
        barrier(ws)
        for _ in range(args.steps):
            flush()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            one()
            stream.synchronize()
            times.append(time.perf_counter() - t0)
        barrier(ws)
        return times

    t_direct = timed(direct, side)
    assert torch.equal(h_out, ref_out)
    h_out.zero_()
    t_graph = timed(run_graph, torch.cuda.current_stream())
    assert torch.equal(h_out, ref_out)
    mean_g = reduce_max(statistics.fmean(t_graph), ws)
    mean_d = reduce_max(statistics.fmean(t_direct), ws)
    return {"value": round(ws * step_bytes / mean_g / 1e9, 2), "unit": "GB/s",
            "us_per_step": round(mean_g * 1e6, 3), "us_per_step_median": round(statistics.median(t_graph) * 1e6, 3),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "call": "fp8kv_decode_step_host (one H2D copy of the packed inputs, the step; its kernels store out "
                    "straight into the pinned host buffer across NVLink-C2C), captured once per layer cache in a "
                    "CUDA graph and replayed every step",
            "direct_call": {"value": round(ws * step_bytes / mean_d / 1e9, 2), "unit": "GB/s",
                            "us_per_step": round(mean_d * 1e6, 3),
                            "us_per_step_median": round(statistics.median(t_direct) * 1e6, 3),
                            "call": "fp8kv_decode_step_host called every step"},
            "timer": "host wall clock per step: the launch through the stream synchronisation"}


# ---------------------------------------------------------------- the CPU oracle

def oracle_sample_step(w, window, kc, vc, seqs, nthreads):
    """One decode step of the oracle restricted to sequences `seqs`: quantise
    their newest K/V row, then fp64 attention over their caches."""
    import oracle
    rows = w.new_token_rows()[seqs]
    oracle.quantize_bf16(workload.bf16_bits(w.k[rows]), w.k_scale)
    oracle.quantize_bf16(workload.bf16_bits(w.v[rows]), w.v_scale)
    lens = w.seq_lens.numpy()[seqs]
    starts = w.seq_starts.numpy()[seqs]
    idx = np.concatenate([np.arange(s, s + L) for s, L in zip(starts, lens)])
    return oracle.decode_attention(workload.bf16_bits(w.q[seqs]), kc[idx], vc[idx], lens,
                                   w.k_scale, w.v_scale, w.sm_scale, window, nthreads=nthreads)


def oracle_codes(w):
    import oracle
    return (oracle.quantize_bf16(workload.bf16_bits(w.k), w.k_scale),
            oracle.quantize_bf16(workload.bf16_bits(w.v), w.v_scale))


def cpu_baseline(w, window, step_bytes_full):
    import oracle
    kc, vc = oracle_codes(w)
    n = oracle.max_threads()
    B = w.q.shape[0]
    seqs = np.arange(B)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle_sample_step(w, window, kc, vc, seqs, n)
        reps += 1
        el = time.perf_counter() - t0
        if el * n >= 10.0 or reps >= 3:
            break
    per = el / reps
    return {"value": round(step_bytes_full / per / 1e9, 4), "unit": "GB/s", "cores": n, "kind": "oracle",
            "us_per_step": round(per * 1e6, 1),
            "sample": "%d full decode step(s) of %s (all %d sequences): E4M3 quantisation of the new rows + "
                      "fp64 two-pass attention, OpenMP over (sequence, head)" % (reps, w.shape.name, B)}


def run_reference(args, rank, ws):
    import oracle
    w = workload.make_workload(args.config, seed=args.seed)
    s = w.shape
    window = s.windows[0] if args.window is None else args.window
    lens = w.seq_lens.numpy()
    kc, vc = oracle_codes(w)
    n = oracle.max_threads()
    B = len(lens)
    times, nbytes = [], []
    for i in range(args.warmup + args.steps):
        seqs = np.array([i % B])
        t0 = time.perf_counter()
        oracle_sample_step(w, window, kc, vc, seqs, n)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            nbytes.append(accounting.decode_bytes(lens[seqs], s.num_q_heads, s.num_kv_heads, s.head_dim, window)
                          + accounting.append_bytes(1, s.num_kv_heads, s.head_dim))
    tot = sum(times)
    value = sum(nbytes) / tot / 1e9
    sample = ("one sequence of %s per step (cycling through the %d sequences): E4M3 quantisation of its new "
              "row + fp64 attention over its cache" % (args.config, B))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": args.config, "window": window, "batch": B},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": n, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------- context sweep

SWEEP_LENS = (1024, 2048, 4096, 8192, 16384, 32768, 65536, 131072)
# one attention layer, batch 1: (name, q heads, kv heads, head_dim)
SWEEP_LAYOUTS = {"llama": ("llama31_8b_layer_b1", 32, 8, 128), "gemma": ("gemma4e2b_layer_b1", 8, 1, 256)}


def _fit(xs, ys):
    """Least-squares line y = slope * x + intercept."""
    A = np.stack([np.asarray(xs, dtype=np.float64), np.ones(len(xs))], axis=1)
    (slope, icpt), *_ = np.linalg.lstsq(A, np.asarray(ys, dtype=np.float64), rcond=None)
    return float(slope), float(icpt)


def run_sweep(args, rank, ws):
    """Decode time of one attention layer at batch 1 against context length,
    for the fp8 cache (fp8kv_paged_decode) and the bf16 cache
    (fp8kv_paged_decode_bf16): the per-token cost of each and their ratio,
    the GB300 counterpart of the fitted ITL slopes the pages compare.  Layouts
    (--sweep-layout): Llama-3.1-8B (32 q / 8 kv heads, d = 128) and
    gemma-4-E2B-like (8 q / 1 kv head, d = 256)."""
    from fp8_kv_cache_fp8kv_gb300 import binding as fk
    fk.load(build_if_missing=True)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    points = []
    for L in SWEEP_LENS:
        name, hq, hkv, hd = SWEEP_LAYOUTS[args.sweep_layout]
        shape = workload.LayerShape(name, hq, hkv, hd, 1, L, L, (0,))
        w = workload.make_workload(shape, seed=args.seed, lens=[L])
        s = w.shape
        cshape = (w.num_blocks, s.num_kv_heads, workload.BLOCK_SIZE, s.head_dim)
        sm = w.slot_mapping.to(dev)
        blk, off = sm // workload.BLOCK_SIZE, sm % workload.BLOCK_SIZE
        k8 = torch.zeros(cshape, dtype=torch.uint8, device=dev)
        v8 = torch.zeros_like(k8)
        fk.fp8kv_quant_append(w.k.to(dev), w.v.to(dev), sm, k8, v8, w.k_scale, w.v_scale)
        k5 = torch.zeros(cshape, dtype=torch.uint8, device=dev)
        v5 = torch.zeros_like(k5)
        ks5 = float(np.float32(w.k.float().abs().max() / 57344.0))
        vs5 = float(np.float32(w.v.float().abs().max() / 57344.0))
        fk.fp8kv_quant_append_e5m2(w.k.to(dev), w.v.to(dev), sm, k5, v5, ks5, vs5)
        kb = torch.zeros(cshape, dtype=torch.bfloat16, device=dev)
        vb = torch.zeros_like(kb)
        kb[blk, :, off, :] = w.k.to(dev)
        vb[blk, :, off, :] = w.v.to(dev)
        q = w.q.to(dev)
        bt = w.block_tables.to(dev)
        lens = w.seq_lens.to(dev)
        out = torch.empty_like(q)
        wsp = fk.alloc_workspace(1, s.num_q_heads, s.num_kv_heads, s.head_dim, L, 16, 0, device=dev)
        calls = {
            "fp8": fk.prepare_paged_decode(q, k8, v8, bt, lens, L, w.k_scale, w.v_scale, w.sm_scale, 0, out, wsp),
            "bf16": fk.prepare_paged_decode_bf16(q, kb, vb, bt, lens, L, w.sm_scale, 0, out, wsp),
            "e5m2": fk.PreparedCall("fp8kv_paged_decode_e5m2", fk.load().fp8kv_paged_decode_e5m2,
                                    fk.prepare_paged_decode(q, k5, v5, bt, lens, L, ks5, vs5, w.sm_scale, 0, out,
                                                            wsp).args),
        }
        read = {"fp8": accounting.decode_bytes([L], hq, hkv, hd, 0),
                "e5m2": accounting.decode_bytes([L], hq, hkv, hd, 0),
                "bf16": 2 * accounting.decode_bytes([L], hq, hkv, hd, 0)}
        rec = {"context": L}
        for name, call in calls.items():
            flush = L2Policy(read[name], dev)
            for _ in range(args.warmup):
                call()
            torch.cuda.synchronize()
            evs = []
            for _ in range(args.steps):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call()
                e1.record(stream)
                evs.append((e0, e1))
            torch.cuda.synchronize()
            assert fk.fp8kv_read_error(wsp) == 0
            us = reduce_max(statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3, ws)
            rec[name + "_us"] = round(us, 3)
            rec[name + "_l2"] = "flushed" if flush.buf is not None else "larger than L2"
        points.append(rec)
        del k8, v8, k5, v5, kb, vb
        torch.cuda.empty_cache()
    fit = {}
    for name in ("fp8", "e5m2", "bf16"):
        slope, icpt = _fit([p["context"] for p in points], [p[name + "_us"] for p in points])
        fit[name] = {"us_per_1k_tokens": round(slope * 1e3, 5), "intercept_us": round(icpt, 3)}
    ratio = fit["fp8"]["us_per_1k_tokens"] / fit["bf16"]["us_per_1k_tokens"]
    d_icpt = fit["fp8"]["intercept_us"] - fit["bf16"]["intercept_us"]
    d_slope = (fit["bf16"]["us_per_1k_tokens"] - fit["fp8"]["us_per_1k_tokens"]) / 1e3
    breakeven = round(d_icpt / d_slope) if d_icpt > 0 and d_slope > 0 else None  # None: fp8 never slower
    return {"sweep": "paged decode time against context length: E4M3 ('fp8') and E5M2 caches vs the bf16 cache",
            "config": {"workload": SWEEP_LAYOUTS[args.sweep_layout][0], "num_q_heads": SWEEP_LAYOUTS[args.sweep_layout][1],
                       "num_kv_heads": SWEEP_LAYOUTS[args.sweep_layout][2], "head_dim": SWEEP_LAYOUTS[args.sweep_layout][3],
                       "batch": 1, "block_size": 16, "window": 0, "timer": "CUDA events per call, median of %d"
                       % args.steps},
            "points": points, "fit": fit, "slope_ratio_fp8_over_bf16": round(ratio, 4),
            "slope_ratio_e5m2_over_bf16": round(fit["e5m2"]["us_per_1k_tokens"] / fit["bf16"]["us_per_1k_tokens"], 4),
            "breakeven_context_tokens": breakeven, "n_gpus": ws}


# ---------------------------------------------------------------- chunked prefill

def run_prefill(args, rank, ws):
    """fp8kv_paged_prefill on the workload's sequences with the last CHUNK
    tokens of each as the query chunk (causal over the whole cached prefix,
    the workload's window).  Algorithmic work: 4 * head_dim flops per (query
    row, query head, attended key) -- the score and the P.V products -- and
    the distinct cache pages the chunk attends plus q and out in bytes."""
    from fp8_kv_cache_fp8kv_gb300 import binding as fk
    fk.load(build_if_missing=True)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    window = workload.CONFIGS[args.config].windows[0] if args.window is None else args.window
    w = workload.make_workload(args.config, seed=args.seed)
    s = w.shape
    cshape = (w.num_blocks, s.num_kv_heads, workload.BLOCK_SIZE, s.head_dim)
    k8 = torch.zeros(cshape, dtype=torch.uint8, device=dev)
    v8 = torch.zeros_like(k8)
    fk.fp8kv_quant_append(w.k.to(dev), w.v.to(dev), w.slot_mapping.to(dev), k8, v8, w.k_scale, w.v_scale)
    bt = w.block_tables.to(dev)
    lens = w.seq_lens.to(dev)
    L = w.seq_lens.to(torch.int64).numpy()
    tflops_peak, peak_src = measured_tensor_peak()
    points = []
    for chunk in [int(c) for c in args.prefill.split(",")]:
        q_lens = np.minimum(L, chunk)
        q, qs = workload.prefill_queries(w, q_lens, seed=args.seed)
        q = q.to(dev)
        qs_d = qs.to(dev)
        out = torch.empty_like(q)
        wsp = fk.alloc_prefill_workspace(int(L.size), int(q_lens.max()), w.max_seq_len, s.num_q_heads,
                                         s.num_kv_heads, s.head_dim, 16, window, device=dev)
        call = fk.prepare_paged_prefill(q, k8, v8, bt, lens, qs_d, int(q_lens.max()), w.max_seq_len, w.k_scale,
                                        w.v_scale, w.sm_scale, window, out, wsp)
        pairs = 0
        pages = 0
        for Lb, n in zip(L.tolist(), q_lens.tolist()):
            pos = np.arange(Lb - n, Lb, dtype=np.int64)
            lo = np.maximum(0, pos + 1 - window) if window > 0 else np.zeros_like(pos)
            pairs += int((pos + 1 - lo).sum())
            if n:
                pages += int(pos[-1] // 16 - lo[0] // 16 + 1)
        flops = 4.0 * s.head_dim * s.num_q_heads * pairs
        nbytes = 2 * pages * s.num_kv_heads * 16 * s.head_dim + 2 * 2 * q.numel()
        flush = L2Policy(nbytes, dev)
        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize()
        clocks = ClockSampler(torch.cuda.current_device()) if not args.no_clocks else None
        if clocks:
            clocks.start()
        t_wall0 = time.time()
        evs = []
        for _ in range(args.steps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        t_wall1 = time.time()
        clk = clocks.summary(t_wall0, t_wall1) if clocks else None
        if clocks:
            clocks.stop()
        assert fk.fp8kv_read_error(wsp) == 0
        us = reduce_max(statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3, ws)
        points.append({"chunk": chunk, "workspace_bytes": int(wsp.numel()), "query_rows": int(q_lens.sum()), "us": round(us, 2),
                       "tflops": round(flops / us / 1e6, 2), "frac_of_tensor_peak": round(flops / us / 1e6 / tflops_peak, 4),
                       "gbs": round(nbytes / us / 1e3, 1), "flops": flops, "bytes": nbytes, "l2": flush.describe(),
                       "clocks": clk})
        del q, out, wsp
    return {"prefill": "fp8kv_paged_prefill: chunked prefill over the E4M3 cache",
            "config": {"workload": args.config, "window": window, "batch": int(L.size),
                       "timer": "CUDA events per call, median of %d" % args.steps},
            "tensor_peak_tflops": tflops_peak, "tensor_peak_source": peak_src, "points": points, "n_gpus": ws}


def run_copy_probe(args, rank, ws):
    """Builds csrc/probe/copy_probe.cu with nvcc and runs it: the 8x20K step's
    2 KB pages streamed into shared memory by TMA boxes from 2, 4 or 8
    producer warps per CTA, by per-warp cp.async rings, and by plain loads."""
    import re
    src = os.path.join(ROOT, "fp8_kv_cache_fp8kv_gb300", "csrc", "probe", "copy_probe.cu")
    exe = os.path.join(ROOT, "fp8_kv_cache_fp8kv_gb300", "_build", "copy_probe")
    os.makedirs(os.path.dirname(exe), exist_ok=True)
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", src, "-o", exe],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True, check=True)
    rates = {}
    for line in r.stdout.splitlines():
        m = re.match(r"(.+?): ([0-9.]+) us ([0-9.]+) GB/s", line)
        if m:
            rates[m.group(1)] = {"us": float(m.group(2)), "gbs": float(m.group(3))}
    return {"copy_probe": "page streaming into shared memory, no attention math (8x20K step's pages)",
            "header": r.stdout.splitlines()[0], "rates": rates, "n_gpus": ws}


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        # the oracle runs on rank 0 alone (host cores); other ranks have no work
        # and join no process group
        rank = int(os.environ.get("RANK", "0"))
        ws = int(os.environ.get("WORLD_SIZE", "1"))
        if rank == 0:
            print(json.dumps(run_reference(args, rank, ws)), flush=True)
        return 0
    rank, ws = dist_setup(args)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl fp8kv")
    if args.sweep or args.prefill or args.copy_probe:
        line = (run_sweep(args, rank, ws) if args.sweep else
                run_prefill(args, rank, ws) if args.prefill else run_copy_probe(args, rank, ws))
        if rank == 0:
            print(json.dumps(line), flush=True)
        return 0
    line = run_fp8kv(args, rank, ws)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
