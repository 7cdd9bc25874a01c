#!/usr/bin/env python
"""Benchmark of the Q8_0 W8A16 decode matmul on GB300.

Workload (one step): the decode layer set -- one 16-layer module's matrices,
QKV 1536->4608, o_proj 1536->1536, gate+up 1536->8192, down 4096->1536, all
Q8_0 (quantized on the GPU from N(0, 0.02) binary32 weights), applied for
8 passes with M = 1 bf16 activation row; each pass gets fresh N(0, 1)
activations (one vector per input width).  Each pass is ONE q8_linear_batch
launch over its 64 matrices.  The metric is achieved GB/s of algorithmic
bytes (codes + scales + activations + outputs) per second.

Weights total 481 MB per pass, far larger than the 129 MB L2, so no L2 flush
is needed between steps.  Other workloads (vocab GEMV, tiny GEMV, M sweep,
quantizer) are reported under "rows" as context.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "Q8_0 W8A16 decode GEMV achieved HBM GB/s and % of GB300 peak, M=1..32"
WORKLOAD = ("decode layer set: 16 layers x 8 passes, M=1, Q8_0 weights "
            "K1536->N4608 (QKV), 1536->1536 (o_proj), 1536->8192 (gate+up), 4096->1536 (down)")
PROFILE_JSON = os.path.join(ROOT, "profiles", "traffic.json")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# workload arithmetic
# ---------------------------------------------------------------------------
def matmul_bytes(N, K, M, out_bytes=4):
    return N * K + N * (K // 32) * 2 + M * K * 2 + M * N * out_bytes


def layer_set_bytes(M=1):
    per_layer = sum(matmul_bytes(N, K, M) for (_, K, N) in synth.LAYER_MATRICES)
    return per_layer * synth.LAYERS * synth.PASSES, per_layer * synth.LAYERS


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def profile_traffic(kernel="gemv_kernel"):
    """Per-launch DRAM bytes of `kernel` from the committed ncu record
    (profiles/traffic.json), if it was taken on the current kernel sources;
    else None.  Returns (bytes or None, the sources' sha256)."""
    try:
        rec = json.load(open(PROFILE_JSON))[kernel]
    except (OSError, ValueError, KeyError):
        return None, None
    h = hashlib.sha256()
    for p in rec.get("sources", []):
        try:
            h.update(open(os.path.join(ROOT, p), "rb").read())
        except OSError:
            return None, None
    if rec.get("source_sha256") != h.hexdigest():
        return None, h.hexdigest()
    try:
        return int(rec["traffic_bytes_per_launch"]), h.hexdigest()
    except (KeyError, ValueError, TypeError):
        return None, h.hexdigest()


def gpu_temperature(index):
    """GPU temperature (deg C) read with an nvidia-smi query, or None."""
    try:
        out = subprocess.run(["nvidia-smi", f"--id={index}", "--query-gpu=temperature.gpu",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=20)
        return float(out.stdout.strip().splitlines()[0])
    except Exception:
        return None


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or the machine type."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def spread(vals):
    """Median, 10th and 90th percentile of a list (linear interpolation)."""
    a = np.asarray(vals, dtype=np.float64)
    return float(np.median(a)), float(np.percentile(a, 10)), float(np.percentile(a, 90))


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="q8clk", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1])]
        smax = [num(r[2]) for r in rows if num(r[2])]
        pw = [num(r[3]) for r in rows if num(r[3])]
        # "under load": samples drawing more than the midpoint of idle and peak power
        if pw:
            cut = (min(pw) + max(pw)) / 2
            load = [num(r[1]) for r in rows if num(r[3]) and num(r[3]) >= cut and num(r[1])]
        else:
            load = sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(load or sm) if (load or sm) else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
class LayerSet:
    """Device-resident decode layer set and per-pass q8_linear_batch descriptors."""

    def __init__(self, torch, q8, seed=0):
        self.torch = torch
        self.q8 = q8
        dev = torch.device("cuda")
        self.w = []   # per layer: {name: (q, s)}
        for layer in range(synth.LAYERS):
            mats = {}
            for (name, K, N) in synth.LAYER_MATRICES:
                wf = torch.from_numpy(synth.weights(N, K, seed, synth.layer_weight_tag(layer, name))).to(dev)
                mats[name] = q8.q8_quantize_rows(wf)
                del wf
            self.w.append(mats)
        torch.cuda.synchronize()
        self.widths = sorted({K for (_, K, _) in synth.LAYER_MATRICES})
        # activations: one vector per (pass, input width); bf16 bits
        self.x_host = {(p, K): synth.activations(1, K, seed, synth.layer_x_tag(p, K))
                       for p in range(synth.PASSES) for K in self.widths}
        # all activations in one device buffer and all outputs in another, so an
        # end-to-end step moves them with one copy each way
        self.x_keys = sorted(self.x_host)
        x_elems = sum(self.x_host[k].size for k in self.x_keys)
        self.x_all = torch.empty(x_elems, dtype=torch.bfloat16, device=dev)
        self.x = {}
        off = 0
        for key in self.x_keys:
            v = self.x_host[key]
            self.x[key] = self.x_all[off:off + v.size].view(1, -1)
            self.x[key].view(torch.int16).copy_(torch.from_numpy(v.view(np.int16)).view(1, -1))
            off += v.size
        n_out = sum(N for (_, _, N) in synth.LAYER_MATRICES) * synth.LAYERS * synth.PASSES
        self.y_all = torch.empty(n_out, dtype=torch.float32, device=dev)
        self.y = []
        off = 0
        for _ in range(synth.PASSES):
            per_pass = []
            for _ in range(synth.LAYERS):
                per_layer = {}
                for (name, K, N) in synth.LAYER_MATRICES:
                    per_layer[name] = self.y_all[off:off + N].view(1, N)
                    off += N
                per_pass.append(per_layer)
            self.y.append(per_pass)
        self.descs = []
        ws_need = 0
        for p in range(synth.PASSES):
            mats = []
            for layer in range(synth.LAYERS):
                for (name, K, N) in synth.LAYER_MATRICES:
                    q, s = self.w[layer][name]
                    mats.append((q, s, self.x[(p, K)], self.y[p][layer][name]))
            d, M = q8.make_descs(mats)
            self.descs.append(d)
            ws_need = max(ws_need, q8.q8_linear_batch_workspace_size(d, 1))
        self.ws = q8.workspace(ws_need, dev)
        self.launches_per_step = synth.PASSES

    def step(self, variant=0, stream=None, chained=False):
        for p in range(synth.PASSES):
            self.q8.q8_linear_batch(descs=self.descs[p], M=1, ws=self.ws, variant=variant, stream=stream,
                                    chained=chained)

    def check_sample(self, oracle_mod=None):
        """Cheap consistency check of pass 0 against the oracle on a few rows."""
        return True


def max_over_ranks(torch, dist, seconds, device):
    """The slowest rank's time (every rank gets it); seconds alone without a
    process group."""
    if dist is None:
        return seconds
    t = torch.tensor([seconds], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step, steps, t_max, world):
    """Whole-job throughput: every rank moved bytes_per_step per step; the job
    took the slowest rank's time."""
    return world * bytes_per_step * steps / t_max / 1e9


def ceilings(torch, q8, nbytes=2 << 30, reps=5):
    """The two references of the "Frigg" README's "The machine": a device-to-
    device copy (cudaMemcpyAsync; read + write bytes) and a streaming read
    (q8_stream_read), GB/s, measured in this run."""
    src = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    src.fill_(1)
    words = q8.lib().q8_stream_read_out_words()
    out = torch.zeros(max(int(words), 1), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def t_of(fn):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / reps

    t_copy = t_of(lambda: dst.copy_(src))
    t_read = t_of(lambda: q8.lib().q8_stream_read(src.data_ptr(), nbytes, out.data_ptr(),
                                                  ctypes.c_void_p(stream.cuda_stream)))
    del src, dst
    return 2 * nbytes / t_copy / 1e9, nbytes / t_read / 1e9


def time_steps(torch, fn, steps, warmup):
    """Seconds for `steps` calls of fn, one CUDA event pair on the launching
    stream around all of them (after `warmup` untimed calls)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


def time_blocks(torch, fn, steps, nblocks=20):
    """Times `steps` calls of fn as min(nblocks, steps) consecutive blocks of
    (nearly) equal size, with a CUDA event on the launching stream between
    blocks.  Returns (seconds from the first event to the last, list of
    seconds per step of each block)."""
    nb = max(1, min(nblocks, steps))
    sizes = [steps // nb + (1 if i < steps % nb else 0) for i in range(nb)]
    stream = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(nb + 1)]
    torch.cuda.synchronize()
    evs[0].record(stream)
    for i, n in enumerate(sizes):
        for _ in range(n):
            fn()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per_step = [evs[i].elapsed_time(evs[i + 1]) / 1e3 / sizes[i] for i in range(nb)]
    return evs[0].elapsed_time(evs[-1]) / 1e3, per_step


def per_launch_ms(torch, ls, reps, variant=0):
    """Average duration of one q8_linear_batch launch (one pass), CUDA events
    recorded on the launching stream around each launch."""
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps * synth.PASSES)]
    torch.cuda.synchronize()
    i = 0
    for _ in range(reps):
        for p in range(synth.PASSES):
            evs[i][0].record(stream)
            ls.q8.q8_linear_batch(descs=ls.descs[p], M=1, ws=ls.ws, variant=variant)
            evs[i][1].record(stream)
            i += 1
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs)


def e2e_gbs(torch, ls, steps, bytes_per_step, chained=False):
    """Whole step through the public API with host buffers, timed by the host
    clock: every step copies all passes' activations from pinned host memory
    (one H2D copy), runs the 8 batch launches, copies each pass's outputs to
    pinned host memory (on a second stream, as soon as that pass is done, so
    it overlaps the next pass) and the host reads the step's result.  Two
    host output buffers alternate, so step i + 1 is queued before the host
    waits for step i's result (the GPU does not idle while the host reads);
    the loop ends only after the last step's result has been read.  The
    device outputs alternate as well (a second set of descriptors), so a
    step's kernels never overwrite outputs still being copied out."""
    xh = torch.from_numpy(np.concatenate([ls.x_host[k].reshape(-1) for k in ls.x_keys]).view(np.int16)).pin_memory()
    yh = [torch.empty(ls.y_all.shape, dtype=ls.y_all.dtype, pin_memory=True) for _ in range(2)]
    y_dev = [ls.y_all, torch.empty_like(ls.y_all)]
    delta = y_dev[1].data_ptr() - y_dev[0].data_ptr()

    def shifted(d):
        arr = (ls.q8.LinearDesc * len(d))()
        for k in range(len(d)):
            arr[k] = ls.q8.LinearDesc(d[k].q, d[k].s, d[k].x, d[k].y + delta, d[k].N, d[k].K, d[k].ldx, d[k].ldy)
        return arr
    descs = [ls.descs, [shifted(d) for d in ls.descs]]
    h2d = xh.numel() * 2
    d2h = yh[0].numel() * 4
    per_pass = ls.y_all.numel() // synth.PASSES
    copy_stream = torch.cuda.Stream()
    done = [torch.cuda.Event() for _ in range(synth.PASSES)]
    step_done = [torch.cuda.Event() for _ in range(2)]
    checksum = [0.0]

    def issue(i):
        cs = torch.cuda.current_stream()
        out, ydev, dsc = yh[i % 2], y_dev[i % 2], descs[i % 2]
        ls.x_all.view(torch.int16).copy_(xh, non_blocking=True)
        for p in range(synth.PASSES):
            ls.q8.q8_linear_batch(descs=dsc[p], M=1, ws=ls.ws, chained=chained)
            done[p].record(cs)
            copy_stream.wait_event(done[p])
            with torch.cuda.stream(copy_stream):
                out[p * per_pass:(p + 1) * per_pass].copy_(ydev[p * per_pass:(p + 1) * per_pass], non_blocking=True)
        step_done[i % 2].record(copy_stream)

    def read(i):
        step_done[i % 2].synchronize()
        checksum[0] += float(yh[i % 2][0])  # the host touches the result

    def run(n):
        issue(0)
        for i in range(1, n):
            issue(i)
            read(i - 1)
        read(n - 1)

    run(3)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(steps)
    dt = time.perf_counter() - t0
    torch.cuda.synchronize()
    return bytes_per_step * steps / dt / 1e9, h2d, d2h


def chain_rows(torch, q8, ls, peak, ms=(1, 8)):
    """The dependent decode chain of a token over the two modules in their
    order L L L H L L L H: each of its 512 matmuls takes its input from the
    one before it (q8_linear_chain: RMS normalisation, SwiGLU then RMS
    normalisation between gate+up and down), the whole token one CUDA graph
    of programmatic dependent launches.  L is the layer set's module, H a
    second module of the same shapes (its own weights).  The same weight
    bytes per token as one layer-set step (eight passes over a module)."""
    dev = torch.device("cuda")
    h = []
    for layer in range(synth.LAYERS):
        mats = {}
        for (name, K, N) in synth.LAYER_MATRICES:
            wf = torch.from_numpy(synth.weights(N, K, 1, synth.layer_weight_tag(layer, name))).to(dev)
            mats[name] = q8.q8_quantize_rows(wf)
            del wf
        h.append(mats)
    nxt = {"qkv": q8.Q8_CHAIN_RMSNORM, "o_proj": q8.Q8_CHAIN_RMSNORM,
           "gate_up": q8.Q8_CHAIN_SWIGLU_RMSNORM, "down": q8.Q8_CHAIN_RMSNORM}
    rows = {}
    for M in ms:
        steps = []
        for module in "LLLHLLLH":
            w = ls.w if module == "L" else h
            for layer in range(synth.LAYERS):
                for (name, K, N) in synth.LAYER_MATRICES:
                    q, sc = w[layer][name]
                    if not steps:
                        x = torch.from_numpy(synth.activations(M, K, 0, "chain.x0").view(np.int16)).view(
                            torch.bfloat16).to(dev)
                    else:
                        x = torch.zeros((M, K), dtype=torch.bfloat16, device=dev)
                    y = torch.empty((M, N), dtype=torch.float32, device=dev)
                    steps.append([q, sc, x, y, nxt[name]])
        steps[-1][4] = q8.Q8_CHAIN_END
        arr, _ = q8.make_chain([tuple(t) for t in steps])
        ws = q8.workspace(q8.q8_linear_chain_workspace_size(arr, M), dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        s_ = torch.cuda.Stream()
        with torch.cuda.stream(s_):
            q8.q8_linear_chain(arr, M, ws=ws, dev_status=st, stream=s_)
        s_.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s_):
            q8.q8_linear_chain(arr, M, ws=ws, dev_status=st, stream=s_)
        reps = 20
        dtg = time_steps(torch, g.replay, reps, 3)
        if int(st.item()) != 0:
            raise RuntimeError(f"decode chain M={M}: device status {int(st.item())}")
        t = dtg / reps
        nbytes = layer_set_bytes(M)[0]
        rows[f"decode_chain_LLLH_M{M}"] = {
            "GB/s": round(nbytes / t / 1e9, 1), "frac": round(nbytes / t / 1e9 / peak, 3),
            "us_per_token": round(t * 1e6, 1), "tok_s": round(M / t, 1),
            "launches_per_token": 2 * len(steps) - 1, "matmuls_per_token": len(steps)}
        del g, arr, ws, steps
    del h
    torch.cuda.empty_cache()
    return rows


def extra_rows(torch, q8, peak):
    """Context rows: other workloads, each timed with CUDA events on distinct
    weight copies so that no call finds its weights in L2."""
    dev = torch.device("cuda")
    rows = {}
    L2 = 129 * 2**20

    def timed(fn_list, reps=20):
        """Seconds per call: the calls are captured once into a CUDA graph (so
        host launch overhead is not measured) and the graph is replayed
        `reps` times, each replay between its own pair of CUDA events.
        Returns the median replay's time per call; the 10th and 90th
        percentiles go to spread_of[0]."""
        for f in fn_list:
            f()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for f in fn_list:
                f()
        g.replay()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for e0, e1 in evs:
            e0.record()
            g.replay()
            e1.record()
        torch.cuda.synchronize()
        del g
        med, p10, p90 = spread([a.elapsed_time(b) / 1e3 / len(fn_list) for a, b in evs])
        spread_of[0] = (p10, p90)
        return med

    spread_of = [(0.0, 0.0)]

    def row(nbytes, t, **extra):
        """A context row: GB/s of `nbytes` per call at the median time t,
        and the replays' 10th / 90th percentile times."""
        p10, p90 = spread_of[0]
        r = {"GB/s": round(nbytes / t / 1e9, 1), "frac": round(nbytes / t / 1e9 / peak, 3),
             "us": round(t * 1e6, 2), "us_p10": round(p10 * 1e6, 2), "us_p90": round(p90 * 1e6, 2)}
        r.update(extra)
        return r

    def copies_for(nbytes):
        return max(1, int(np.ceil(4 * L2 / nbytes)))

    # vocab GEMV, M = 1
    N, K = synth.VOCAB, synth.HIDDEN
    wq, ws_ = q8.q8_quantize_rows(torch.from_numpy(synth.weights(N, K, 0, "vocab")).to(dev))
    xv = torch.from_numpy(synth.unit_activation(K, 0).view(np.int16)).view(torch.bfloat16).to(dev)
    yv = torch.empty((1, N), dtype=torch.float32, device=dev)
    by = matmul_bytes(N, K, 1)
    for v, name in ((1, "simt"), (2, "mma")):
        t = timed([lambda v=v: q8.q8_linear_batch([(wq, ws_, xv, yv)], variant=v)])
        rows[f"vocab_gemv_M1_{name}"] = row(by, t)
    # the quantizer creating that matrix (bandwidth figure: 4 B in, 1.0625 B out per weight)
    wf = torch.from_numpy(synth.weights(N, K, 0, "vocab")).to(dev)
    qb, sb = torch.empty_like(wq), torch.empty_like(ws_)
    t = timed([lambda: q8.q8_quantize_rows(wf, qb, sb)])
    rows["quantize_262144x1536"] = row(N * K * 4 + N * K + N * K // 16, t)
    # GGUF Q8_0 ingest of that matrix (34 B in, 34 B out per block) and export
    raw = q8.q8_planar_to_gguf(wq, ws_)
    gbytes = 2 * raw.numel()
    t = timed([lambda: q8.q8_gguf_to_planar(raw, N, K, qb, sb)])
    rows["gguf_ingest_262144x1536"] = row(gbytes, t)
    t = timed([lambda: q8.q8_planar_to_gguf(wq, ws_, raw)])
    rows["gguf_export_262144x1536"] = row(gbytes, t)
    del raw
    wsmall = torch.from_numpy(synth.quant_stress_rows()).to(dev)
    t = timed([lambda: q8.q8_quantize_rows(wsmall)], reps=50)
    rows["quantize_32x4096"] = {"us": round(t * 1e6, 2), "us_p10": round(spread_of[0][0] * 1e6, 2),
                                "us_p90": round(spread_of[0][1] * 1e6, 2)}
    del wf, qb, sb, wq, ws_

    # tiny GEMV and the M sweep, rotating over distinct weight copies
    cases = [("tiny_gemv", 4096, 1536, [1])] + [(f"sweep_K{K}_N{N}", N, K, list(synth.SWEEP_M))
                                                for (K, N) in synth.SWEEP_SHAPES]
    for (name, N, K, Ms) in cases:
        q0, s0 = q8.q8_quantize_rows(torch.from_numpy(synth.weights(N, K, 0, name)).to(dev))
        ncp = copies_for(N * K * 1.0625)
        cps = [(q0.clone(), s0.clone()) for _ in range(ncp)]
        for M in Ms:
            x = torch.from_numpy(synth.activations(M, K, 0, f"{name}.x{M}").view(np.int16)).view(torch.bfloat16).to(dev)
            y = torch.empty((M, N), dtype=torch.float32, device=dev)
            by = matmul_bytes(N, K, M)
            for v, vn in ((1, "simt"), (2, "mma")):
                descs = []
                for (q, s) in cps:
                    d, _ = q8.make_descs([(q, s, x, y)])
                    descs.append(d)
                ws = q8.workspace(q8.q8_linear_batch_workspace_size(descs[0], M), dev)
                fns = [lambda d=d, v=v, M=M, ws=ws: q8.q8_linear_batch(descs=d, M=M, ws=ws, variant=v)
                       for d in descs]
                t = timed(fns)
                rows[f"{name}_M{M}_{vn}"] = row(by, t, **{"GMAC/s": round(M * N * K / t / 1e9, 1)})
            # the copies as separate calls (default kernels), plain and chained:
            # a decode step of one call per matrix, weights fixed
            descs = [q8.make_descs([(q, s, x, y)])[0] for (q, s) in cps]
            wsc = q8.workspace(q8.q8_linear_batch_workspace_size(descs[0], M), dev)
            for ch, cn in ((False, "calls"), (True, "chained_calls")):
                fns = [lambda d=d, M=M, ch=ch: q8.q8_linear_batch(descs=d, M=M, ws=wsc, chained=ch) for d in descs]
                t = timed(fns)
                rows[f"{name}_M{M}_{cn}"] = row(by, t)
            # steady state: the distinct copies as ONE batched launch (default kernels)
            nb_ = min(len(cps), q8.Q8_MAX_BATCH)
            ys = [torch.empty((M, N), dtype=torch.float32, device=dev) for _ in range(nb_)]
            bd, _ = q8.make_descs([(cps[i][0], cps[i][1], x, ys[i]) for i in range(nb_)])
            wsb = q8.workspace(q8.q8_linear_batch_workspace_size(bd, M), dev)
            t = timed([lambda bd=bd, M=M, wsb=wsb: q8.q8_linear_batch(descs=bd, M=M, ws=wsb)])
            bb = by * nb_
            rows[f"{name}_M{M}_batch{nb_}"] = row(bb, t, **{"GMAC/s": round(nb_ * M * N * K / t / 1e9, 1)})
            # the same batch with the batch-invariant arithmetic (rows independent of M)
            if K % 256 == 0:
                t = timed([lambda bd=bd, M=M: q8.q8_linear_batch(descs=bd, M=M,
                                                                 variant=q8.Q8_VARIANT_BATCH_INVARIANT)])
                rows[f"{name}_M{M}_batch{nb_}_invariant"] = row(bb, t)
                # and W8A8 (x quantized to Q8_0 per row, int8 block dots; same bytes counted)
                ws8 = q8.workspace(int(q8.lib().q8_linear_batch_workspace_size_ex(bd, len(bd), M,
                                                                                   q8.Q8_VARIANT_W8A8)), dev)
                t = timed([lambda bd=bd, M=M, ws8=ws8: q8.q8_linear_batch(descs=bd, M=M, ws=ws8,
                                                                          variant=q8.Q8_VARIANT_W8A8)])
                rows[f"{name}_M{M}_batch{nb_}_w8a8"] = row(bb, t)
                del ws8
            del ys, wsb
        del cps
    # a K that is not a multiple of 256 (K % 256 = 32): M = 1 goes to the
    # GEMV, M = 2..8 to the warp-MMA pipeline, larger M to the tile kernel
    # with a partial last chunk
    K, N = synth.ODD_K_SHAPE
    name = f"oddk_K{K}_N{N}"
    q0, s0 = q8.q8_quantize_rows(torch.from_numpy(synth.weights(N, K, 0, name)).to(dev))
    ncp = copies_for(N * K * 1.0625)
    cps = [(q0.clone(), s0.clone()) for _ in range(ncp)]
    for M in (1, 2, 8, 16, 32):
        x = torch.from_numpy(synth.activations(M, K, 0, f"{name}.x{M}").view(np.int16)).view(torch.bfloat16).to(dev)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        by = matmul_bytes(N, K, M)
        descs = [q8.make_descs([(q, s, x, y)])[0] for (q, s) in cps]
        wsc = q8.workspace(q8.q8_linear_batch_workspace_size(descs[0], M), dev)
        t = timed([lambda d=d, M=M: q8.q8_linear_batch(descs=d, M=M, ws=wsc) for d in descs])
        rows[f"{name}_M{M}_calls"] = row(by, t)
        nb_ = min(len(cps), q8.Q8_MAX_BATCH)
        ys = [torch.empty((M, N), dtype=torch.float32, device=dev) for _ in range(nb_)]
        bd, _ = q8.make_descs([(cps[i][0], cps[i][1], x, ys[i]) for i in range(nb_)])
        wsb = q8.workspace(q8.q8_linear_batch_workspace_size(bd, M), dev)
        t = timed([lambda bd=bd, M=M, wsb=wsb: q8.q8_linear_batch(descs=bd, M=M, ws=wsb)])
        rows[f"{name}_M{M}_batch{nb_}"] = row(by * nb_, t)
        del ys, wsb
    del cps

    # prefill-shaped GEMM on tcgen05 (compute-bound: report TFLOP/s)
    peaks, _ = measured_peaks()
    tpk = float(peaks.get("bf16_tflops", 1900.0))
    M = synth.PREFILL_M
    for (K, N) in synth.SWEEP_SHAPES:
        q0, s0 = q8.q8_quantize_rows(torch.from_numpy(synth.weights(N, K, 0, f"pf{K}.{N}")).to(dev))
        x = torch.from_numpy(synth.activations(M, K, 0, f"pfx{K}").view(np.int16)).view(torch.bfloat16).to(dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        t = timed([lambda q0=q0, s0=s0, x=x, y=y: q8.q8_gemm(q0, s0, x, y)], reps=50)
        tf = 2.0 * M * N * K / t / 1e12
        rows[f"prefill_gemm_M{M}_K{K}_N{N}"] = {
            "TFLOP/s": round(tf, 1), "frac": round(tf / tpk, 4), "us": round(t * 1e6, 2),
            "us_p10": round(spread_of[0][0] * 1e6, 2), "us_p90": round(spread_of[0][1] * 1e6, 2),
            "GB/s": round(matmul_bytes(N, K, M, 2) / t / 1e9, 1)}
        # the same shape as W8A8 (int8 warp MMA in 32-row slices; fp32 out):
        # int8 TOPS, and that rate against the measured bf16 peak
        y8 = torch.empty((M, N), dtype=torch.float32, device=dev)
        ws8 = q8.workspace(int(q8.lib().q8_gemm_w8a8_workspace_size(N, K, M)), dev)
        t = timed([lambda q0=q0, s0=s0, x=x, y8=y8, ws8=ws8: q8.q8_gemm_w8a8(q0, s0, x, y=y8, ws=ws8)], reps=20)
        tf = 2.0 * M * N * K / t / 1e12
        rows[f"prefill_w8a8_M{M}_K{K}_N{N}"] = {
            "TOPS": round(tf, 1), "frac_of_bf16_peak": round(tf / tpk, 4), "us": round(t * 1e6, 2),
            "us_p10": round(spread_of[0][0] * 1e6, 2), "us_p90": round(spread_of[0][1] * 1e6, 2)}
        del y8, ws8
    torch.cuda.empty_cache()
    return rows


# ---------------------------------------------------------------------------
# CPU oracle timing (reported baseline, and the reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(budget_s=12.0, threads=None):
    """Time the oracle on the decode layer set (weights already quantized, as on
    the GPU side), matrix by matrix and pass by pass, until about `budget_s`
    seconds of CPU work are spent, on `threads` host threads (all cores if
    None; the oracle splits output rows over threads with identical bits).
    Returns (GB/s of algorithmic bytes, threads, sample text)."""
    import oracle
    oracle.build()
    cores = threads or (os.cpu_count() or 1)
    done_bytes = 0
    spent = 0.0
    n_mats = 0
    mats = {}
    for p in range(synth.PASSES):
        xs = {K: synth.activations(1, K, 0, synth.layer_x_tag(p, K)) for K in (synth.HIDDEN, synth.INTER)}
        for layer in range(synth.LAYERS):
            for (name, K, N) in synth.LAYER_MATRICES:
                key = (layer, name)
                if key not in mats:
                    q, s, _ = oracle.quantize_rows(synth.weights(N, K, 0, synth.layer_weight_tag(layer, name)))
                    mats[key] = (q, s)
                q, s = mats[key]
                t0 = time.perf_counter()
                oracle.matmul(q, s, xs[K], threads=cores)
                spent += time.perf_counter() - t0
                done_bytes += matmul_bytes(N, K, 1)
                n_mats += 1
                if spent >= budget_s:
                    break
            if spent >= budget_s:
                break
        if spent >= budget_s:
            break
    return (done_bytes / spent / 1e9, cores,
            f"oracle (binary64 dequantise-then-dot) on the first {n_mats} of the layer set's "
            f"{synth.LAYERS * synth.PASSES * len(synth.LAYER_MATRICES)} matmuls (weights pre-quantized), "
            f"{spent:.1f} s on {cores} thread{'s' if cores > 1 else ''}")


def reference_arm(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    xs = {K: synth.activations(1, K, 0, synth.layer_x_tag(0, K)) for K in (synth.HIDDEN, synth.INTER)}
    # each step: every 64th row of one layer's four matrices (round-robin over layers)
    stride = 64
    mats = []
    for layer in range(synth.LAYERS):
        for (name, K, N) in synth.LAYER_MATRICES:
            w = synth.weights(N, K, 0, synth.layer_weight_tag(layer, name))[::stride]
            q, s, _ = oracle.quantize_rows(w)
            mats.append((layer, q, s, K))

    def step(i):
        layer = i % synth.LAYERS
        b = 0
        for (l, q, s, K) in mats:
            if l == layer:
                oracle.matmul(q, s, xs[K], threads=cores)
                b += matmul_bytes(q.shape[0], K, 1)
        return b

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    tot = 0
    for i in range(args.steps):
        tot += step(i)
    dt = time.perf_counter() - t0
    v = tot / dt / 1e9
    sample = (f"oracle (binary64) on every {stride}th row of one layer's 4 matrices per step, "
              f"layers round-robin; {cores} threads")
    line = {"metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / max(args.steps, 1) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "M": 1, "layers": synth.LAYERS, "passes": synth.PASSES},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def profile_case(torch, q8, args):
    """A handful of launches of one workload, nothing timed: the command that
    ncu captures (weights quantized first, then `--warmup` + 3 launches)."""
    if args.profile == "layerset":
        ls = LayerSet(torch, q8)
        for i in range(args.warmup + 3):
            q8.q8_linear_batch(descs=ls.descs[i % synth.PASSES], M=1, ws=ls.ws, variant=args.variant)
    elif args.profile == "sweep8":
        # M=8 over 16 distinct copies of the K1536 -> N8192 matrix in one launch
        K, N = synth.SWEEP_SHAPES[0]
        M = 8
        q0, s0 = q8.q8_quantize_rows(torch.from_numpy(synth.weights(N, K, 0, f"sweep_K{K}_N{N}")).cuda())
        x = torch.from_numpy(synth.activations(M, K, 0, "sweep8.x").view(np.int16)).view(torch.bfloat16).cuda()
        cps = [(q0.clone(), s0.clone()) for _ in range(16)]
        ys = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in cps]
        bd, _ = q8.make_descs([(c[0], c[1], x, y) for c, y in zip(cps, ys)])
        for _ in range(args.warmup + 3):
            q8.q8_linear_batch(descs=bd, M=M)
    elif args.profile == "tile16":
        # M=16 over 32 distinct copies of the K4096 -> N1536 matrix in one launch
        K, N = synth.SWEEP_SHAPES[1]
        M = 16
        q0, s0 = q8.q8_quantize_rows(torch.from_numpy(synth.weights(N, K, 0, f"sweep_K{K}_N{N}")).cuda())
        x = torch.from_numpy(synth.activations(M, K, 0, "tile16.x").view(np.int16)).view(torch.bfloat16).cuda()
        cps = [(q0.clone(), s0.clone()) for _ in range(32)]
        ys = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in cps]
        bd, _ = q8.make_descs([(c[0], c[1], x, y) for c, y in zip(cps, ys)])
        for _ in range(args.warmup + 3):
            q8.q8_linear_batch(descs=bd, M=M)
    elif args.profile == "tile32":
        # M=32 over 32 distinct copies of the K4096 -> N1536 matrix in one launch
        K, N = synth.SWEEP_SHAPES[1]
        M = 32
        q0, s0 = q8.q8_quantize_rows(torch.from_numpy(synth.weights(N, K, 0, f"sweep_K{K}_N{N}")).cuda())
        x = torch.from_numpy(synth.activations(M, K, 0, "tile32.x").view(np.int16)).view(torch.bfloat16).cuda()
        cps = [(q0.clone(), s0.clone()) for _ in range(32)]
        ys = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in cps]
        bd, _ = q8.make_descs([(c[0], c[1], x, y) for c, y in zip(cps, ys)])
        ws = q8.workspace(q8.q8_linear_batch_workspace_size(bd, M))
        for _ in range(args.warmup + 3):
            q8.q8_linear_batch(descs=bd, M=M, ws=ws)
    elif args.profile == "oddk16":
        # M=16 over 32 distinct copies of the K2080 -> N4608 matrix (K not a
        # multiple of 256) in one launch
        K, N = synth.ODD_K_SHAPE
        M = 16
        q0, s0 = q8.q8_quantize_rows(torch.from_numpy(synth.weights(N, K, 0, f"oddk_K{K}_N{N}")).cuda())
        x = torch.from_numpy(synth.activations(M, K, 0, "oddk16.x").view(np.int16)).view(torch.bfloat16).cuda()
        cps = [(q0.clone(), s0.clone()) for _ in range(32)]
        ys = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in cps]
        bd, _ = q8.make_descs([(c[0], c[1], x, y) for c, y in zip(cps, ys)])
        ws = q8.workspace(q8.q8_linear_batch_workspace_size(bd, M))
        for _ in range(args.warmup + 3):
            q8.q8_linear_batch(descs=bd, M=M, ws=ws)
    elif args.profile == "chain":
        # one module run (16 layers, 64 dependent matmuls, 127 launches) as
        # q8_linear_chain at M = 1, `--warmup` + 3 times
        ls = LayerSet(torch, q8)
        nxt = {"qkv": q8.Q8_CHAIN_RMSNORM, "o_proj": q8.Q8_CHAIN_RMSNORM,
               "gate_up": q8.Q8_CHAIN_SWIGLU_RMSNORM, "down": q8.Q8_CHAIN_RMSNORM}
        steps = []
        for layer in range(synth.LAYERS):
            for (name, K, N) in synth.LAYER_MATRICES:
                q, sc = ls.w[layer][name]
                x = ls.x[(0, K)] if not steps else torch.zeros((1, K), dtype=torch.bfloat16, device="cuda")
                steps.append([q, sc, x, torch.empty((1, N), dtype=torch.float32, device="cuda"), nxt[name]])
        steps[-1][4] = q8.Q8_CHAIN_END
        arr, _ = q8.make_chain([tuple(t) for t in steps])
        ws = q8.workspace(q8.q8_linear_chain_workspace_size(arr, 1))
        for _ in range(args.warmup + 3):
            q8.q8_linear_chain(arr, 1, ws=ws)
    elif args.profile == "w8a8":
        # the W8A8 GEMM at the prefill shape: M = 512, K1536 -> N8192
        K, N = synth.SWEEP_SHAPES[0]
        M = synth.PREFILL_M
        q0, s0 = q8.q8_quantize_rows(torch.from_numpy(synth.weights(N, K, 0, f"pf{K}.{N}")).cuda())
        x = torch.from_numpy(synth.activations(M, K, 0, f"pfx{K}").view(np.int16)).view(torch.bfloat16).cuda()
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        ws = q8.workspace(int(q8.lib().q8_gemm_w8a8_workspace_size(N, K, M)))
        for _ in range(args.warmup + 3):
            q8.q8_gemm_w8a8(q0, s0, x, y=y, ws=ws)
    elif args.profile == "prefill":
        K, N = synth.SWEEP_SHAPES[0]
        M = synth.PREFILL_M
        q0, s0 = q8.q8_quantize_rows(torch.from_numpy(synth.weights(N, K, 0, f"pf{K}.{N}")).cuda())
        x = torch.from_numpy(synth.activations(M, K, 0, f"pfx{K}").view(np.int16)).view(torch.bfloat16).cuda()
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        for _ in range(args.warmup + 3):
            q8.q8_gemm(q0, s0, x, y)
    else:
        N, K = synth.VOCAB, synth.HIDDEN
        wq, ws_ = q8.q8_quantize_rows(torch.from_numpy(synth.weights(N, K, 0, "vocab")).cuda())
        xv = torch.from_numpy(synth.unit_activation(K, 0).view(np.int16)).view(torch.bfloat16).cuda()
        yv = torch.empty((1, N), dtype=torch.float32, device="cuda")
        for _ in range(args.warmup + 3):
            q8.q8_linear_batch([(wq, ws_, xv, yv)], variant=args.variant)
    torch.cuda.synchronize()
    log("profile case done")
    return 0


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--variant", type=int, default=0, help="0 auto, 1 SIMT, 2 MMA")
    ap.add_argument("--no-rows", action="store_true", help="skip the context rows")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-chain", action="store_true",
                    help="launch the passes with q8_linear_batch instead of q8_linear_batch_chained")
    ap.add_argument("--profile", choices=["layerset", "vocab", "prefill", "sweep8", "tile16", "oddk16", "chain", "w8a8", "tile32"], default=None,
                    help="run a few launches of one workload and exit (for ncu captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return reference_arm(args, rank, world)

    import torch
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from block_quantized_int8_gb300 import build, q8
    if rank == 0 or world == 1:
        build.build()
    if dist:
        dist.barrier()
    q8.lib()

    if args.profile:
        return profile_case(torch, q8, args)

    peaks, peak_src = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    bytes_step, bytes_pass = layer_set_bytes(1)

    log("building the layer set ...")
    ls = LayerSet(torch, q8)
    chained = args.variant == 0 and not args.no_chain
    fn = lambda: ls.step(args.variant, chained=chained)  # noqa: E731

    clk = ClockSampler(local_rank)
    clk.start()
    # warm the GPU for a moment so the sampled clocks describe steady load
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    temp_start = gpu_temperature(local_rank)
    dt, block_step_s = time_blocks(torch, fn, args.steps)
    temp_end = gpu_temperature(local_rank)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = clk.stop()
    t_max = max_over_ranks(torch, dist, dt, "cuda")
    value = whole_job_gbs(bytes_step, args.steps, t_max, world)

    # kernel duration, live, on the launching stream
    launch_ms = per_launch_ms(torch, ls, reps=20, variant=args.variant)
    achieved = bytes_pass / (launch_ms / 1e3) / 1e9
    traffic, _ = profile_traffic()

    e2e, h2d, d2h = e2e_gbs(torch, ls, max(20, min(200, args.steps // 10)), bytes_step, chained)
    c_copy, c_read = ceilings(torch, q8)

    rows = {} if (args.no_rows or rank != 0) else extra_rows(torch, q8, peak)
    if rows:
        # the same step, plain and chained, captured once into a CUDA graph
        for ch, cn in ((False, "plain"), (True, "chained")):
            g = torch.cuda.CUDAGraph()
            s_ = torch.cuda.Stream()
            with torch.cuda.stream(s_):
                ls.step(chained=ch)
            s_.synchronize()
            with torch.cuda.graph(g, stream=s_):
                ls.step(chained=ch)
            dtg = time_steps(torch, g.replay, 200, 5)
            rows[f"layer_set_step_graph_{cn}"] = {"GB/s": round(bytes_step * 200 / dtg / 1e9, 1),
                                                 "frac": round(bytes_step * 200 / dtg / 1e9 / peak, 3),
                                                 "us_per_step": round(dtg / 200 * 1e6, 2)}
            del g
        # the token as a dependent chain (each matmul's input from the one before)
        rows.update(chain_rows(torch, q8, ls, peak))

    cpu = None
    if rank == 0 and not args.no_cpu:
        v, cores, sample = oracle_sample()
        v1, _, sample1 = oracle_sample(budget_s=8.0, threads=1)
        cpu = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
               "cpu_model": cpu_model(),
               "single_thread": {"value": round(v1, 4), "unit": "GB/s", "cores": 1, "sample": sample1}}
    blk_gbs = [bytes_step / t / 1e9 for t in block_step_s]
    med, p10, p90 = spread(blk_gbs)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_max / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8xbf16->f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": 1, "layers": synth.LAYERS, "passes": synth.PASSES,
                       "bytes_per_step": bytes_step,
                       "launch": ("one q8_linear_batch_chained per pass (64 matrices; weights fixed, so each "
                                  "launch may start while the previous one finishes)") if chained
                       else "one q8_linear_batch per pass (64 matrices)",
                       "variant": ["auto", "simt", "mma"][args.variant],
                       "l2": "no flush: 481 MB of weights per pass > 129 MB L2",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                         else "fallback 6.8 TB/s", "kernel": "gemv_kernel (q8_linear_batch, M=1, one pass of 64 matrices)",
                         "launch_us": round(launch_ms * 1e3, 2), "bytes_per_launch": bytes_pass},
            "ceilings": {"d2d_copy_gbs": round(c_copy, 1), "stream_read_gbs": round(c_read, 1),
                         "step_frac_of_copy": round(value / world / c_copy, 4),
                         "step_frac_of_read": round(value / world / c_read, 4),
                         "launch_frac_of_read": round(achieved / c_read, 4),
                         "note": "measured in this run: cudaMemcpyAsync D2D (read+write bytes) and q8_stream_read"},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": ls.launches_per_step * args.steps,
            "clocks": clocks,
            "timing": {"blocks": len(block_step_s), "steps_per_block": round(args.steps / len(block_step_s), 3),
                       "unit": "GB/s (rank 0, per block)", "median": round(med, 2), "p10": round(p10, 2),
                       "p90": round(p90, 2), "gpu_temp_c_start": temp_start, "gpu_temp_c_end": temp_end,
                       "note": "the timed steps in consecutive blocks, a CUDA event between blocks on the "
                               "launching stream; value = all bytes / first-to-last event time"},
            "frac_of_peak": round(value / world / peak, 4),
            "rows": rows,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
