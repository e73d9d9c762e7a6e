"""Benchmark of the folded-Hadamard ternary Packed layer on GB300.

Default workload (one "step" = one decode token, M = 1): the embedding lookup of
one token id plus the 401 packed linears of a synthetic 64-layer Bonsai-2 27B text
stack (48 linear-attention layers: in_proj_qkv, in_proj_z, out_proj; 16 full-
attention layers: q, k, v, o; 64 MLPs: gate, up, down; lm_head), every linear
the fused sign*FWHT + W2-g128 GEMV.  25.1e9 weights = 7.06 GB of packed codes,
scales and biases stream from HBM per token; the step is replayed as one CUDA
graph.  Weights are far larger than L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  ``--config`` picks other workloads for profiling
(layers, prefill, batched, embed, fwht, transcode, all); they print one JSON line each.
``--impl reference`` times the float64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import tb_inputs as ti  # noqa: E402

METRIC = "decode tok/s at 27B shapes (M=1) + fused W2 GEMV HBM GB/s as % of GB300 peak"
# DRAM bytes (read + write) of one chain launch from an ncu capture, or None until taken
CHAIN_TRAFFIC = None
# DRAM bytes per launch of the per-call decode GEMV over its algorithmic bytes, from an ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum) of the kernel as it is now (scales and
# biases in the TMA ring): 25,150,208 B read, 0 written, for 25,067,520 B of 5120 -> 17408
# weights (profiles/w2_gemv_tma_5120x17408_traffic.md).
GEMV_TRAFFIC_RATIO = 25150208 / 25067520
GEMV_TRAFFIC_NOTE = "not captured"
CHAIN_TRAFFIC_NOTE = "not captured yet for this kernel"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)),
                "measured")
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS, "fallback"


# ---------------------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Dist:
    def __init__(self, backend):
        import torch
        import torch.distributed as td

        self.world, self.rank, self.local = dist_env()
        self.td = td if self.world > 1 else None
        if self.td is not None:
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            td.init_process_group(backend)
        self.torch = torch

    def barrier(self):
        if self.td is not None:
            self.td.barrier()

    def max(self, v: float) -> float:
        if self.td is None:
            return v
        t = self.torch.tensor([v], dtype=self.torch.float64,
                              device="cuda" if self.td.get_backend() == "nccl" else "cpu")
        self.td.all_reduce(t, op=self.td.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.td is not None:
            self.td.destroy_process_group()


# ---------------------------------------------------------------------------- clocks
class NvmlSampler:
    """Read-only NVML sampling (ctypes into the driver's libnvidia-ml) in a background thread:
    SM clock, its maximum, power and the clock-event reasons every `period` seconds.  Short timed
    regions (tens of ms) still get samples, which nvidia-smi's 100 ms loop would miss."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_dev: int, period: float = 0.002):
        import ctypes
        import threading

        self.ok = False
        self.samples = []
        self.period = period
        self.stop_ev = threading.Event()
        self.thread = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            bus = None
            try:
                import torch
                pr = torch.cuda.get_device_properties(torch_dev)
                bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
            except Exception:
                bus = None
            if bus is None or lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(torch_dev), ctypes.byref(h)) != 0:
                    return
            self.lib, self.h = lib, h
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 else None
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _one(self):
        import ctypes
        c, p, r = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) != 0:
            return None
        self.lib.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(p))
        self.reasons_fn(self.h, ctypes.byref(r))
        return time.time(), float(c.value), p.value / 1000.0, int(r.value)

    def _run(self):
        while not self.stop_ev.is_set():
            v = self._one()
            if v is not None:
                self.samples.append(v)
            time.sleep(self.period)

    def start(self):
        if self.ok:
            import threading
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()

    def stop(self, window):
        if self.thread is not None:
            self.stop_ev.set()
            self.thread.join(timeout=5)
        sel = [v for v in self.samples if window[0] <= v[0] <= window[1]]
        if not sel:
            return None
        reasons = set()
        for _, _, _, r in sel:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": float(np.median([v[1] for v in sel])), "sm_max_mhz": self.max_mhz,
                "power_w_max": round(max(v[2] for v in sel), 1), "reasons": sorted(reasons),
                "samples": len(sel), "source": f"NVML every {self.period * 1e3:.0f} ms in the timed region"}


class Clocks:
    """Clock samples during the timed region: NVML at 2 ms (read-only), with nvidia-smi's
    100 ms loop as the fallback where NVML cannot be loaded."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.window = None
        self.nvml = NvmlSampler(index)

    def mark(self, t0: float, t1: float):
        """Keep only samples taken between these wall-clock times (the timed region)."""
        self.window = (t0, t1)

    def start(self):
        self.nvml.start()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        fast = self.nvml.stop(self.window or (0.0, float("inf")))
        slow = self._stop_smi()
        if fast is not None:
            fast["nvidia_smi_samples"] = slow.get("samples", 0)
            return fast
        return slow

    def _stop_smi(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            if self.window is not None:
                try:
                    ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    ts = None
                if ts is not None and not (self.window[0] <= ts <= self.window[1]):
                    continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi every 100 ms"}


# ---------------------------------------------------------------------------- GPU workloads
class Packed:
    """One packed W2-g128 linear on the device (codes drawn by the device generator)."""

    def __init__(self, tb, tdev, torch, seed, N, K, tmp):
        dev = torch.device("cuda")
        self.N, self.K, self.G = N, K, K // 128
        self.w = torch.empty((N, K // 16), dtype=torch.int32, device=dev)
        self.s = torch.empty((N, self.G), dtype=torch.float16, device=dev)
        self.b = torch.empty((N, self.G), dtype=torch.float16, device=dev)
        step = tmp.numel() // K
        for r0 in range(0, N, step):
            n = min(step, N - r0)
            c = tmp[: n * K].view(n, K)
            tdev.fill_codes(c, seed, r0, K)
            tdev.fill_scales(self.s[r0:r0 + n], seed, r0, self.G)
            tb.tb_pack_w2(c, self.s[r0:r0 + n], self.w[r0:r0 + n], self.b[r0:r0 + n])

    @property
    def algo_bytes(self):
        return ti.packed_bytes(self.K, self.N)


class Stack:
    """The synthetic 64-layer stack on the device, wired as a dependent chain of links.

    Every link is one call of the layer: an input x and the 1..3 matrices of one layer that
    read it (in_proj_qkv + in_proj_z, q + k + v, gate + up) or one matrix alone.  A link's
    input is an earlier link's output, as in the model's decode step (the ops the model runs
    between the linears, attention, norms and the MLP gate, are not part of this layer and
    are left out): layer l reads h (x0 for l = 0); out_proj reads the in_proj_z output and
    o_proj the q output, and both write h; gate + up read h; down reads the gate output and
    writes h; lm_head reads h.  257 links per token.
    """

    def __init__(self, tb, tdev, torch):
        dev = torch.device("cuda")
        tmp = torch.empty(1 << 30, dtype=torch.int8, device=dev)
        self.layers = []
        for i, (name, K, N) in enumerate(ti.sweep_layers()):
            self.layers.append((name, Packed(tb, tdev, torch, ti.config_seed(3, i), N, K, tmp), i))
        self.emb = Packed(tb, tdev, torch, ti.config_seed(3, 999), ti.VOCAB, ti.HIDDEN, tmp)
        del tmp
        torch.cuda.synchronize()
        H, MLPW = ti.HIDDEN, ti.MLP
        self.x0 = torch.from_numpy(ti.activations(ti.config_seed(3, 1000), 1, H)).to(dev)
        self.signs = {K: torch.from_numpy(ti.rademacher_signs(ti.config_seed(3, 2000 + K), K)).to(dev)
                      for K in (H, 6144, MLPW)}

        def buf(n):
            return torch.zeros((1, n), dtype=torch.float16, device=dev)

        self.h, self.qkv, self.z = buf(H), buf(10240), buf(6144)
        self.q, self.k, self.v = buf(6144), buf(1024), buf(1024)
        self.gate, self.up = buf(MLPW), buf(MLPW)
        self.logits = buf(ti.VOCAB)
        out_of = {"in_proj_qkv": self.qkv, "in_proj_z": self.z, "out_proj": self.h, "q_proj": self.q,
                  "k_proj": self.k, "v_proj": self.v, "o_proj": self.h, "gate_proj": self.gate,
                  "up_proj": self.up, "down_proj": self.h, "lm_head": self.logits}
        in_of = {"out_proj": self.z, "o_proj": self.q, "down_proj": self.gate}
        # links: (x, K, [(name, Packed, layer index, y)])
        self.links = []
        first, i = True, 0
        while i < len(self.layers):
            name = self.layers[i][0]
            fam = next((f for f in SHARED_INPUT if name in f), None)
            j = i + 1
            if fam is not None:
                while j < len(self.layers) and self.layers[j][0] in fam and self.layers[j][0] != name:
                    j += 1
            grp = self.layers[i:j]
            x = in_of.get(name, self.h)
            if first:
                x, first = self.x0, False
            self.links.append((x, grp[0][1].K, [(n, p, li, out_of[n]) for n, p, li in grp]))
            i = j

    def link_args(self):
        """Arguments of every link for tb.chain_link / tb_packed_linear_multi."""
        return [(x, self.signs[K], 1024, [(p.w, p.s, p.b) for _, p, _, _ in mats],
                 [y[:, : p.N] for _, p, _, y in mats]) for x, K, mats in self.links]

    @property
    def algo_bytes(self):
        return sum(p.algo_bytes for _, p, _ in self.layers)

    @property
    def scale_only_bytes(self):
        """Bytes of the step's matrices without the biases (1/64 byte per weight less)."""
        return sum(p.algo_bytes - p.N * p.G * 2 for _, p, _ in self.layers)


SHARED_INPUT = ({"in_proj_qkv", "in_proj_z"}, {"q_proj", "k_proj", "v_proj"}, {"gate_proj", "up_proj"})


def run_calls(tb, link_args, ws, status):
    """The links as one tb_packed_linear(_multi) call each, in order on the current stream."""
    for x, sg, block, mats, ys in link_args:
        if len(mats) == 1:
            w, s, b = mats[0]
            tb.tb_packed_linear(x, sg, block, w, s, b, ys[0], ws, status)
        else:
            tb.tb_packed_linear_multi(x, sg, block, mats, ys, ws, status)


def gguf_links(tb, torch, links0, fmt, status):
    """The scale-only links with every matrix re-encoded on the device as GGUF blocks of fmt
    (tb_encode_gguf), each matrix one tb_gguf_linear call (its own rotation of the link's input).
    Returns (calls, bytes of the blocks, the block tensors)."""
    dev = torch.device("cuda")
    bpb = 34 if fmt == tb.TB_FMT_PQ2_0 else 28
    calls, keep, nbytes = [], [], 0
    for x, sg, block, mats, ys in links0:
        for (w, s, _), y in zip(mats, ys):
            N, G = s.shape
            blk = torch.empty(N * G * bpb, dtype=torch.uint8, device=dev)
            tb.tb_encode_gguf(w, s, fmt, blk, status)
            keep.append(blk)
            nbytes += blk.numel()
            calls.append((x, sg, block, blk, y))
    return calls, nbytes, keep


def run_gguf(tb, calls, fmt, ws, status):
    for x, sg, block, blk, y in calls:
        tb.tb_gguf_linear(x, sg, block, blk, fmt, y, ws, status)


def embed(tb, st, ids, e_out, status, biases=True):
    tb.tb_embed_lookup(ids, st.emb.w, st.emb.s, st.emb.b if biases else None, st.signs[ti.HIDDEN],
                       1024, e_out, status)


def time_graph(torch, graph, steps, dist):
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    start.record()
    for _ in range(steps):
        graph.replay()
    end.record()
    torch.cuda.synchronize()
    dist.barrier()
    return start.elapsed_time(end) / 1e3


def capture(torch, fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # attributes set, lazy loads done before capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def sub_results(tb, st, torch, status, reps: int = 5):
    """Compact per-kernel numbers on the resident stack (no new weights): every distinct link of
    the decode step as its own CUDA graph over all its copies (GEMV GB/s), batched decode on the
    64 gate_proj matrices, prefill on gate_proj and down_proj with the L2 flushed, and the
    embedding of 256 ids."""
    hbm, tf, _, _ = peaks()
    dev = torch.device("cuda")
    links = st.link_args()
    ws = torch.zeros(tb.tb_packed_linear_workspace_size(64, ti.MLP, ti.HIDDEN), dtype=torch.uint8, device=dev)
    out = {}

    def timed_graph(fn, n_calls):
        g = capture(torch, fn)
        for _ in range(2):
            g.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3 / (reps * n_calls)

    # the decode step's links, grouped by kind (M = 1)
    kinds = {}
    for (x, K, mats), la in zip(st.links, links):
        kinds.setdefault("+".join(m[0] for m in mats), []).append((la, sum(p.algo_bytes for _, p, _, _ in mats)))
    rows = []
    for name, lst in kinds.items():
        sec = timed_graph(lambda lst=lst: run_calls(tb, [la for la, _ in lst], ws, status), len(lst))
        byts = lst[0][1]
        rows.append({"link": name, "count": len(lst), "us": round(sec * 1e6, 2),
                     "GB/s": round(byts / sec / 1e9, 1), "frac": round(byts / sec / 1e9 / hbm, 4)})
    out["decode_links_m1"] = rows

    # batched decode on the 64 gate_proj matrices (5120 -> 17408; far more than L2 per pass)
    gates = [p for n, p, _ in st.layers if n == "gate_proj"]
    sg = st.signs[ti.HIDDEN]
    rows = []
    for M in (1, 2, 4, 8, 16, 32, 64):
        x = torch.from_numpy(ti.activations(ti.config_seed(5, M), M, ti.HIDDEN)).to(dev)
        y = torch.empty((M, ti.MLP), dtype=torch.float16, device=dev)

        def fn(x=x, y=y):
            for p in gates:
                tb.tb_packed_linear(x, sg, 1024, p.w, p.s, p.b, y, ws, status)

        sec = timed_graph(fn, len(gates))
        byts = gates[0].algo_bytes
        rows.append({"M": M, "us": round(sec * 1e6, 2), "frac_hbm": round(byts / sec / 1e9 / hbm, 4),
                     "TFLOP/s": round(2 * M * ti.MLP * ti.HIDDEN / sec / 1e12, 1)})
    out["batched_5120x17408"] = rows

    # prefill on one gate_proj and one down_proj matrix, L2 flushed before every call
    flush = torch.empty(256 << 20, dtype=torch.int8, device=dev)
    down = next(p for n, p, _ in st.layers if n == "down_proj")
    rows = []
    for M in (512, 4096):
        for p in (gates[0], down):
            x = torch.from_numpy(ti.activations(ti.config_seed(4, p.K), M, p.K)).to(dev)
            y = torch.empty((M, p.N), dtype=torch.float16, device=dev)
            wsp = torch.zeros(tb.tb_packed_linear_workspace_size(M, p.K, p.N), dtype=torch.uint8, device=dev)
            sgp = st.signs[p.K]
            for _ in range(2):
                tb.tb_packed_linear(x, sgp, 1024, p.w, p.s, p.b, y, wsp, status)
            tot = 0.0
            for _ in range(3):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                tb.tb_packed_linear(x, sgp, 1024, p.w, p.s, p.b, y, wsp, status)
                b.record()
                torch.cuda.synchronize()
                tot += a.elapsed_time(b) / 1e3
            sec = tot / 3
            tfl = 2.0 * M * p.N * p.K / sec / 1e12
            rows.append({"shape": f"M={M} {p.K}->{p.N}", "ms": round(sec * 1e3, 3), "TFLOP/s": round(tfl, 1),
                         "frac": round(tfl / tf, 4)})
            del x, y, wsp
    out["prefill"] = rows

    # embedding: 256 uniform ids from the 248320-row table, L2 flushed
    T = 256
    ids = torch.from_numpy(ti.token_ids(ti.config_seed(5, 99), T, ti.VOCAB)).to(dev)
    e = torch.empty((T, ti.HIDDEN), dtype=torch.float16, device=dev)
    tot = []
    for r in range(4):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        tb.tb_embed_lookup(ids, st.emb.w, st.emb.s, st.emb.b, sg, 1024, e, status)
        b.record()
        torch.cuda.synchronize()
        tot.append(a.elapsed_time(b) / 1e3)
    sec = float(np.median(tot[1:]))
    byts = T * (ti.HIDDEN // 4 + ti.HIDDEN // 32) + T * ti.HIDDEN * 2
    out["embedding_256_ids"] = {"us": round(sec * 1e6, 2), "GB/s": round(byts / sec / 1e9, 1),
                                "frac_hbm": round(byts / sec / 1e9 / hbm, 4)}
    del flush
    out["note"] = ("builder-side sub-results measured in this run: per-link CUDA graphs over every copy of a "
                   "link (M = 1), batched decode over the 64 gate_proj copies, prefill and embedding with "
                   "the L2 flushed before each call")
    return out


def stack_parity(st, x, y, rows: int = 256):
    """The oracle on `rows` sampled rows of lm_head, on the input h of the last timed step (x),
    against that step's logits (y): max and RMS error over RMS(y) (the float64 oracle runs in
    the CPU-baseline leg only)."""
    import oracle

    _, K, mats = st.links[-1]
    _, p, layer, _ = mats[0]
    rng = np.random.default_rng(17)
    sel = np.sort(rng.choice(p.N, size=rows, replace=False))
    seed = ti.config_seed(3, layer)
    codes = np.concatenate([ti.ternary_codes(seed, r, r + 1, K) for r in sel])
    scales = np.concatenate([ti.group_scales(seed, r, r + 1, K // 128) for r in sel])
    words = oracle.pack_w2(codes)
    xf = x.cpu().numpy().astype(np.float64)
    ref = oracle.packed_linear(xf, st.signs[K].cpu().numpy(), 1024, words, scales, oracle.biases_for(scales))
    got = y[:, : p.N].cpu().numpy()[:, sel].astype(np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2))) or 1.0
    err = np.abs(got - ref)
    return {"link": "lm_head 5120->248320", "rows": rows, "max_err_over_rms_y": round(float(err.max()) / rms, 6),
            "rms_err_over_rms_y": round(float(np.sqrt(np.mean(err ** 2))) / rms, 6)}


def cpu_baseline_sample(budget_s: float = 12.0):
    """The float64 oracle on sampled rows of every distinct sweep shape, M = 1.

    Returns (tok/s extrapolated to the full 401-linear step + embedding, description).
    """
    import oracle

    shapes = {}
    for _, K, N in ti.sweep_layers():
        shapes[(K, N)] = shapes.get((K, N), 0) + 1
    per_shape = budget_s / len(shapes)
    sec_per_token = 0.0
    desc = []
    for (K, N), count in sorted(shapes.items()):
        x = ti.activations(7, 1, K)
        sg = ti.rademacher_signs(7, K)
        rows = 64
        while True:
            codes = ti.ternary_codes(11, 0, rows, K)
            sc = ti.group_scales(11, 0, rows, K // 128)
            w = oracle.pack_w2(codes)
            b = oracle.biases_for(sc)
            t0 = time.perf_counter()
            oracle.packed_linear(x, sg, 1024, w, sc, b)
            dt = time.perf_counter() - t0
            if dt > per_shape / 3 or rows >= N:
                break
            rows = min(N, rows * 4)
        sec_per_token += count * dt * (N / rows)
        desc.append(f"{K}->{N}x{count}: {rows} rows")
    # embedding of one id: dequantise one 5120 row + inverse transform
    codes = ti.ternary_codes(12, 0, 16, ti.HIDDEN)
    sc = ti.group_scales(12, 0, 16, ti.HIDDEN // 128)
    w = oracle.pack_w2(codes)
    t0 = time.perf_counter()
    oracle.embed_lookup(np.arange(16), w, sc, oracle.biases_for(sc), ti.rademacher_signs(1, ti.HIDDEN), 1024)
    sec_per_token += (time.perf_counter() - t0) / 16
    return 1.0 / sec_per_token, "; ".join(desc)


def run_sweep(args, dist, tb, tdev, torch):
    """The decode step (embedding + 257 dependent links) timed on one of two paths:
    `chain` (one persistent tb_chain_run launch for all links) or `calls` (one launch per
    link, replayed as a CUDA graph).  The other path is timed too and reported in config."""
    hbm, _, _, peak_kind = peaks()
    st = Stack(tb, tdev, torch)
    links = st.link_args()
    dev = torch.device("cuda")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ids = torch.tensor([int(ti.token_ids(ti.config_seed(3, 3000), 1, ti.VOCAB)[0])], dtype=torch.int32,
                       device=dev)
    e_out = torch.empty((1, ti.HIDDEN), dtype=torch.float16, device=dev)
    chain = tb.Chain(links, 1)
    n_links = len(links)
    step_bytes = st.algo_bytes
    ws = torch.zeros(tb.tb_packed_linear_workspace_size(1, ti.MLP, ti.HIDDEN), dtype=torch.uint8, device=dev)
    call_graph = capture(torch, lambda: (embed(tb, st, ids, e_out, status), run_calls(tb, links, ws, status)))
    # scale-only form: no biases passed, each taken as -scale by the kernels (same results)
    links0 = [(x, sg, blk, [(w, s, None) for w, s, _ in mats], ys) for x, sg, blk, mats, ys in links]
    scale_graph = capture(torch, lambda: (embed(tb, st, ids, e_out, status, biases=False),
                                          run_calls(tb, links0, ws, status)))
    gemv_graph = capture(torch, lambda: run_calls(tb, links, ws, status))
    # the same step read straight from GGUF blocks (PTQ1_0: 1.75 bits per weight; PQ2_0: 2.125)
    gws = torch.empty(tb.tb_gguf_linear_workspace_size(1, ti.MLP, 1024), dtype=torch.uint8, device=dev)
    gguf = {}
    for name, fmt in (("PTQ1_0", tb.TB_FMT_PTQ1_0), ("PQ2_0", tb.TB_FMT_PQ2_0)):
        calls, nbytes, keep = gguf_links(tb, torch, links0, fmt, status)
        g = capture(torch, lambda calls=calls, fmt=fmt: (embed(tb, st, ids, e_out, status, biases=False),
                                                         run_gguf(tb, calls, fmt, gws, status)))
        gguf[name] = (g, nbytes, keep)

    def chain_step():
        embed(tb, st, ids, e_out, status)
        chain.run(status)

    def calls_step():
        call_graph.replay()

    step = chain_step if args.path == "chain" else calls_step

    def time_steps(fn, steps):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        dist.barrier()
        torch.cuda.synchronize()
        start.record()
        for _ in range(steps):
            fn()
        end.record()
        torch.cuda.synchronize()
        dist.barrier()
        return start.elapsed_time(end) / 1e3

    clocks = Clocks(dist.local)
    clocks.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    t_pre = time.time()
    while time.time() - t_pre < 0.3:  # the sampler is up and the GPU busy before the timed region
        step()
        torch.cuda.synchronize()
    w0 = time.time()
    secs = dist.max(time_steps(step, args.steps))
    clocks.mark(w0, time.time())
    clk = clocks.stop()
    # the dominant kernel alone: the chain launch, or the 257 per-link GEMV launches
    if args.path == "chain":
        ksecs = dist.max(time_steps(lambda: chain.run(status), args.steps))
        launches_per_link = 1.0 / n_links
        kernel = ("w2_gemv_chain_kernel<1> (257 links: fused FWHT prologue + W2-g128 GEMV each), "
                  "algorithmic bytes of the 401 matrices per launch over its CUDA-event time")
    else:
        for _ in range(2):
            gemv_graph.replay()
        ksecs = dist.max(time_steps(gemv_graph.replay, args.steps))
        launches_per_link = 1.0
        kernel = ("w2_gemv_tma_kernel<1> (fused FWHT prologue + W2-g128 GEMV), its 257 launches per "
                  "token averaged")
    other = calls_step if args.path == "chain" else chain_step
    for _ in range(3):
        other()
    osecs = dist.max(time_steps(other, args.steps))
    for _ in range(3):
        scale_graph.replay()
    ssecs = dist.max(time_steps(scale_graph.replay, args.steps))
    gsecs = {}
    for name, (g, nbytes, _) in gguf.items():
        for _ in range(3):
            g.replay()
        gsecs[name] = (dist.max(time_steps(g.replay, args.steps)), nbytes)
    del gguf
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    assert bool(torch.isfinite(st.logits).all()), "non-finite logits"
    launches = n_links * launches_per_link
    achieved = step_bytes / launches / (ksecs / (args.steps * launches)) / 1e9

    # end to end through the public C ABI with host buffers: H2D of the token id, the
    # step's calls, D2H of the logits, every step (no graph)
    h_id = torch.empty(1, dtype=torch.int32).pin_memory()
    h_id[0] = int(ids[0])
    h_logits = torch.empty((1, ti.VOCAB), dtype=torch.float16).pin_memory()

    def e2e_step():
        ids.copy_(h_id, non_blocking=True)
        if args.path == "chain":
            chain_step()
        else:
            embed(tb, st, ids, e_out, status)
            run_calls(tb, links, ws, status)
        h_logits.copy_(st.logits, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = dist.max(time.perf_counter() - t0)
    dist.barrier()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    n = dist.world
    per_step = 2 if args.path == "chain" else 1 + n_links
    line = {
        "metric": METRIC,
        "value": round(n * args.steps / secs, 3),
        "unit": "tok/s",
        "n_gpus": n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic",
        "config": {
            "workload": "decode step, M=1: embedding of 1 id + 401 fused sign*FWHT-1024 + W2-g128 "
                        "linears of a 64-layer 27B stack (hidden 5120, MLP 17408, vocab 248320) as a "
                        "dependent chain of 257 links (each link reads an earlier link's output)",
            "weights_gb_per_step": round((step_bytes + ti.HIDDEN // 4 + ti.HIDDEN // 32) / 1e9, 4),
            "l2": "no flush: 7.06 GB of weights per step, far larger than the 129 MB L2",
            "path": ("chain: embedding + one persistent tb_chain_run launch per step" if args.path == "chain"
                     else "calls: embedding + one tb_packed_linear(_multi) launch per link, one CUDA graph per step"),
            "links_per_step": n_links,
            "shared_input_links": "in_proj_qkv+in_proj_z, q+k+v and gate+up each one link",
            ("tok_s_calls_path" if args.path == "chain" else "tok_s_chain_path"): round(n * args.steps / osecs, 3),
            "scale_only": {
                "tok_s": round(n * args.steps / ssecs, 3),
                "weights_gb_per_step": round((st.scale_only_bytes + ti.HIDDEN // 4 + ti.HIDDEN // 64) / 1e9, 4),
                "note": "calls path with biases = NULL (each bias is the pack's -scale, not read); "
                        "the same arithmetic on the same values as the stored-bias step",
            },
            "gguf": {
                **{name: {"tok_s": round(n * args.steps / sec, 3),
                          "weights_gb_per_step": round((nb + ti.HIDDEN // 4 + ti.HIDDEN // 64) / 1e9, 4)}
                   for name, (sec, nb) in gsecs.items()},
                "note": "the same trits and scales re-encoded on the device as GGUF blocks (tb_encode_gguf) "
                        "and read straight from them (tb_gguf_linear, decoded on the CUDA cores), one call "
                        "per matrix with its own rotation of the link's input; embedding as in scale_only",
            },
            "parallelism": f"replicas x{n}",
        },
        "roofline": {
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": hbm,
            "unit": "GB/s",
            "frac": round(achieved / hbm, 4),
            "traffic": CHAIN_TRAFFIC if args.path == "chain" else
            (round(GEMV_TRAFFIC_RATIO * step_bytes / n_links) if GEMV_TRAFFIC_RATIO else None),
            "traffic_note": CHAIN_TRAFFIC_NOTE if args.path == "chain" else
            ("ncu DRAM bytes of the 5120->17408 launch, scaled to the step's average launch"
             if GEMV_TRAFFIC_RATIO else GEMV_TRAFFIC_NOTE),
            "kernel": kernel,
            "peak_kind": f"{peak_kind} hbm_gbs",
        },
        "e2e": {
            "value": round(n * args.steps / e2e_s, 3),
            "unit": "tok/s",
            "h2d_bytes_per_step": 4,
            "d2h_bytes_per_step": ti.VOCAB * 2,
            "note": "C-ABI calls per step from the host: token id H2D, the step's launches, logits D2H",
        },
        "gpu_launches": per_step * args.steps,
        "clocks": clk,
    }
    # the last step's lm_head input and output, kept for the parity diagnostic below
    h_last, logits_last = st.h.clone(), st.logits.clone()
    if not args.no_sub_results:
        line["sub_results"] = sub_results(tb, st, torch, status)
    if dist.rank == 0 and n == 1 and not args.no_cpu_baseline:
        v, desc = cpu_baseline_sample()
        line["cpu_baseline"] = {"value": round(v, 6), "unit": "tok/s",
                                "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                                "sample": "float64 NumPy oracle, M=1, sampled rows of every distinct "
                                          "sweep shape, extrapolated to the 401 linears + embedding: " + desc}
        # the same leg's oracle on sampled lm_head rows of the last step, against its logits
        line["parity"] = stack_parity(st, h_last, logits_last)
    return line


def profile_step(args, dist, tb, tdev, torch):
    """Two decode steps (embedding + chain run) after building the stack, nothing timed; with
    --per-call the 257 links run as one launch each instead of one chain launch."""
    st = Stack(tb, tdev, torch)
    links = st.link_args()
    dev = torch.device("cuda")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ids = torch.tensor([7], dtype=torch.int32, device=dev)
    e_out = torch.empty((1, ti.HIDDEN), dtype=torch.float16, device=dev)
    if args.per_call:
        ws = torch.zeros(tb.tb_packed_linear_workspace_size(1, ti.MLP, ti.HIDDEN), dtype=torch.uint8,
                         device=dev)
        for _ in range(2):
            embed(tb, st, ids, e_out, status)
            run_calls(tb, links, ws, status)
    else:
        chain = tb.Chain(links, 1)
        for _ in range(2):
            embed(tb, st, ids, e_out, status)
            chain.run(status)
    torch.cuda.synchronize()
    return {"profile_step": "done", "links": len(links), "status": int(status.item())}


def profile_fwht(args, dist, tb, tdev, torch):
    """Four tb_fwht calls (forward, with signs) on M x K activations, nothing timed."""
    M, K = args.profile_fwht
    dev = torch.device("cuda")
    x = torch.from_numpy(ti.activations(6, M, K)).to(dev)
    y = torch.empty_like(x)
    sg = torch.from_numpy(ti.rademacher_signs(6, K)).to(dev)
    for _ in range(4):
        tb.tb_fwht(x, y, sg, 1024, False)
    torch.cuda.synchronize()
    return {"profile_fwht": [M, K]}


def profile_linear(args, dist, tb, tdev, torch):
    """Four calls of one K -> N packed linear on M tokens with algorithm ALGO, nothing timed."""
    K, N, M, algo = args.profile_linear
    dev = torch.device("cuda")
    tmp = torch.empty(min(N * K, 1 << 30), dtype=torch.int8, device=dev)
    p = Packed(tb, tdev, torch, 1, N, K, tmp)
    del tmp
    x = torch.from_numpy(ti.activations(1, M, K)).to(dev)
    sg = torch.from_numpy(ti.rademacher_signs(1, K)).to(dev)
    y = torch.empty((M, N), dtype=torch.float16, device=dev)
    ws = torch.zeros(max(16, tb.tb_packed_linear_workspace_size(M, K, N, 1024, algo)), dtype=torch.uint8,
                     device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(4):
        tb.tb_packed_linear(x, sg, 1024, p.w, p.s, p.b, y, ws, status, algo=algo)
    torch.cuda.synchronize()
    return {"profile_linear": [K, N, M, algo], "status": int(status.item())}


def profile_embed(args, dist, tb, tdev, torch):
    """Four tb_embed_lookup calls of 256 uniform ids on the 248320 x 5120 table, nothing timed."""
    dev = torch.device("cuda")
    tmp = torch.empty(1 << 30, dtype=torch.int8, device=dev)
    p = Packed(tb, tdev, torch, ti.config_seed(5, 99), ti.VOCAB, ti.HIDDEN, tmp)
    del tmp
    sg = torch.from_numpy(ti.rademacher_signs(5, ti.HIDDEN)).to(dev)
    ids = torch.from_numpy(ti.token_ids(ti.config_seed(5, 99), 256, ti.VOCAB)).to(dev)
    out = torch.empty((256, ti.HIDDEN), dtype=torch.float16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(4):
        tb.tb_embed_lookup(ids, p.w, p.s, p.b, sg, 1024, out, status)
    torch.cuda.synchronize()
    return {"profile_embed": 256, "status": int(status.item())}


def run_layers(args, dist, tb, tdev, torch):
    """Per-shape decode GEMV at the 27B layer shapes (M = 1)."""
    hbm, _, _, peak_kind = peaks()
    dev = torch.device("cuda")
    tmp = torch.empty(1 << 30, dtype=torch.int8, device=dev)
    rows = []
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for name, K, N in ti.LAYER_SHAPES + [("qkv", 5120, 10240), ("lm_head", 5120, ti.VOCAB)]:
        # enough distinct copies that one pass exceeds L2
        copies = max(1, -(-(512 << 20) // ti.packed_bytes(K, N)))
        ps = [Packed(tb, tdev, torch, ti.config_seed(2, j), N, K, tmp) for j in range(copies)]
        x = torch.from_numpy(ti.activations(5, 1, K)).to(dev)
        sg = torch.from_numpy(ti.rademacher_signs(5, K)).to(dev)
        y = torch.empty((1, N), dtype=torch.float16, device=dev)
        ws = torch.zeros(tb.tb_packed_linear_workspace_size(1, K, N), dtype=torch.uint8, device=dev)

        def fn(biases=True):
            for p in ps:
                tb.tb_packed_linear(x, sg, 1024, p.w, p.s, p.b if biases else None, y, ws, status)

        reps = max(3, args.steps)
        per = {}
        for biases in (True, False):
            g = capture(torch, lambda: fn(biases))
            for _ in range(3):
                g.replay()
            per[biases] = time_graph(torch, g, reps, dist) / (reps * copies)
        gbs = ti.packed_bytes(K, N) / per[True] / 1e9
        gbs0 = (ti.packed_bytes(K, N) - N * (K // 128) * 2) / per[False] / 1e9
        rows.append({"shape": f"{name} {K}->{N}", "us": round(per[True] * 1e6, 2), "GB/s": round(gbs, 1),
                     "frac": round(gbs / hbm, 4), "copies": copies,
                     "scale_only_us": round(per[False] * 1e6, 2),
                     "scale_only_frac": round(gbs0 / hbm, 4)})
        del ps
    del tmp
    return {"metric": "decode GEMV per layer shape (M=1)", "unit": "GB/s", "peak": hbm,
            "peak_kind": peak_kind, "layers": rows}


def run_prefill(args, dist, tb, tdev, torch):
    _, tf, tfs, peak_kind = peaks()
    dev = torch.device("cuda")
    tmp = torch.empty(1 << 30, dtype=torch.int8, device=dev)
    rows = []
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for M in (512, 4096):
        for K, N in ((5120, 17408), (17408, 5120)):
            p = Packed(tb, tdev, torch, ti.config_seed(4, K), N, K, tmp)
            x = torch.from_numpy(ti.activations(4, M, K)).to(dev)
            sg = torch.from_numpy(ti.rademacher_signs(4, K)).to(dev)
            y = torch.empty((M, N), dtype=torch.float16, device=dev)
            ws = torch.zeros(tb.tb_packed_linear_workspace_size(M, K, N), dtype=torch.uint8, device=dev)
            flush = torch.empty(256 << 20, dtype=torch.int8, device=dev)

            def fn():
                tb.tb_packed_linear(x, sg, 1024, p.w, p.s, p.b, y, ws, status)

            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            reps = max(3, args.steps)
            tot = 0.0
            for _ in range(reps):
                flush.zero_()  # L2 flush between timed iterations
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b.record()
                torch.cuda.synchronize()
                tot += a.elapsed_time(b) / 1e3
            per = tot / reps
            tflops = 2.0 * M * N * K / per / 1e12
            rows.append({"shape": f"M={M} {K}->{N}", "ms": round(per * 1e3, 4), "TFLOP/s": round(tflops, 1),
                         "frac": round(tflops / tf, 4)})
            del p, x, y, ws, flush
    del tmp
    return {"metric": "prefill GEMM (FWHT prologue + tcgen05 GEMM)", "unit": "TFLOP/s", "peak": tf,
            "peak_kind": f"{peak_kind} bf16 burst (fp16 dense rate equal)", "rows": rows}


def run_batched(args, dist, tb, tdev, torch):
    hbm, _, _, peak_kind = peaks()
    dev = torch.device("cuda")
    tmp = torch.empty(1 << 30, dtype=torch.int8, device=dev)
    K, N = 5120, 17408
    copies = 8
    ps = [Packed(tb, tdev, torch, ti.config_seed(5, j), N, K, tmp) for j in range(copies)]
    del tmp
    sg = torch.from_numpy(ti.rademacher_signs(5, K)).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    rows = []
    for M in (1, 2, 4, 8, 16, 32, 64):
        x = torch.from_numpy(ti.activations(5, M, K)).to(dev)
        y = torch.empty((M, N), dtype=torch.float16, device=dev)
        ws = torch.zeros(tb.tb_packed_linear_workspace_size(M, K, N), dtype=torch.uint8, device=dev)

        def fn():
            for p in ps:
                tb.tb_packed_linear(x, sg, 1024, p.w, p.s, p.b, y, ws, status)

        g = capture(torch, fn)
        for _ in range(3):
            g.replay()
        reps = max(3, args.steps)
        per = time_graph(torch, g, reps, dist) / (reps * copies)
        gbs = ti.packed_bytes(K, N) / per / 1e9
        rows.append({"M": M, "us": round(per * 1e6, 2), "GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4),
                     "TFLOP/s": round(2 * M * N * K / per / 1e12, 2)})
    return {"metric": "batched decode 5120->17408", "unit": "GB/s", "peak": hbm, "peak_kind": peak_kind,
            "rows": rows}


def run_fwht(args, dist, tb, tdev, torch):
    """tb_fwht alone (forward, with signs) on activations larger than L2."""
    hbm, _, _, peak_kind = peaks()
    dev = torch.device("cuda")
    rows = []
    # the pack's block (1024) on both model widths, then the other blocks the loader accepts
    cases = [(4096, 17408, 1024), (16384, 5120, 1024), (8192, 8192, 512), (8192, 8192, 2048), (8192, 8192, 4096)]
    for M, K, block in cases:
        x = torch.from_numpy(ti.activations(6, M, K)).to(dev)
        y = torch.empty_like(x)
        sg = torch.from_numpy(ti.rademacher_signs(6, K)).to(dev)
        flush = torch.empty(256 << 20, dtype=torch.int8, device=dev)
        for _ in range(3):
            tb.tb_fwht(x, y, sg, block, False)
        torch.cuda.synchronize()
        reps = max(3, args.steps)
        tot = 0.0
        for _ in range(reps):
            flush.zero_()  # L2 flush between timed iterations
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            tb.tb_fwht(x, y, sg, block, False)
            b.record()
            torch.cuda.synchronize()
            tot += a.elapsed_time(b) / 1e3
        per = tot / reps
        byts = 4 * M * K + K  # x read, y written, signs
        rows.append({"shape": f"M={M} K={K} block={block}", "us": round(per * 1e6, 2),
                     "GB/s": round(byts / per / 1e9, 1), "frac": round(byts / per / 1e9 / hbm, 4)})
        del x, y, flush
    return {"metric": "sign * FWHT (tb_fwht, forward)", "unit": "GB/s", "peak": hbm, "peak_kind": peak_kind,
            "rows": rows}


def run_transcode(args, dist, tb, tdev, torch):
    """tb_transcode_gguf on the lm_head-sized table (248320 x 5120), both GGUF formats.

    The blocks are random valid blocks built on the device: fp16 scales in [0.005, 0.02];
    PQ2_0 code bytes drawn from the 81 bytes whose four 2-bit slots are all trits, PTQ1_0 bytes
    uniform in [0, 243) (the last byte of a block in [0, 27)).  Bytes moved: the blocks read,
    the words, scales and biases written."""
    hbm, _, _, peak_kind = peaks()
    dev = torch.device("cuda")
    V, D = ti.VOCAB, ti.HIDDEN
    nb = V * (D // 128)
    g = torch.Generator(device=dev)
    g.manual_seed(ti.config_seed(5, 700))
    sc = (torch.rand(nb, generator=g, device=dev) * 0.015 + 0.005).half()
    valid_pq = torch.tensor([v for v in range(256) if all(((v >> (2 * i)) & 3) < 3 for i in range(4))],
                            dtype=torch.uint8, device=dev)
    rows = []
    for name, fmt, nbytes in (("PQ2_0", 1, 34), ("PTQ1_0", 2, 28)):
        blocks = torch.empty((nb, nbytes), dtype=torch.uint8, device=dev)
        blocks[:, 0:2] = sc.view(torch.uint8).view(nb, 2)
        if fmt == 1:
            idx = torch.randint(0, 81, (nb, 32), generator=g, device=dev)
            blocks[:, 2:] = valid_pq[idx]
        else:
            blocks[:, 2:27] = torch.randint(0, 243, (nb, 25), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
            blocks[:, 27] = torch.randint(0, 27, (nb,), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
        w = torch.empty((V, D // 16), dtype=torch.int32, device=dev)
        s_ = torch.empty((V, D // 128), dtype=torch.float16, device=dev)
        b_ = torch.empty((V, D // 128), dtype=torch.float16, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        for _ in range(3):
            tb.tb_transcode_gguf(blocks, fmt, V, D, w, s_, b_, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        reps = max(3, args.steps)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            tb.tb_transcode_gguf(blocks, fmt, V, D, w, s_, b_, st)
        b.record()
        torch.cuda.synchronize()
        per = a.elapsed_time(b) / 1e3 / reps
        byts = nb * (nbytes + 32 + 4)
        rows.append({"format": name, "us": round(per * 1e6, 1), "GB/s": round(byts / per / 1e9, 1),
                     "frac": round(byts / per / 1e9 / hbm, 4), "bytes": byts})
        del blocks, w, s_, b_
    return {"metric": "GGUF -> W2 transcode (tb_transcode_gguf), 248320 x 5120 table", "unit": "GB/s",
            "peak": hbm, "peak_kind": peak_kind, "l2": "inputs and outputs of 0.6-0.7 GB, far larger than L2",
            "rows": rows}


def run_embed(args, dist, tb, tdev, torch):
    hbm, _, _, peak_kind = peaks()
    dev = torch.device("cuda")
    tmp = torch.empty(1 << 30, dtype=torch.int8, device=dev)
    V, D, T = ti.VOCAB, ti.HIDDEN, 256
    p = Packed(tb, tdev, torch, ti.config_seed(5, 99), V, D, tmp)
    del tmp
    sg = torch.from_numpy(ti.rademacher_signs(5, D)).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    rows = []
    for r in range(max(3, args.steps)):
        ids = torch.from_numpy(ti.token_ids(100 + r, T, V)).to(dev)
        out = torch.empty((T, D), dtype=torch.float16, device=dev)
        flush = torch.empty(256 << 20, dtype=torch.int8, device=dev)
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        tb.tb_embed_lookup(ids, p.w, p.s, p.b, sg, 1024, out, status)
        b.record()
        torch.cuda.synchronize()
        rows.append(a.elapsed_time(b) / 1e3)
    per = float(np.median(rows[1:]))
    byts = T * (D // 4 + D // 64) + T * D * 2
    return {"metric": "embedding lookup 256 ids, 248320x5120 packed table", "us": round(per * 1e6, 2),
            "GB/s": round(byts / per / 1e9, 1), "peak": hbm, "peak_kind": peak_kind}


# ---------------------------------------------------------------------------- reference arm
def run_reference(args):
    """The float64 CPU oracle as the reference arm: bounded sample per step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle

    shapes = {}
    for _, K, N in ti.sweep_layers():
        shapes[(K, N)] = shapes.get((K, N), 0) + 1
    rows = 32

    emb_codes = ti.ternary_codes(12, 0, 16, ti.HIDDEN)
    emb_sc = ti.group_scales(12, 0, 16, ti.HIDDEN // 128)
    emb_w = oracle.pack_w2(emb_codes)
    emb_sg = ti.rademacher_signs(1, ti.HIDDEN)

    def one_step():
        t0 = time.perf_counter()
        oracle.embed_lookup(np.array([3]), emb_w, emb_sc, oracle.biases_for(emb_sc), emb_sg, 1024)
        sec = time.perf_counter() - t0
        for (K, N), count in sorted(shapes.items()):
            x = ti.activations(7, 1, K)
            sg = ti.rademacher_signs(7, K)
            codes = ti.ternary_codes(11, 0, rows, K)
            sc = ti.group_scales(11, 0, rows, K // 128)
            w = oracle.pack_w2(codes)
            t0 = time.perf_counter()
            oracle.packed_linear(x, sg, 1024, w, sc, oracle.biases_for(sc))
            sec += count * (time.perf_counter() - t0) * N / rows
        return sec

    for _ in range(args.warmup):
        one_step()
    w0 = time.perf_counter()
    t = [one_step() for _ in range(args.steps)]
    wall = (time.perf_counter() - w0) / args.steps
    sec = float(np.mean(t))
    v = 1.0 / sec
    return {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "extrapolated": True,
            "config": {"workload": "decode step, M=1: embedding of 1 id + 401 W2-g128 linears of the "
                                   "64-layer 27B stack (float64 CPU oracle, linears extrapolated from "
                                   "sampled rows)",
                       "ms_per_step": "extrapolated: the oracle runs on sampled rows of each distinct "
                                      "shape and its time is scaled by rows and by the shape's count; "
                                      "the wall time of one sampled step is in sample_wall_s"},
            "cpu_baseline": {"value": round(v, 6), "unit": "tok/s", "cores": len(os.sched_getaffinity(0)),
                             "kind": "oracle",
                             "sample": f"{rows} rows of each distinct shape per step, extrapolated"},
            "sample_wall_s": round(wall, 3),
            "e2e": {"value": round(v, 6), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="sweep", choices=["sweep", "layers", "prefill", "batched", "embed", "fwht", "transcode", "all"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub-results", action="store_true",
                    help="skip the per-link, batched, prefill and embedding numbers of the default line")
    ap.add_argument("--profile-step", action="store_true",
                    help="build the decode stack, run two steps and exit (for an ncu launch list)")
    ap.add_argument("--path", default="calls", choices=["chain", "calls"],
                    help="decode step path timed for `value` (the other one is reported in config)")
    ap.add_argument("--per-call", action="store_true",
                    help="with --profile-step: one launch per link instead of the chain launch")
    ap.add_argument("--profile-fwht", type=int, nargs=2, metavar=("M", "K"),
                    help="four tb_fwht calls on M x K activations (for ncu)")
    ap.add_argument("--profile-embed", action="store_true",
                    help="four embedding lookups of 256 ids on the 248320 x 5120 table (for ncu)")
    ap.add_argument("--profile-linear", type=int, nargs=4, metavar=("K", "N", "M", "ALGO"),
                    help="one packed K->N matrix, four tb_packed_linear calls on M tokens (for ncu)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if args.impl == "reference":
        line = run_reference(args)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = Dist("nccl")
    import ternary_hadamard_rotated_gb300 as tb
    from tb_inputs import device as tdev

    tb.load()
    configs = (["sweep", "layers", "prefill", "batched", "embed", "fwht", "transcode"] if args.config == "all"
               else [args.config])
    if args.profile_step:
        configs = ["profile"]
    if args.profile_linear:
        configs = ["profile_linear"]
    if args.profile_fwht:
        configs = ["profile_fwht"]
    if args.profile_embed:
        configs = ["profile_embed"]
    for c in configs:
        fn = {"sweep": run_sweep, "layers": run_layers, "prefill": run_prefill, "batched": run_batched,
              "embed": run_embed, "fwht": run_fwht, "transcode": run_transcode, "profile": profile_step,
              "profile_linear": profile_linear, "profile_embed": profile_embed,
              "profile_fwht": profile_fwht}[c]
        line = fn(args, dist, tb, tdev, torch)
        if rank == 0:
            print(json.dumps(line), flush=True)
        torch.cuda.empty_cache()
    dist.close()


if __name__ == "__main__":
    main()
