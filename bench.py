"""Benchmark of the quantized_matmul hot path on GB300.

One step = one pass of the decode workload over a batch of R independent
4-bit weights W_r [4096, 4096] (group 64), y_r = x . dequant(W_r)^T with
x [1, 4096] -- like R layers of a decode step.  R is chosen so the weights
span more than 3x the L2 cache, so every launch streams its weight from HBM.
The R launches are captured once in a CUDA graph and replayed; time is taken
with CUDA events on the launching stream.

`value` is the step's algorithmic bytes (packed codes + scales + biases + x +
y, per launch) over the step time, in GB/s.  `detail` carries the other
decode shapes (M in 1, 4, 8, 16 at 4 and 8 bits), the prefill GEMM in TFLOP/s
and the dequantize / rows throughputs, each measured the same way.

`--impl reference` times the CPU oracle (plain C, all host cores) on a bounded
sample of the same workload: this is the only reference there is, since the
pages publish no implementation that runs here.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized_matmul GB/s (M=1) and TFLOP/s (M=2048), % of HBM / bf16 TC roofline"
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["source"] = "fallback"
    return d


def max_over_ranks(value, dist=None, device="cpu"):
    """The largest value over all ranks (the slowest rank's time)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank, world, max_seconds):
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return world * units_per_rank / max_seconds


def gemv_bytes(M, N, K, bits, group):
    """Algorithmic bytes of one launch: codes + scales + biases + x + y (bf16)."""
    return N * K * bits // 8 + 4 * N * (K // group) + 2 * M * K + 2 * M * N


# ------------------------------------------------------------------ clocks ---

class ClockSampler:
    """Samples SM clocks, power and throttle reasons with a read-only
    nvidia-smi query every 100 ms while the `with` block runs.  Entering waits
    (up to 5 s) for the first sample, so that even a short timed region is
    covered by the samples taken during its warm-up and itself."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.device = device
        self.proc = None
        self.samples = []

    def _target(self):
        """nvidia-smi's name for this process's device: its UUID when torch
        reports one (device indices differ when CUDA_VISIBLE_DEVICES is set)."""
        try:
            import torch
            u = str(torch.cuda.get_device_properties(self.device).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            return str(self.device)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8 and parts[0].replace(".", "").isdigit():
                self.samples.append(parts)

    def __enter__(self):
        import threading
        self.samples = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self._target(), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.samples and self.proc.poll() is None and time.time() - t0 < 5.0:
            time.sleep(0.02)
        return self

    def __exit__(self, *exc):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(p[0]) for p in self.samples if p[0].replace(".", "").isdigit()]
        mx = [float(p[1]) for p in self.samples if p[1].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for p in self.samples for n, v in zip(names, p[4:8]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.samples)}


# ------------------------------------------------------------------- GPU ----

class Case:
    """R rotating weights and one CUDA graph of R quantized_matmul launches."""

    def __init__(self, torch, qmm, synth, M, N, K, bits, group, transpose=True, seed=1,
                 min_bytes=3 * L2_BYTES, max_copies=64):
        self.torch, self.qmm = torch, qmm
        self.M, self.N, self.K, self.bits, self.group, self.transpose = M, N, K, bits, group, transpose
        rows, cols = (N, K) if transpose else (K, N)
        base = synth.quant_weight(seed, rows, cols, bits, group)
        per = base.nbytes
        self.R = int(max(1, min(max_copies, -(-min_bytes // per))))
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(
            {np.dtype(np.uint32): np.int32, np.dtype(np.uint16): np.int16}[a.dtype])).cuda()
        # Copies differ by a rotation of the random words, so no two are equal.
        self.w = []
        for r in range(self.R):
            self.w.append((dev(np.roll(base.packed, r, axis=0)), dev(np.roll(base.scales, r, axis=0)),
                           dev(np.roll(base.biases, r, axis=0))))
        self.x_host = synth.x_bf16(seed + 1000, M, K)
        self.x = torch.from_numpy(self.x_host.view(np.int16)).cuda()
        self.y = torch.empty((self.R, M, N), dtype=torch.int16, device="cuda")
        self.graph = None

    def launch_all(self):
        for r in range(self.R):
            pw, ps, pb = self.w[r]
            self.qmm.qmm_quantized_matmul(self.x, self.M, pw, ps, pb, self.N, self.K,
                                          int(self.transpose), self.group, self.bits, self.y[r],
                                          self.qmm.QMM_BF16)

    def capture(self):
        torch = self.torch
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.launch_all()                 # eager once (and warms the library)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.launch_all()
        torch.cuda.synchronize()

    def bytes_per_launch(self):
        return gemv_bytes(self.M, self.N, self.K, self.bits, self.group)

    def flops_per_launch(self):
        return 2 * self.M * self.N * self.K


def graph_of(torch, fn):
    """Run fn once eagerly on a side stream, then capture it in a CUDA graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def dequant_rows_detail(torch, qmm, synth, peaks, steps, warmup):
    """Standalone dequantize to bf16 and the rows gather, as GB/s of their
    algorithmic bytes (codes + scales + biases read, bf16 written, indices)."""
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(
        {np.dtype(np.uint32): np.int32, np.dtype(np.uint16): np.int16}[a.dtype])).cuda()
    out = {}
    N, K = 14336, 4096
    for bits in (4, 8):
        w = synth.quant_weight(40 + bits, N, K, bits, 64)
        # Rotating weights and outputs whose bytes together exceed 3x L2.
        R = max(2, -(-3 * L2_BYTES // (w.nbytes + 2 * N * K)))
        copies = [(dev(np.roll(w.packed, r, 0)), dev(np.roll(w.scales, r, 0)),
                   dev(np.roll(w.biases, r, 0))) for r in range(R)]
        o = torch.empty((R, N, K), dtype=torch.int16, device="cuda")
        def fn():
            for r in range(R):
                pw, ps, pb = copies[r]
                qmm.qmm_dequantize(pw, ps, pb, N, K, 64, bits, o[r], qmm.QMM_BF16)
        t = time_graph(torch, graph_of(torch, fn), steps, warmup) / R
        nbytes = w.nbytes + 2 * N * K
        out["dequantize_b%d_%dx%d_bf16" % (bits, N, K)] = {
            "us": round(t * 1e3, 2), "GB/s": round(nbytes / (t * 1e-3) / 1e9, 1),
            "frac_hbm": round(nbytes / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)}
        del copies, o
    # quantize: bf16 [N, K] read, packed codes + bf16 scales and biases written
    R = max(2, -(-3 * L2_BYTES // (2 * N * K + N * K + 4 * N * (K // 64))))
    wsrc = [dev(synth.x_bf16(45 + r, N, K)) for r in range(R)]
    for bits in (4, 8):
        p = torch.empty((R, N, K * bits // 32), dtype=torch.int32, device="cuda")
        sc = torch.empty((R, N, K // 64), dtype=torch.int16, device="cuda")
        bi = torch.empty_like(sc)

        def fn():
            for r in range(R):
                qmm.qmm_quantize(wsrc[r], N, K, 64, bits, p[r], sc[r], bi[r])
        t = time_graph(torch, graph_of(torch, fn), steps, warmup) / R
        nbytes = 2 * N * K + N * K * bits // 8 + 4 * N * (K // 64)
        out["quantize_b%d_%dx%d_bf16" % (bits, N, K)] = {
            "us": round(t * 1e3, 2), "GB/s": round(nbytes / (t * 1e-3) / 1e9, 1),
            "frac_hbm": round(nbytes / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)}
        del p, sc, bi
    del wsrc
    T, C = synth.ROWS_TABLE
    w = synth.quant_weight(2, T, C, 4, 64)
    pw, ps, pb = dev(w.packed), dev(w.scales), dev(w.biases)
    idxs = [dev(synth.indices(3 + r, synth.ROWS_GATHER, T)) for r in range(4)]
    o = torch.empty((4, synth.ROWS_GATHER, C), dtype=torch.int16, device="cuda")
    def fn():
        for r in range(4):
            qmm.qmm_rows(pw, ps, pb, T, C, idxs[r], synth.ROWS_GATHER, 64, 4, o[r], qmm.QMM_BF16)
    t = time_graph(torch, graph_of(torch, fn), steps, warmup) / 4
    row_bytes = C * 4 // 8 + 4 * (C // 64)
    nbytes = synth.ROWS_GATHER * (row_bytes + 2 * C + 4)
    out["rows_4096_of_%dx%d_b4_bf16" % (T, C)] = {
        "us": round(t * 1e3, 2), "GB/s": round(nbytes / (t * 1e-3) / 1e9, 1),
        "frac_hbm": round(nbytes / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)}
    return out


def sweep_detail(torch, qmm, synth, peaks, warmup):
    """The remaining workloads, one line each: odd widths at M=1, the prefill
    GEMM with W stored [K, N], the layer-shape sweep (GB/s and TFLOP/s, both
    against their measured peaks), and bf16 dequantize of each sweep weight."""
    out = {}

    def one(name, M, N, K, bits, group, transpose, seed):
        c = Case(torch, qmm, synth, M, N, K, bits, group, transpose=transpose, seed=seed)
        c.capture()
        steps = 200 if M <= 16 else 30 if M <= 128 else 4
        t = time_graph(torch, c.graph, steps, warmup) / c.R
        gbs = c.bytes_per_launch() / (t * 1e-3) / 1e9
        tf = c.flops_per_launch() / (t * 1e-3) / 1e12
        out[name] = {"us": round(t * 1e3, 3), "GB/s": round(gbs, 1),
                     "frac_hbm": round(gbs / peaks["hbm_gbs"], 3), "TFLOP/s": round(tf, 2),
                     "frac_bf16": round(tf / peaks["bf16_tflops"], 4)}
        del c
        torch.cuda.empty_cache()

    N, K = synth.ODD_SHAPE
    for bits in synth.ODD_BITS:
        for g in synth.ODD_GROUPS:
            one("odd_b%d_g%d_%dx%d_M1" % (bits, g, N, K), 1, N, K, bits, g, True, 60 + bits + g)
    p = synth.PREFILL
    one("prefill_b4_M2048_w_stored_KxN", p["M"], p["N"], p["K"], 4, 64, False, 31)
    for (N, K) in synth.SWEEP_SHAPES:
        for bits in (4, 8):
            for M in synth.SWEEP_M:
                one("sweep_b%d_%dx%d_M%d" % (bits, N, K, M), M, N, K, bits, 64, True, 70 + M + bits)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(
        {np.dtype(np.uint32): np.int32, np.dtype(np.uint16): np.int16}[a.dtype])).cuda()
    for (N, K) in synth.SWEEP_SHAPES:
        for bits in (4, 8):
            w = synth.quant_weight(90 + bits, N, K, bits, 64)
            # Rotate weights and outputs whose bytes together exceed 3x L2.
            R = max(2, -(-3 * L2_BYTES // (w.nbytes + 2 * N * K)))
            copies = [(dev(np.roll(w.packed, r, 0)), dev(np.roll(w.scales, r, 0)),
                       dev(np.roll(w.biases, r, 0))) for r in range(R)]
            o = torch.empty((R, N, K), dtype=torch.int16, device="cuda")

            def fn():
                for r in range(R):
                    pw, ps, pb = copies[r]
                    qmm.qmm_dequantize(pw, ps, pb, N, K, 64, bits, o[r], qmm.QMM_BF16)
            t = time_graph(torch, graph_of(torch, fn), 20, warmup) / R
            nbytes = w.nbytes + 2 * N * K
            out["sweep_dequantize_b%d_%dx%d_bf16" % (bits, N, K)] = {
                "us": round(t * 1e3, 2), "GB/s": round(nbytes / (t * 1e-3) / 1e9, 1),
                "frac_hbm": round(nbytes / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)}
            del copies, o
            torch.cuda.empty_cache()
    return out


def gather_detail(torch, qmm, synth, peaks, warmup):
    """Mixture-of-experts decode through gather_qmm: 8 experts [14336, 4096]
    4-bit g64, 32 routed token slots (16 tokens x top 2, one x row each),
    indices drawn once (seeded).  GB/s counts the bytes of the experts used
    (each read once) plus x and y; sorted = the slots grouped by expert.  Then
    the prefill form: 4096 sorted slots on the same experts."""
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(
        {np.dtype(np.uint32): np.int32, np.dtype(np.uint16): np.int16}[a.dtype])).cuda()
    E, N, K, B = 8, 14336, 4096, 32
    ws = [synth.quant_weight(120 + e, N, K, 4, 64) for e in range(E)]
    packed = dev(np.stack([w.packed for w in ws]))
    sc = dev(np.stack([w.scales for w in ws]))
    bi = dev(np.stack([w.biases for w in ws]))
    rhs_host = synth.indices(121, B, E)
    used = len(set(rhs_host.tolist()))
    nbytes = used * ws[0].nbytes + B * K * 2 + B * N * 2
    x = dev(synth.x_bf16(122, B, K))
    y = torch.empty((B, 1, N), dtype=torch.int16, device="cuda")
    out = {}
    for name, rhs, sorted_ in (("sorted", np.sort(rhs_host), 1), ("unsorted", rhs_host, 0)):
        r = dev(rhs.astype(np.uint32))

        def fn():
            qmm.qmm_gather_qmm(x, B, 1, packed, sc, bi, E, N, K, None, r, B, 1, 64, 4, sorted_,
                               y, qmm.QMM_BF16)
        t = time_graph(torch, graph_of(torch, fn), 100, warmup)
        out["gather_qmm_moe_8x%dx%d_b4_32slots_%s" % (N, K, name)] = {
            "us": round(t * 1e3, 2), "experts_used": used, "GB/s": round(nbytes / (t * 1e-3) / 1e9, 1),
            "frac_hbm": round(nbytes / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)}
    # Prefill: 2048 tokens x top 2 = 4096 sorted slots (the grouped tensor-core
    # path); TFLOP/s = 2 * slots * N * K.
    B = 4096
    rhs = dev(np.sort(synth.indices(123, B, E)).astype(np.uint32))
    x = dev(synth.x_bf16(124, B, K))
    y = torch.empty((B, 1, N), dtype=torch.int16, device="cuda")

    def prefill():
        qmm.qmm_gather_qmm(x, B, 1, packed, sc, bi, E, N, K, None, rhs, B, 1, 64, 4, 1, y,
                           qmm.QMM_BF16)
    t = time_graph(torch, graph_of(torch, prefill), 10, warmup)
    tf = 2.0 * B * N * K / (t * 1e-3) / 1e12
    out["gather_qmm_moe_prefill_8x%dx%d_b4_%dslots_sorted" % (N, K, B)] = {
        "us": round(t * 1e3, 1), "TFLOP/s": round(tf, 1), "frac_bf16": round(tf / peaks["bf16_tflops"], 4)}
    del packed, sc, bi, x, y
    torch.cuda.empty_cache()
    return out


def fused_detail(torch, qmm, synth, peaks, warmup):
    """The fused decode GEMVs of an 8B-class gated feed-forward block at M=1,
    4-bit g64, each against the unfused calls it replaces: gate_up (two
    [14336, 4096] weights, one x) and silu_gate with the residual (down
    projection [4096, 14336]).  GB/s counts weights + inputs + outputs; rotating
    weight copies keep every launch on HBM; programmatic dependent launch on."""
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(
        {np.dtype(np.uint32): np.int32, np.dtype(np.uint16): np.int16}[a.dtype])).cuda()
    out = {}
    flags = qmm.qmm_set_launch_flags(qmm.QMM_LAUNCH_PDL)
    N, K = 14336, 4096
    base_g, base_u = synth.quant_weight(130, N, K, 4, 64), synth.quant_weight(131, N, K, 4, 64)
    R = max(2, -(-3 * L2_BYTES // (2 * base_g.nbytes)))
    ws = [tuple(dev(np.roll(a, r, 0)) for w in (base_g, base_u) for a in (w.packed, w.scales, w.biases))
          for r in range(R)]
    x = dev(synth.x_bf16(132, 1, K))
    yg = torch.empty((R, 1, N), dtype=torch.int16, device="cuda")
    yu = torch.empty_like(yg)
    nbytes = 2 * base_g.nbytes + 2 * K + 4 * N

    def fused():
        for r in range(R):
            qmm.qmm_gemv_gate_up(x, 1, *ws[r], N, K, 64, 4, yg[r], yu[r], qmm.QMM_BF16)

    def unfused():
        for r in range(R):
            pg, sg, bg, pu, su, bu = ws[r]
            qmm.qmm_quantized_matmul(x, 1, pg, sg, bg, N, K, 1, 64, 4, yg[r], qmm.QMM_BF16)
            qmm.qmm_quantized_matmul(x, 1, pu, su, bu, N, K, 1, 64, 4, yu[r], qmm.QMM_BF16)
    for name, fn in (("gemv_gate_up_2x%dx%d_b4_M1" % (N, K), fused),
                     ("gemv_gate_up_unfused_2x%dx%d_b4_M1" % (N, K), unfused)):
        t = time_graph(torch, graph_of(torch, fn), 200, warmup) / R
        out[name] = {"us": round(t * 1e3, 2), "GB/s": round(nbytes / (t * 1e-3) / 1e9, 1),
                     "frac_hbm": round(nbytes / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)}
    del ws, yg, yu
    N, K = 4096, 14336
    base = synth.quant_weight(133, N, K, 4, 64)
    R = max(2, -(-3 * L2_BYTES // base.nbytes))
    ws = [tuple(dev(np.roll(a, r, 0)) for a in (base.packed, base.scales, base.biases)) for r in range(R)]
    gate, up = dev(synth.x_bf16(134, 1, K)), dev(synth.x_bf16(135, 1, K))
    resid = dev(synth.x_bf16(136, 1, N))
    y = torch.empty((R, 1, N), dtype=torch.int16, device="cuda")
    nbytes = base.nbytes + 4 * K + 4 * N

    def fused_silu():
        for r in range(R):
            qmm.qmm_gemv_silu_gate(gate, up, 1, *ws[r], N, K, 64, 4, resid, y[r], qmm.QMM_BF16)
    # The calls it replaces: x = RN_bf16(silu(gate) * up) and y + resid as
    # PyTorch elementwise kernels around the plain GEMV (bf16 in and out).
    gb, ub = gate.view(torch.bfloat16), up.view(torch.bfloat16)
    rb = resid.view(torch.bfloat16)
    xs = torch.empty((1, K), dtype=torch.bfloat16, device="cuda")
    yt = torch.empty((R, 1, N), dtype=torch.int16, device="cuda")

    def unfused_silu():
        for r in range(R):
            torch.mul(torch.nn.functional.silu(gb.float()), ub.float(), out=xs)
            qmm.qmm_quantized_matmul(xs.view(torch.int16), 1, *ws[r], N, K, 1, 64, 4, yt[r], qmm.QMM_BF16)
            y[r].view(torch.bfloat16).copy_(yt[r].view(torch.bfloat16) + rb)
    for name, fn in (("gemv_silu_gate_resid_%dx%d_b4_M1" % (N, K), fused_silu),
                     ("gemv_silu_gate_resid_unfused_%dx%d_b4_M1" % (N, K), unfused_silu)):
        t = time_graph(torch, graph_of(torch, fn), 200, warmup) / R
        out[name] = {"us": round(t * 1e3, 2), "GB/s": round(nbytes / (t * 1e-3) / 1e9, 1),
                     "frac_hbm": round(nbytes / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)}
    qmm.qmm_set_launch_flags(flags)
    del ws, y, yt
    torch.cuda.empty_cache()
    return out


def dtype_detail(torch, qmm, synth, peaks, warmup):
    """quantized_matmul in the other compute types at 4 bits, group 64: fp16
    (fp16 x, scales and biases: the tensor-core kernels in fp16) and fp32 (fp32
    x, scales and biases: the CUDA-core path), at the decode shapes (W [4096,
    4096], M = 1 and 16) and the prefill shape (x [2048, 4096], W [14336,
    4096]).  GB/s counts codes, scales, biases, x and y in their own types;
    TFLOP/s is 2 M N K.  Decode lines rotate weight copies above L2."""
    out = {}
    flags = qmm.qmm_set_launch_flags(qmm.QMM_LAUNCH_PDL)
    Q = {"f16": qmm.QMM_F16, "f32": qmm.QMM_F32}
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(
        {np.dtype(np.uint32): np.int32, np.dtype(np.uint16): np.int16,
         np.dtype(np.float32): np.float32}[a.dtype])).cuda()
    for d in ("f16", "f32"):
        esz = 2 if d == "f16" else 4
        for (M, N, K) in ((1, 4096, 4096), (16, 4096, 4096), (2048, 14336, 4096)):
            w = synth.quant_weight_typed(140 + M, N, K, 4, 64, d)
            nw = w.packed.nbytes + w.scales.nbytes + w.biases.nbytes
            R = max(2, -(-3 * L2_BYTES // nw)) if M <= 16 else 2
            ws = [tuple(dev(np.roll(a, r, 0)) for a in (w.packed, w.scales, w.biases))
                  for r in range(R)]
            x = dev(synth.x_typed(141 + M, M, K, d))
            y = torch.empty((R, M, N), dtype=torch.float32 if d == "f32" else torch.int16,
                            device="cuda")

            def fn():
                for r in range(R):
                    pw, ps, pb = ws[r]
                    qmm.qmm_quantized_matmul_typed(x, Q[d], M, pw, ps, pb, Q[d], N, K, 1, 64, 4,
                                                   y[r], Q[d])
            steps = 200 if M <= 16 else (6 if d == "f16" else 2)
            t = time_graph(torch, graph_of(torch, fn), steps, min(warmup, 3)) / R
            nbytes = nw + esz * (M * K + M * N)
            gbs = nbytes / (t * 1e-3) / 1e9
            tf = 2.0 * M * N * K / (t * 1e-3) / 1e12
            out["%s_b4_%dx%d_M%d" % (d, N, K, M)] = {
                "us": round(t * 1e3, 2), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 3),
                "TFLOP/s": round(tf, 2), "frac_bf16": round(tf / peaks["bf16_tflops"], 4)}
            del ws, y
            torch.cuda.empty_cache()
    qmm.qmm_set_launch_flags(flags)
    return out


def measured_traffic():
    """DRAM bytes per launch of the decode kernel from the committed ncu capture,
    or None if the kernel source changed since it was taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "decode_gemv_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    return d.get("dram_bytes_per_launch") if d.get("sources_sha256") == decode_sources_sha() else None


def decode_sources_sha():
    """sha256 over the decode kernel's device code (the kernel templates, then
    the device helpers they include); host launch code is not part of it."""
    import hashlib
    h = hashlib.sha256()
    for name in ("gemv_impl.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "mlx_grouped_affine_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def time_graph(torch, graph, steps, warmup, barrier=None):
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        graph.replay()
    end.record()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return start.elapsed_time(end) / steps  # ms per step


def run_gpu(args):
    import torch
    from mlx_grouped_affine_gb300 import qmm, synth

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    barrier = (lambda: dist.barrier()) if dist else None
    peaks = load_peaks()
    qmm.lib()

    N, K = synth.DECODE_SHAPE
    # Decode launches go out with programmatic dependent launch (each GEMV
    # starts streaming its weights while the previous kernel finishes), the
    # way a serving loop would run them.
    qmm.qmm_set_launch_flags(0 if args.no_pdl else qmm.QMM_LAUNCH_PDL)
    head = Case(torch, qmm, synth, 1, N, K, 4, 64, seed=1 + rank)
    head.capture()
    with ClockSampler(local) as clk:
        # Keep the GPU under this load for half a second before the timed
        # region (extra warm-up), so the clock samples describe it.
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 0.5:
            for _ in range(50):
                head.graph.replay()
            torch.cuda.synchronize()
        ms = time_graph(torch, head.graph, args.steps, args.warmup, barrier)
    clocks = clk.summary()
    clocks["window"] = "0.5 s of the step's replays before the timed region, and the timed region"

    ms = max_over_ranks(ms, dist, device="cuda")
    launch_ms = ms / head.R
    per_launch = head.bytes_per_launch()
    value = job_value(head.R * per_launch, world, ms * 1e-3) / 1e9
    achieved = per_launch / (launch_ms * 1e-3) / 1e9

    # End to end through the public API with host buffers: per step, x for the
    # R launches comes from pinned host memory and y goes back to it.
    x_pin = torch.from_numpy(np.repeat(head.x_host.view(np.int16)[None], head.R, 0)).pin_memory()
    y_pin = torch.empty((head.R, 1, N), dtype=torch.int16).pin_memory()
    x_dev = torch.empty_like(x_pin, device="cuda")
    # A serving loop keeps its buffers' device addresses and its stream handle;
    # the binding takes them as integers.
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    calls = [(x_dev[r].data_ptr(), head.w[r][0].data_ptr(), head.w[r][1].data_ptr(),
              head.w[r][2].data_ptr(), head.y[r].data_ptr()) for r in range(head.R)]

    def e2e_step():
        x_dev.copy_(x_pin, non_blocking=True)
        for px, pw, ps, pb, py in calls:
            qmm.qmm_quantized_matmul(px, 1, pw, ps, pb, N, K, 1, 64, 4, py, qmm.QMM_BF16, sh)
        y_pin.copy_(head.y, non_blocking=True)
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e_steps = max(10, min(args.steps, 200))
    t0 = time.perf_counter()
    for _ in range(e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / e_steps
    e2e = {"value": world * head.R * per_launch / e2e_s / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": int(x_pin.numel() * 2), "d2h_bytes_per_step": int(y_pin.numel() * 2)}

    detail = {}
    if rank == 0:
        detail.update(reference_case_detail(torch, qmm, synth, peaks, args.warmup))
        flags = qmm.qmm_set_launch_flags(0)
        c = Case(torch, qmm, synth, 1, N, K, 4, 64, seed=2)
        c.capture()
        t = time_graph(torch, c.graph, max(20, args.steps // 4), args.warmup) / c.R
        detail["decode_b4_M1_without_pdl"] = {
            "us": round(t * 1e3, 3), "GB/s": round(c.bytes_per_launch() / (t * 1e-3) / 1e9, 1)}
        del c
        qmm.qmm_set_launch_flags(flags)
        p = synth.PREFILL
        c = Case(torch, qmm, synth, p["M"], p["N"], p["K"], 4, 64, seed=30)
        c.capture()
        t = time_graph(torch, c.graph, max(5, args.steps // 200), args.warmup) / c.R
        tf = c.flops_per_launch() / (t * 1e-3) / 1e12
        detail["prefill_b4_M2048"] = {
            "us": round(t * 1e3, 2), "TFLOP/s": round(tf, 1),
            "frac_bf16": round(tf / peaks["bf16_tflops"], 4),
            "launches_timed": c.R * max(5, args.steps // 200)}
        del c
        torch.cuda.empty_cache()
    if rank == 0 and not args.quick:
        detail.update(dequant_rows_detail(torch, qmm, synth, peaks, max(20, args.steps // 50),
                                          args.warmup))
        torch.cuda.empty_cache()
        for bits in (4, 8):
            for M in synth.DECODE_M:
                c = Case(torch, qmm, synth, M, N, K, bits, 64, seed=10 + bits + M)
                c.capture()
                t = time_graph(torch, c.graph, max(20, args.steps // 4), args.warmup) / c.R
                detail["decode_b%d_M%d" % (bits, M)] = {
                    "us": round(t * 1e3, 3), "GB/s": round(c.bytes_per_launch() / (t * 1e-3) / 1e9, 1),
                    "frac_hbm": round(c.bytes_per_launch() / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)}
                del c
                torch.cuda.empty_cache()
        detail.update(sweep_detail(torch, qmm, synth, peaks, args.warmup))
        detail.update(gather_detail(torch, qmm, synth, peaks, args.warmup))
        detail.update(fused_detail(torch, qmm, synth, peaks, args.warmup))
        detail.update(dtype_detail(torch, qmm, synth, peaks, args.warmup))

    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(budget_s=args.cpu_seconds)
        one = cpu_baseline(budget_s=min(5.0, args.cpu_seconds), threads=1)
        detail["cpu_oracle_1thread"] = {"GB/s": one["value"], "sample": one["sample"]}
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u4->bf16",
        "data": "synthetic (seeded uniform codes, bf16 scales/biases, N(0,1) x)",
        "config": {"workload": "decode GEMV x[1,4096] . W[4096,4096]^T, 4-bit, group 64, bf16 out",
                   "launches_per_step": head.R, "weight_copies_bytes": head.R * per_launch,
                   "l2": "inputs larger than L2: %d rotating weight copies (> 3x L2)" % head.R,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "launch": "CUDA graph of the step's launches; decode kernels with "
                             + ("stream-ordered launch" if args.no_pdl else
                                "programmatic dependent launch")},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": measured_traffic(), "peak_source": peaks["source"]},
        "clocks": clocks, "e2e": e2e, "gpu_launches": args.steps * head.R,
        "detail": detail,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu
    # The headline lines again, last, so that they survive a tail of the line.
    out["headline"] = headline(detail, out)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return out if rank == 0 else None


def headline(detail, out):
    """A compact summary of the lines that carry the metric: decode (GB/s and
    fraction of HBM), the M = 2048 prefill (TFLOP/s and fraction of bf16
    peak), odd widths, rows, dequantize, the fused GEMVs against their unfused
    calls and the 4-bit M = 128 lines."""
    h = {"decode_b4_M1_4096x4096": {"GB/s": out["value"], "frac_hbm": out["roofline"]["frac"]}}
    for k, v in detail.items():
        if k.startswith("prefill_b4_M2048"):
            h[k] = {"us": v.get("us"), "TFLOP/s": v.get("TFLOP/s"), "frac_bf16": v.get("frac_bf16")}
        elif k.startswith(("decode_b", "odd_", "rows_", "dequantize_", "reference_case", "gemv_")):
            h[k] = {kk: v[kk] for kk in ("us", "frac_hbm") if kk in v}
        elif k.startswith("sweep_b4_") and k.endswith("_M128"):
            h[k] = {kk: v[kk] for kk in ("us", "frac_bf16") if kk in v}
    h["clocks_sm_mhz"] = out["clocks"].get("sm_mhz")
    return h


def reference_case_detail(torch, qmm, synth, peaks, warmup):
    """The small reference case: x [1, 512] . W[256, 512]^T at 4 bits, group
    64, fp32 out, and the fp32 dequantize of W.  Both are latency-bound (76 KB
    and 0.6 MB); the line reports time per launch in a CUDA graph of 64
    launches (inputs L2-resident: the workload is smaller than L2) and the
    algorithmic bytes over that time."""
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(
        {np.dtype(np.uint32): np.int32, np.dtype(np.uint16): np.int16}[a.dtype])).cuda()
    w = synth.pr1_weight(0)
    pw, ps, pb = dev(w.packed), dev(w.scales), dev(w.biases)
    x = dev(synth.x_bf16(0, 1, 512))
    y = torch.empty((1, 256), dtype=torch.float32, device="cuda")
    o = torch.empty((256, 512), dtype=torch.float32, device="cuda")
    out = {}
    n = 64

    def mm():
        for _ in range(n):
            qmm.qmm_quantized_matmul(x, 1, pw, ps, pb, 256, 512, 1, 64, 4, y, qmm.QMM_F32)

    def dq():
        for _ in range(n):
            qmm.qmm_dequantize(pw, ps, pb, 256, 512, 64, 4, o, qmm.QMM_F32)
    for name, fn, nbytes in (("reference_case_qmm_1x512_256x512_b4_f32", mm,
                              w.nbytes + 2 * 512 + 4 * 256),
                             ("reference_case_dequantize_256x512_b4_f32", dq, w.nbytes + 4 * 256 * 512)):
        t = time_graph(torch, graph_of(torch, fn), 50, warmup) / n
        out[name] = {"us": round(t * 1e3, 3), "GB/s": round(nbytes / (t * 1e-3) / 1e9, 1),
                     "frac_hbm": round(nbytes / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
    return out


# ------------------------------------------------------------------- CPU ----

def cpu_baseline(budget_s=15.0, steps=None, threads=None):
    """The oracle, as it stands, on all host cores (or `threads` of them):
    whole problems of the headline workload (x [1, 4096] . W[4096, 4096]^T at
    4 bits), repeated until about `budget_s` seconds have passed."""
    import oracle
    from mlx_grouped_affine_gb300 import synth
    N, K = synth.DECODE_SHAPE
    w = synth.quant_weight(1, N, K, 4, 64)
    x = synth.x_bf16(1001, 1, K)
    threads = threads or oracle.default_threads()
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.qmm(x, 1, w.packed, w.scales, w.biases, N, K, True, 64, 4, nthreads=threads)
        done += 1
        el = time.perf_counter() - t0
        if (steps and done >= steps) or (not steps and el >= budget_s):
            break
    gbs = done * gemv_bytes(1, N, K, 4, 64) / el / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "%d full problems x[1,4096].W[4096,4096]^T 4-bit g64 in %.1f s" % (done, el)}


def run_reference(args):
    """The reference arm: the CPU oracle, timed per step on a bounded sample."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle
    from mlx_grouped_affine_gb300 import synth
    N, K = synth.DECODE_SHAPE
    w = synth.quant_weight(1, N, K, 4, 64)
    x = synth.x_bf16(1001, 1, K)
    threads = oracle.default_threads()
    # Size a step (a slice of output columns) so that warmup + steps take
    # about two minutes in all.
    probe_rows = 256
    t0 = time.perf_counter()
    oracle.qmm(x, 1, w.packed[:probe_rows], w.scales[:probe_rows], w.biases[:probe_rows],
               probe_rows, K, True, 64, 4, nthreads=threads)
    per_row = (time.perf_counter() - t0) / probe_rows
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    rows = int(max(16, min(N, budget / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        oracle.qmm(x, 1, w.packed[:rows], w.scales[:rows], w.biases[:rows], rows, K, True, 64, 4,
                   nthreads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.qmm(x, 1, w.packed[:rows], w.scales[:rows], w.biases[:rows], rows, K, True, 64, 4,
                   nthreads=threads)
    el = time.perf_counter() - t0
    step_bytes = gemv_bytes(1, rows, K, 4, 64)
    value = args.steps * step_bytes / el / 1e9
    sample = "first %d of 4096 weight rows per step (x[1,4096], 4-bit, group 64)" % rows
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": "decode GEMV x[1,4096] . W[4096,4096]^T, "
                                            "4-bit, group 64 (CPU oracle sample)"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


PROFILE_CASES = {
    # name: (M, N, K, bits, group, transpose)
    "decode": (1, 4096, 4096, 4, 64, True),
    "decode_m16": (16, 4096, 4096, 4, 64, True),
    "decode_b8": (1, 4096, 4096, 8, 64, True),
    "prefill": (2048, 14336, 4096, 4, 64, True),
    "splitk_m128": (128, 4096, 4096, 4, 64, True),
    "splitk_m128_k14336": (128, 4096, 14336, 4, 64, True),
    "prefill_nt": (2048, 14336, 4096, 4, 64, False),
    "decode_b2_many_tiles": (1, 11008, 4096, 2, 32, True),
    "decode_many_tiles": (1, 14336, 4096, 4, 64, True),
}
OTHER_PROFILES = ("gather_sorted", "silu_gate", "quantize", "dequantize", "rows", "f16_prefill",
                  "f16_decode", "f32_decode", "f32_decode16", "f32_prefill", "gather_prefill",
                  "odd_widths")


def run_other_profile(case, launches):
    """Eager launches, for ncu, of the entry points and dtypes the matmul cases
    above do not cover (inputs larger than L2)."""
    import torch
    from mlx_grouped_affine_gb300 import qmm, synth
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(
        {np.dtype(np.uint32): np.int32, np.dtype(np.uint16): np.int16}[a.dtype])).cuda()
    if case == "gather_sorted":
        E, N, K, B = 8, 14336, 4096, 32
        ws = [synth.quant_weight(120 + e, N, K, 4, 64) for e in range(E)]
        packed = dev(np.stack([w.packed for w in ws]))
        sc, bi = dev(np.stack([w.scales for w in ws])), dev(np.stack([w.biases for w in ws]))
        rhs = dev(np.sort(synth.indices(121, B, E)).astype(np.uint32))
        x = dev(synth.x_bf16(122, B, K))
        y = torch.empty((B, 1, N), dtype=torch.int16, device="cuda")
        for _ in range(launches):
            qmm.qmm_gather_qmm(x, B, 1, packed, sc, bi, E, N, K, None, rhs, B, 1, 64, 4, 1, y,
                               qmm.QMM_BF16)
    elif case == "gather_prefill":
        E, N, K, B = 8, 14336, 4096, 4096
        ws = [synth.quant_weight(120 + e, N, K, 4, 64) for e in range(E)]
        packed = dev(np.stack([w.packed for w in ws]))
        sc, bi = dev(np.stack([w.scales for w in ws])), dev(np.stack([w.biases for w in ws]))
        rhs = dev(np.sort(synth.indices(123, B, E)).astype(np.uint32))
        x = dev(synth.x_bf16(124, B, K))
        y = torch.empty((B, 1, N), dtype=torch.int16, device="cuda")
        for _ in range(launches):
            qmm.qmm_gather_qmm(x, B, 1, packed, sc, bi, E, N, K, None, rhs, B, 1, 64, 4, 1, y,
                               qmm.QMM_BF16)
    elif case == "silu_gate":
        N, K, R = 4096, 14336, 6
        base = synth.quant_weight(133, N, K, 4, 64)
        ws = [tuple(dev(np.roll(a, r, 0)) for a in (base.packed, base.scales, base.biases))
              for r in range(R)]
        gate, up = dev(synth.x_bf16(134, 1, K)), dev(synth.x_bf16(135, 1, K))
        resid = dev(synth.x_bf16(136, 1, N))
        y = torch.empty((1, N), dtype=torch.int16, device="cuda")
        for i in range(launches):
            qmm.qmm_gemv_silu_gate(gate, up, 1, *ws[i % R], N, K, 64, 4, resid, y, qmm.QMM_BF16)
    elif case == "quantize":
        N, K, R = 14336, 4096, 2
        src = [dev(synth.x_bf16(45 + r, N, K)) for r in range(R)]
        p = torch.empty((N, K // 8), dtype=torch.int32, device="cuda")
        sc = torch.empty((N, K // 64), dtype=torch.int16, device="cuda")
        bi = torch.empty_like(sc)
        for i in range(launches):
            qmm.qmm_quantize(src[i % R], N, K, 64, 4, p, sc, bi)
    elif case == "dequantize":
        N, K, R = 14336, 4096, 2
        w = synth.quant_weight(44, N, K, 4, 64)
        cs = [tuple(dev(np.roll(a, r, 0)) for a in (w.packed, w.scales, w.biases)) for r in range(R)]
        o = torch.empty((N, K), dtype=torch.int16, device="cuda")
        for i in range(launches):
            qmm.qmm_dequantize(*cs[i % R], N, K, 64, 4, o, qmm.QMM_BF16)
    elif case in ("f16_prefill", "f16_decode", "f32_decode", "f32_decode16", "f32_prefill"):
        d = case[:3]
        Q = {"f16": qmm.QMM_F16, "f32": qmm.QMM_F32}[d]
        M, N, K = ((2048, 14336, 4096) if case.endswith("prefill") else
                   (16, 4096, 4096) if case.endswith("16") else (1, 4096, 4096))
        w = synth.quant_weight_typed(150, N, K, 4, 64, d)
        nw = w.packed.nbytes + w.scales.nbytes + w.biases.nbytes
        R = max(2, -(-3 * L2_BYTES // nw)) if M <= 16 else 2
        tdev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(
            {np.dtype(np.uint32): np.int32, np.dtype(np.uint16): np.int16,
             np.dtype(np.float32): np.float32}[a.dtype])).cuda()
        ws = [tuple(tdev(np.roll(a, r, 0)) for a in (w.packed, w.scales, w.biases)) for r in range(R)]
        x = tdev(synth.x_typed(151, M, K, d))
        y = torch.empty((M, N), dtype=torch.float32 if d == "f32" else torch.int16, device="cuda")
        for i in range(launches):
            qmm.qmm_quantized_matmul_typed(x, Q, M, *ws[i % R], Q, N, K, 1, 64, 4, y, Q)
    elif case == "odd_widths":
        # The odd-width decode lines at M = 1, each width `launches` times in
        # turn over two weight copies (> L2 together at every width).
        N, K = synth.ODD_SHAPE
        x = dev(synth.x_bf16(61, 1, K))
        y = torch.empty((1, N), dtype=torch.int16, device="cuda")
        for bits in synth.ODD_BITS:
            for g in synth.ODD_GROUPS:
                w = synth.quant_weight(60 + bits + g, N, K, bits, g)
                R = max(2, -(-int(1.5 * L2_BYTES) // w.nbytes))
                ws = [tuple(dev(np.roll(a, r, 0)) for a in (w.packed, w.scales, w.biases)) for r in range(R)]
                for i in range(launches):
                    qmm.qmm_quantized_matmul(x, 1, *ws[i % R], N, K, 1, g, bits, y, qmm.QMM_BF16)
                del ws
    elif case == "rows":
        T, C = synth.ROWS_TABLE
        w = synth.quant_weight(2, T, C, 4, 64)
        pw, ps, pb = dev(w.packed), dev(w.scales), dev(w.biases)
        idx = dev(synth.indices(3, synth.ROWS_GATHER, T))
        o = torch.empty((synth.ROWS_GATHER, C), dtype=torch.int16, device="cuda")
        for _ in range(launches):
            qmm.qmm_rows(pw, ps, pb, T, C, idx, synth.ROWS_GATHER, 64, 4, o, qmm.QMM_BF16)
    torch.cuda.synchronize()
    print(json.dumps({"profile": case, "launches": launches}))


def run_profile(case, launches):
    """A few eager launches of one case over rotating weights (inputs > L2),
    for ncu: a small, fixed amount of device memory and no CUDA graph."""
    import torch
    from mlx_grouped_affine_gb300 import qmm, synth
    M, N, K, bits, group, transpose = PROFILE_CASES[case]
    c = Case(torch, qmm, synth, M, N, K, bits, group, transpose, seed=5,
             min_bytes=int(1.5 * L2_BYTES), max_copies=16)
    for i in range(launches):
        r = i % c.R
        pw, ps, pb = c.w[r]
        qmm.qmm_quantized_matmul(c.x, M, pw, ps, pb, N, K, int(transpose), group, bits, c.y[r],
                                 qmm.QMM_BF16)
    torch.cuda.synchronize()
    print(json.dumps({"profile": case, "launches": launches, "copies": c.R}))


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--profile", choices=sorted(PROFILE_CASES) + sorted(OTHER_PROFILES),
                   help="run a few eager launches of one case (for ncu) and exit")
    p.add_argument("--launches", type=int, default=6)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=("ours", "reference"))
    p.add_argument("--quick", action="store_true", help="headline case only")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-pdl", action="store_true", help="launch decode kernels without PDL")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--ref-seconds", type=float, default=120.0,
                   help="total CPU time budget of the reference arm")
    args = p.parse_args()
    if args.profile:
        if args.profile in OTHER_PROFILES:
            run_other_profile(args.profile, args.launches)
        else:
            run_profile(args.profile, args.launches)
        return
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    out = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
