"""Benchmark of the block-scaled 4-bit hot path on GB300.

Default workload: the W4A16 decode GEMM, N = K = 8192 INT4 g128 weights, bf16
activations at M = 1, 4 and 16.  One step runs the three decode GEMMs, each on
its own copy of the weights (8 rotating copies, 277 MB > L2, so every launch
streams its weights from HBM).  ``value`` is algorithmic HBM bytes per second
over the timed steps, with all inputs resident in HBM; ``e2e`` is the same
metric through the public Python API with the activations copied in from
pinned host memory and the outputs copied back every step.

Other workloads (``--workload``): ``decode_nvfp4`` (the decode step with
NVFP4 weights), ``prefill`` (NVFP4 W4A4, 8192 x 28672 x
8192, A quantized on the fly), ``moe`` (MXFP4 W4A4, 256 x 2048 x 7168, A
quantized on the fly), ``moe_fused`` (the same, A quantized in the GEMM's own
prologue: one launch), ``grouped`` (64-expert routed NVFP4 MoE),
``quantize`` / ``quantize_rne`` (NVFP4 quantization of the prefill
activations alone, E2M1 ties to the smaller magnitude / to even), ``tiny``.

``--impl reference`` times the CPU oracle (the reference arm: a plain, slow
numpy/FP64 restatement of the method) on a bounded sample of the same
workload.  Multi-GPU (torchrun): every rank runs an independent replica
(weak scaling; the decode GEMM has no exchange step); ``value`` sums the
ranks' work over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal dense ratio FP4 : BF16 on GB300 (13.5 vs 2.25 PFLOP/s)
FP4_OVER_BF16 = 6.0

# ncu-measured DRAM traffic per launch of the dominant kernel (bytes), keyed by
# workload; None until a capture of the current kernel exists.
NCU_TRAFFIC = {
    # ncu dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant
    # kernel of the current code, at the bench's own sizes:
    # w4a16_kernel, mean over the M = 1, 4, 16 launches at N = K = 8192
    # (captured again after the 16-token staging change: 34.66 / 34.71 / 34.92 MB)
    "decode": 34.76e6,
    # w4a16_kernel<NVFP4> (f16 form), the same (37.80 / 37.85 / 38.05 MB)
    "decode_nvfp4": 37.90e6,
    # fp4_gemm_kernel (CTA pairs) at 8192 x 28672 x 8192, mean of 3 launches
    # (231 MB read: A and B once each, scales; 435 MB of C written)
    "prefill": 666.5e6,
    # split-K fp4_gemm_kernel (128-wide tiles, partial sums through L2) at
    # 256 x 2048 x 7168, mean of 3 launches (C and the partials stay in L2)
    "moe": 8.83e6,
    # the same with the activation quantization in its prologue (reads raw A)
    "moe_fused": 11.59e6,
    # amax_kernel and nvfp4_kernel, mean per launch over 2 steps (ncu flushes L2
    # before each kernel, so the encode pass's reuse of x from L2 is not in it)
    "quantize": 141.0e6,
    "quantize_rne": 141.0e6,
    # fp8_gemm_pair_kernel at 8192 x 28672 x 8192, mean of 3 launches (681 MB
    # read: B once per band of 4096 A rows; 450 MB of C written)
    "fp8_blockwise": 1131.1e6,
    # w4a8_gemm_pair_kernel at 8192 x 28672 x 8192, mean of 3 launches (385 MB
    # read, 445 MB written)
    "w4a8": 830.2e6,
}


def read_probe_rate(q4, dev, nbytes: float) -> float:
    """GB/s of q4_read_probe streaming `nbytes` per launch, launches back to
    back in a CUDA graph over rotating buffers (> 2 x L2 in total)."""
    nbytes = max(16, int(nbytes) // 16 * 16)
    nbuf = max(2, -(-300_000_000 // nbytes))
    bufs = [torch.ones(nbytes, dtype=torch.uint8, device=dev) for _ in range(nbuf)]
    sink = torch.zeros(int(q4.lib().q4_read_probe_sink_words()), dtype=torch.int32, device=dev)
    inner = nbuf * -(-30 // nbuf)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(inner):
            q4.read_probe(bufs[i % nbuf], sink)
    g.replay()
    torch.cuda.synchronize()
    reps = max(3, -(-300 // inner))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3
    del bufs
    return nbytes * inner * reps / t / 1e9


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- distributed

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, use_gpu: bool):
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if use_gpu else "gloo"
            if use_gpu:
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            if torch.cuda.is_available():
                self.pg.barrier(device_ids=[self.local])
            else:
                self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        dev = torch.device("cuda", self.local) if torch.cuda.is_available() else torch.device("cpu")
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        dev = torch.device("cuda", self.local) if torch.cuda.is_available() else torch.device("cpu")
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


METRIC = "FP4/INT4 GEMM TFLOP/s & HBM GB/s at decode/prefill shapes, % of roofline"


# --------------------------------------------------------------------------- workloads

class Decode:
    """W4A16 decode: INT4 g128 weights N = K = 8192, bf16 activations M = 1, 4, 16."""
    name = "w4a16_decode"
    unit = "GB/s"
    bound = "hbm"
    default_steps = 30000
    N = K = 8192
    Ms = (1, 4, 16)
    copies = 8  # 8 x 34.6 MB of weights rotate, > 2 x L2
    kernel = "w4a16_kernel"
    read_probe = True

    def config(self):
        return {"workload": "w4a16_decode N=K=8192 INT4-g128 weights, bf16 A, M=1,4,16 per step",
                "M": list(self.Ms), "N": self.N, "K": self.K,
                "l2": f"rotating {self.copies} weight copies ({self.copies * self.weight_bytes() / 1e6:.0f} MB > L2)"}

    def weight_bytes(self):
        return self.N * self.K // 2 + self.N * (self.K // 128) * 2

    def bytes_per_gemm(self, M, N=None):
        N = self.N if N is None else N
        return N * self.K // 2 + N * (self.K // 128) * 2 + M * self.K * 2 + M * N * 2

    def units_per_step(self):
        return sum(self.bytes_per_gemm(M) for M in self.Ms)

    def flops_per_step(self):
        return sum(2 * M * self.N * self.K for M in self.Ms)

    launches_per_step = 3

    def setup(self, q4, dev, seed, shape=None):
        self.q4 = q4
        if shape:
            self.N, self.K = shape[1], shape[2]
        w = workloads.int4_weights(self.N, self.K, seed)
        wd = torch.from_numpy(w).to(dev)
        wq, ws = q4.quantize_int4_g128(wd)
        del wd
        self.wq = [wq] + [wq.clone() for _ in range(self.copies - 1)]
        self.ws = [ws] + [ws.clone() for _ in range(self.copies - 1)]
        self.w_host = w
        # the step's three activation matrices (and outputs) are row slices of
        # one buffer each, so that the end-to-end step moves them with one
        # host-to-device and one device-to-host copy
        rows = sum(self.Ms)
        a_all = torch.cat([workloads.to_bf16(workloads.normal(workloads.rng_for(seed, 1), (M, self.K), 1.0))
                           for M in self.Ms])
        self.A_all = a_all.to(dev)
        self.C_all = torch.empty((rows, self.N), dtype=torch.bfloat16, device=dev)
        self.A_pin = a_all.pin_memory()
        self.C_pin = torch.empty((rows, self.N), dtype=torch.bfloat16).pin_memory()
        offs = np.cumsum((0,) + tuple(self.Ms))
        self.A = {M: self.A_all[offs[j]:offs[j + 1]] for j, M in enumerate(self.Ms)}
        self.C = {M: self.C_all[offs[j]:offs[j + 1]] for j, M in enumerate(self.Ms)}
        self.A_host = {M: self.A_pin[offs[j]:offs[j + 1]] for j, M in enumerate(self.Ms)}
        self.h2d = sum(M * self.K * 2 for M in self.Ms)
        self.d2h = sum(M * self.N * 2 for M in self.Ms)

    def step(self, i):
        for j, M in enumerate(self.Ms):
            c = (3 * i + j) % self.copies
            self.q4.gemm_w4a16_int4(self.A[M], self.wq[c], self.ws[c], out=self.C[M])

    def kernel_only(self, i):
        self.step(i)

    kernel_units = units_per_step
    kernel_launches = 3

    def e2e_step(self, i):
        self.A_all.copy_(self.A_pin, non_blocking=True)
        self.step(i)
        self.C_pin.copy_(self.C_all, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    # ---- oracle sample: the first `rows` weight rows, all three M
    def oracle_prepare(self, rows):
        import oracle
        self.o_rows = rows
        self.o_w = oracle.quantize_int4_g128(self.w_host[:rows])
        self.o_a = {M: self.A_host[M].float().numpy() for M in self.Ms}

    def oracle_step(self):
        import oracle
        for M in self.Ms:
            oracle.gemm_w4a16_int4(self.o_a[M], *self.o_w)

    def oracle_units(self):
        return sum(self.bytes_per_gemm(M, self.o_rows) for M in self.Ms)

    def oracle_sample_text(self):
        return (f"first {self.o_rows} of {self.N} weight rows x M=1,4,16 "
                f"(dequantize + FP64 GEMM; codes from the oracle's own quantizer)")

    oracle_grain = 64


class DecodeNvfp4(Decode):
    """W4A16 decode with NVFP4 weights: N = K = 8192, bf16 activations M = 1, 4, 16."""
    name = "w4a16_decode_nvfp4"
    kernel = "w4a16_kernel<NVFP4>"

    def config(self):
        return {"workload": "w4a16_decode_nvfp4 N=K=8192 NVFP4 weights (row-major E4M3 scales), "
                            "bf16 A, M=1,4,16 per step",
                "M": list(self.Ms), "N": self.N, "K": self.K,
                "l2": f"rotating {self.copies} weight copies ({self.copies * self.weight_bytes() / 1e6:.0f} MB > L2)"}

    def weight_bytes(self):
        return self.N * self.K // 2 + self.N * (self.K // 16)

    def bytes_per_gemm(self, M, N=None):
        N = self.N if N is None else N
        return N * self.K // 2 + N * (self.K // 16) + M * self.K * 2 + M * N * 2

    def setup(self, q4, dev, seed, shape=None):
        super().setup(q4, dev, seed, shape)
        del self.wq, self.ws
        wd = torch.from_numpy(self.w_host).to(dev)
        c, s, g = q4.quantize_nvfp4(wd)
        del wd
        self.wq = [c] + [c.clone() for _ in range(self.copies - 1)]
        self.ws = [s] + [s.clone() for _ in range(self.copies - 1)]
        self.wg = [g] + [g.clone() for _ in range(self.copies - 1)]

    def step(self, i):
        for j, M in enumerate(self.Ms):
            c = (3 * i + j) % self.copies
            self.q4.gemm_w4a16_nvfp4(self.A[M], self.wq[c], self.ws[c], self.wg[c], out=self.C[M])

    def kernel_only(self, i):
        self.step(i)

    def oracle_prepare(self, rows):
        import oracle
        self.o_rows = rows
        self.o_w = oracle.quantize_nvfp4(self.w_host, rows=np.arange(rows))
        self.o_a = {M: self.A_host[M].float().numpy() for M in self.Ms}

    def oracle_step(self):
        import oracle
        for M in self.Ms:
            oracle.gemm_w4a16_nvfp4(self.o_a[M], *self.o_w)


class QuantizeNvfp4:
    """NVFP4 quantization of the prefill activations, A bf16 8192 x 8192 into the
    tensor-core scale layout: the amax pass and the encode pass."""
    name = "nvfp4_quantize"
    unit = "GB/s"
    bound = "hbm"
    default_steps = 2000
    kernel = "amax_kernel + nvfp4_kernel"
    rounding = "pages"
    M = K = 8192
    launches_per_step = 2
    kernel_launches = 2

    def config(self):
        return {"workload": f"nvfp4_quantize A bf16 {self.M}x{self.K} (the prefill activations) -> codes + "
                            f"MMA-layout E4M3 scales + tensor scale, E2M1 ties: {self.rounding}",
                "M": self.M, "K": self.K, "l2": "input larger than L2 (134 MB)",
                "bytes": "one read of x + codes + scales (the amax pass's read of x is overhead)"}

    def setup(self, q4, dev, seed, shape=None):
        self.q4 = q4
        if shape:
            self.M, self.K = shape[0], shape[-1]
        a = workloads.prefill_activations(seed, self.M, self.K)
        self.x_host = a.float().numpy()
        self.x = a.to(dev)
        # codes and scales are slices of one buffer: one device-to-host copy
        # returns both in the end-to-end step
        nc, ns = self.M * self.K // 2, q4.mma_scales_bytes(self.M, self.K // 16)
        self.out = torch.empty(nc + ns, dtype=torch.uint8, device=dev)
        self.codes = self.out[:nc].view(self.M, self.K // 2)
        self.sf = self.out[nc:]
        self.g = torch.empty(1, dtype=torch.float32, device=dev)
        self.ws = q4.workspace(q4.OP_QUANTIZE_NVFP4, self.M, 0, self.K, dev)
        self.x_pin = a.pin_memory()
        self.out_host = torch.empty_like(self.out, device="cpu").pin_memory()
        self.h2d = self.M * self.K * 2
        self.d2h = self.codes.numel() + self.sf.numel()

    def step(self, i):
        rc = self.q4.lib().quantize_nvfp4_ex(
            self.x.data_ptr(), 1, self.M, self.K, self.codes.data_ptr(), self.sf.data_ptr(), 1,
            1 if self.rounding == "rne" else 0, self.g.data_ptr(), self.ws.data_ptr(),
            self.ws.numel(), torch.cuda.current_stream().cuda_stream)
        assert rc == 0

    kernel_only = step

    def units_per_step(self):
        # the method's bytes: one read of x, codes and scales written.  The
        # implementation reads x twice (the tensor scale needs the whole
        # tensor's amax before any element is encoded); the second read is
        # overhead, not work, and is not counted
        return self.M * self.K * 2 + self.M * self.K // 2 + self.M * self.K // 16

    kernel_units = units_per_step

    def flops_per_step(self):
        return 0.0

    def e2e_step(self, i):
        self.x.copy_(self.x_pin, non_blocking=True)
        self.step(i)
        self.out_host.copy_(self.out, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    def oracle_prepare(self, rows):
        self.o_rows = rows
        self.o_x = np.ascontiguousarray(self.x_host[:rows])

    def oracle_step(self):
        import oracle
        oracle.quantize_nvfp4(self.o_x, rounding=self.rounding)

    def oracle_units(self):
        return self.o_rows * self.K * 2 + self.o_rows * self.K // 2 + self.o_rows * self.K // 16

    def oracle_sample_text(self):
        return (f"the first {self.o_rows} rows as their own tensor (amax, E4M3 block scales, "
                f"E2M1 codes, ties: {self.rounding})")

    oracle_grain = 64


class QuantizeNvfp4Rne(QuantizeNvfp4):
    name = "nvfp4_quantize_rne"
    rounding = "rne"


class W4A4:
    """W4A4 GEMM with A quantized on the fly; B pre-quantized (MMA scale layout)."""
    nvfp4 = True

    def setup_common(self, q4, dev, a_bf16, b_f32, a_copies=1, b_copies=1):
        self.q4 = q4
        self.M, self.K = a_bf16.shape
        self.N = b_f32.shape[0]
        bd = torch.from_numpy(b_f32).to(dev)
        if self.nvfp4:
            bc, bs, bg = q4.quantize_nvfp4(bd, scale_layout="mma")
            bop = q4.Fp4Operand(bc, bs, "mma", bg)
        else:
            bc, bs = q4.quantize_mxfp4(bd, scale_layout="mma")
            bop = q4.Fp4Operand(bc, bs, "mma", None)
        del bd
        self.B = [bop] + [q4.Fp4Operand(bop.codes.clone(), bop.scales.clone(), "mma",
                                        None if bop.tensor_scale is None else bop.tensor_scale.clone())
                          for _ in range(b_copies - 1)]
        a = a_bf16.to(dev)
        self.A = [a] + [a.clone() for _ in range(a_copies - 1)]
        self.a_host = a_bf16
        self.b_host = b_f32
        op = q4.OP_GEMM_W4A4_NVFP4 if self.nvfp4 else q4.OP_GEMM_W4A4_MXFP4
        self.ws = q4.workspace(op, self.M, self.N, self.K, dev)
        self.C = torch.empty((self.M, self.N), dtype=torch.bfloat16, device=dev)
        self.fn = q4.gemm_w4a4_nvfp4 if self.nvfp4 else q4.gemm_w4a4_mxfp4
        # pre-quantized copy of A for timing the GEMM kernel alone
        if self.nvfp4:
            ac, as_, ag = q4.quantize_nvfp4(self.A[0], scale_layout="mma")
            self.Aq = q4.Fp4Operand(ac, as_, "mma", ag)
        else:
            ac, as_ = q4.quantize_mxfp4(self.A[0], scale_layout="mma")
            self.Aq = q4.Fp4Operand(ac, as_, "mma", None)
        self.A_pin = a_bf16.pin_memory()
        self.C_host = torch.empty((self.M, self.N), dtype=torch.bfloat16).pin_memory()
        self.h2d = self.M * self.K * 2
        self.d2h = self.M * self.N * 2

    launches_per_step = 3  # amax or memset-free quantize kernels + GEMM (see gpu_launches)

    def step(self, i):
        self.fn(self.A[i % len(self.A)], self.B[i % len(self.B)], self.K, out=self.C, ws=self.ws)

    def kernel_only(self, i):
        self.fn(self.Aq, self.B[i % len(self.B)], self.K, out=self.C, ws=self.ws)

    kernel_launches = 1

    def e2e_step(self, i):
        self.A[0].copy_(self.A_pin, non_blocking=True)
        self.fn(self.A[0], self.B[i % len(self.B)], self.K, out=self.C, ws=self.ws)
        self.C_host.copy_(self.C, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    def flops_per_step(self):
        return 2.0 * self.M * self.N * self.K

    def bytes_per_step(self):
        nsf = self.K // (16 if self.nvfp4 else 32)
        return (self.M * self.K * 2 + self.N * self.K // 2 + self.N * nsf + self.M * self.N * 2)

    def oracle_prepare(self, rows):
        self.o_rows = rows
        self.o_a = self.a_host.float().numpy()

    def oracle_step(self):
        import oracle
        ra = np.arange(min(self.M, 64))
        rb = np.arange(self.o_rows)
        if self.nvfp4:
            qa = oracle.quantize_nvfp4(self.o_a, rows=ra)
            qb = oracle.quantize_nvfp4(self.b_host, rows=rb)
            oracle.gemm_w4a4_nvfp4(*qa, *qb)
        else:
            qa = oracle.quantize_mxfp4(self.o_a, rows=ra)
            qb = oracle.quantize_mxfp4(self.b_host, rows=rb)
            oracle.gemm_w4a4_mxfp4(*qa, *qb)

    def oracle_sample_text(self):
        return (f"A rows 0..{min(self.M, 64) - 1} x B rows 0..{self.o_rows - 1}: quantize both "
                f"(tensor scale over the whole operand) + FP64 GEMM")

    oracle_grain = 128


class Prefill(W4A4):
    name = "nvfp4_prefill"
    unit = "TFLOP/s"
    bound = "tensor"
    default_steps = 400
    kernel = "fp4_gemm_kernel"
    nvfp4 = True

    def config(self):
        return {"workload": f"nvfp4_prefill A bf16 {self.M}x{self.K} (quantized on the fly), B NVFP4 {self.N}x{self.K}",
                "M": self.M, "N": self.N, "K": self.K, "l2": "inputs larger than L2 (A 134 MB bf16, B 132 MB)"}

    def setup(self, q4, dev, seed, shape=None):
        a, b = workloads.prefill(seed, *(shape or ()))
        self.setup_common(q4, dev, a, b)

    def units_per_step(self):
        return self.flops_per_step()

    def kernel_units(self):
        return self.flops_per_step()

    def oracle_units(self):
        return 2.0 * min(self.M, 64) * self.o_rows * self.K


class Moe(W4A4):
    name = "mxfp4_moe"
    unit = "GB/s"
    bound = "hbm"
    default_steps = 5000
    kernel = "fp4_gemm_kernel"
    nvfp4 = False
    launches_per_step = 2  # activation quantizer + GEMM
    read_probe = True

    def config(self):
        return {"workload": f"mxfp4_moe A bf16 {self.M}x{self.K} (0.5% channels x20, quantized on the fly), B MXFP4 {self.N}x{self.K}",
                "M": self.M, "N": self.N, "K": self.K, "l2": "rotating 8 A and 16 B copies (> L2)"}

    def setup(self, q4, dev, seed, shape=None):
        a, b = workloads.moe(seed, *(shape or ()))
        self.setup_common(q4, dev, a, b, a_copies=8, b_copies=16)

    def units_per_step(self):
        return self.bytes_per_step()

    def kernel_units(self):
        return self.N * self.K // 2 + self.N * self.K // 32 + self.M * self.K // 2 + self.M * self.K // 32 + self.M * self.N * 2

    def oracle_units(self):
        m = min(self.M, 64)
        return m * self.K * 2 + self.o_rows * self.K // 2 + self.o_rows * self.K // 32 + m * self.o_rows * 2


class MoeFused(Moe):
    """The MoE shape through the single-launch call: the GEMM quantizes its
    bf16 activations in its own prologue (no separate quantizer launch)."""
    name = "mxfp4_moe_fused"
    launches_per_step = 1
    kernel_launches = 1

    def config(self):
        c = super().config()
        c["workload"] = c["workload"].replace("quantized on the fly", "quantized in the GEMM prologue")
        return c

    def setup(self, q4, dev, seed, shape=None):
        super().setup(q4, dev, seed, shape)
        self.ws_fused = q4.workspace(q4.OP_GEMM_W4A4_MXFP4_FUSED, self.M, self.N, self.K, dev)

    def step(self, i):
        self.q4.gemm_w4a4_mxfp4_fused(self.A[i % len(self.A)], self.B[i % len(self.B)], self.K,
                                      out=self.C, ws=self.ws_fused)

    kernel_only = step

    def kernel_units(self):
        return self.bytes_per_step()  # the one launch reads raw A itself

    def e2e_step(self, i):
        self.A[0].copy_(self.A_pin, non_blocking=True)
        self.q4.gemm_w4a4_mxfp4_fused(self.A[0], self.B[i % len(self.B)], self.K, out=self.C,
                                      ws=self.ws_fused)
        self.C_host.copy_(self.C, non_blocking=True)
        torch.cuda.current_stream().synchronize()


class Fp8Blockwise:
    """FP8 blockwise GEMM: A quantized on the fly into (1, 128) blocks, B
    pre-quantized into 128 x 128 blocks, block-promoted tcgen05 GEMM."""
    name = "fp8_blockwise"
    unit = "TFLOP/s"
    bound = "tensor"
    tensor_fmt = "fp8"  # the roofline peak: a library FP8 GEMM measured live
    tensor_over_bf16 = 2.0  # else nominal dense FP8 : BF16 on GB300 (4.5 vs 2.25 PFLOP/s)
    default_steps = 200
    kernel = "fp8_gemm_pair_kernel"  # CTA pairs (M > 128)
    launches_per_step = 2  # activation quantizer + GEMM
    kernel_launches = 1
    oracle_grain = 128

    def config(self):
        return {"workload": f"fp8_blockwise A bf16 {self.M}x{self.K} (quantized on the fly, 1x128 blocks), "
                            f"B E4M3 {self.N}x{self.K} (128x128 blocks)",
                "M": self.M, "N": self.N, "K": self.K,
                "l2": "inputs larger than L2 (A 134 MB bf16, B 235 MB)"}

    def setup(self, q4, dev, seed, shape=None):
        self.q4 = q4
        a, b = workloads.prefill(seed, *(shape or ()))
        self.M, self.K = a.shape
        self.N = b.shape[0]
        self.a_host, self.b_host = a, b
        bd = torch.from_numpy(b).to(dev)
        self.qb, self.sb = q4.quantize_fp8_blockwise(bd, 128)
        del bd
        self.A = a.to(dev)
        self.qa = torch.empty((self.M, self.K), dtype=torch.uint8, device=dev)
        self.sa = torch.empty((self.M, self.K // 128), dtype=torch.float32, device=dev)
        q4.quantize_fp8_blockwise(self.A, 1, codes=self.qa, scales=self.sa)
        self.C = torch.empty((self.M, self.N), dtype=torch.bfloat16, device=dev)
        self.A_pin = a.pin_memory()
        self.C_host = torch.empty((self.M, self.N), dtype=torch.bfloat16).pin_memory()
        self.h2d = self.M * self.K * 2
        self.d2h = self.M * self.N * 2

    def step(self, i):
        self.q4.quantize_fp8_blockwise(self.A, 1, codes=self.qa, scales=self.sa)
        self.q4.gemm_fp8_blockwise(self.qa, self.sa, self.qb, self.sb, out=self.C)

    def kernel_only(self, i):
        self.q4.gemm_fp8_blockwise(self.qa, self.sa, self.qb, self.sb, out=self.C)

    def e2e_step(self, i):
        self.A.copy_(self.A_pin, non_blocking=True)
        self.step(i)
        self.C_host.copy_(self.C, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    def flops_per_step(self):
        return 2.0 * self.M * self.N * self.K

    def units_per_step(self):
        return self.flops_per_step()

    def kernel_units(self):
        return self.flops_per_step()

    def oracle_prepare(self, rows):
        self.o_rows = rows
        self.o_a = self.a_host.float().numpy()

    def oracle_step(self):
        import oracle
        qa = oracle.quantize_fp8_blockwise(self.o_a[:min(self.M, 64)], (1, 128))
        qb = oracle.quantize_fp8_blockwise(self.b_host[:self.o_rows], (128, 128))
        oracle.gemm_fp8_blockwise(*qa, *qb)

    def oracle_units(self):
        return 2.0 * min(self.M, 64) * self.o_rows * self.K

    def oracle_sample_text(self):
        return (f"A rows 0..{min(self.M, 64) - 1} x B rows 0..{self.o_rows - 1}: FP8 blockwise quantize "
                f"both + FP64 block-promoted GEMM")


class W4a8(Fp8Blockwise):
    """W4A8: A quantized on the fly into FP8 (1, 128) blocks, INT4 g128 weights
    converted to E4M3 inside the GEMM (their FP16 group scales in the promotion)."""
    name = "w4a8"
    kernel = "w4a8_gemm_pair_kernel"  # CTA pairs (M > 128)

    def config(self):
        return {"workload": f"w4a8 A bf16 {self.M}x{self.K} (FP8 1x128 blocks, quantized on the fly), "
                            f"W INT4 g128 {self.N}x{self.K}",
                "M": self.M, "N": self.N, "K": self.K,
                "l2": "inputs larger than L2 (A 134 MB bf16, W 117 MB INT4)"}

    def setup(self, q4, dev, seed, shape=None):
        self.q4 = q4
        a, b = workloads.prefill(seed, *(shape or ()))
        self.M, self.K = a.shape
        self.N = b.shape[0]
        self.a_host, self.b_host = a, b
        bd = torch.from_numpy(b).to(dev)
        self.wq, ws16 = q4.quantize_int4_g128(bd)
        del bd
        self.wsk = q4.w4a8_weight_scales(ws16)
        self.A = a.to(dev)
        self.qa = torch.empty((self.M, self.K), dtype=torch.uint8, device=dev)
        self.sa = torch.empty((self.M, self.K // 128), dtype=torch.float32, device=dev)
        q4.quantize_fp8_blockwise(self.A, 1, codes=self.qa, scales=self.sa)
        self.C = torch.empty((self.M, self.N), dtype=torch.bfloat16, device=dev)
        self.A_pin = a.pin_memory()
        self.C_host = torch.empty((self.M, self.N), dtype=torch.bfloat16).pin_memory()
        self.h2d = self.M * self.K * 2
        self.d2h = self.M * self.N * 2

    def step(self, i):
        self.q4.quantize_fp8_blockwise(self.A, 1, codes=self.qa, scales=self.sa)
        self.q4.gemm_w4a8(self.qa, self.sa, self.wq, self.wsk, out=self.C)

    def kernel_only(self, i):
        self.q4.gemm_w4a8(self.qa, self.sa, self.wq, self.wsk, out=self.C)

    def oracle_step(self):
        import oracle
        qa = oracle.quantize_fp8_blockwise(self.o_a[:min(self.M, 64)], (1, 128))
        wc, ws = oracle.quantize_int4_g128(self.b_host[:self.o_rows])
        oracle.gemm_w4a8(*qa, wc, ws)

    def oracle_sample_text(self):
        return (f"A rows 0..{min(self.M, 64) - 1} x W rows 0..{self.o_rows - 1}: FP8 blockwise quantize A, "
                f"INT4 g128 quantize W + FP64 block-promoted GEMM")


class Grouped:
    """64-expert routed NVFP4 MoE: tokens quantized once, grouped tcgen05 GEMM."""
    name = "grouped_moe"
    unit = "GB/s"
    bound = "hbm"
    default_steps = 200
    kernel = "grouped step (quantize tokens + routed scales + grouped GEMM)"
    T, E, N, K, top = 4096, 64, 2048, 7168, 8
    launches_per_step = 6  # amax, quantize, schedule, routed scales, routed copy, grouped GEMM
    kernel_launches = 6

    def config(self):
        return {"workload": "grouped_moe 64 experts NVFP4 2048x7168, 4096 bf16 tokens, top-8 routing",
                "T": self.T, "E": self.E, "N": self.N, "K": self.K, "top_k": self.top,
                "l2": "inputs larger than L2 (528 MB of expert weights)"}

    def setup(self, q4, dev, seed, shape=None):
        self.q4 = q4
        tok, _, offs, rt = workloads.grouped(seed, T=self.T, E=self.E, N=self.N, K=self.K,
                                             top_k=self.top, experts=False)
        self.R = int(offs[-1])
        self.wc = torch.empty((self.E, self.N, self.K // 2), dtype=torch.uint8, device=dev)
        sfb = q4.mma_scales_bytes(self.N, self.K // 16)
        self.wsf = torch.empty(self.E * sfb, dtype=torch.uint8, device=dev)
        self.wg = torch.empty(self.E, dtype=torch.float32, device=dev)
        self.seed = seed
        for e in range(self.E):
            w = torch.from_numpy(workloads.expert_weight(seed, e, self.N, self.K)).to(dev)
            c, s, g = q4.quantize_nvfp4(w, scale_layout="mma")
            self.wc[e].copy_(c)
            self.wsf[e * sfb:(e + 1) * sfb].copy_(s)
            self.wg[e:e + 1].copy_(g)
            del w
        self.tok_host = tok
        self.tok = tok.to(dev)
        self.offs_h, self.rt_h = offs, rt
        self.offs = torch.from_numpy(offs).to(dev)
        self.rt = torch.from_numpy(rt).to(dev)
        self.ws = q4.moe_workspace(self.T, self.N, self.K, self.E, self.R, dev)
        self.C = torch.empty((self.R, self.N), dtype=torch.bfloat16, device=dev)
        self.tok_pin = tok.pin_memory()
        self.C_host = torch.empty((self.R, self.N), dtype=torch.bfloat16).pin_memory()
        self.h2d = self.T * self.K * 2
        self.d2h = self.R * self.N * 2

    def step(self, i):
        self.q4.grouped_gemm_moe(self.tok, self.offs, self.rt, self.wc, self.wsf, self.wg, self.N,
                                 ws=self.ws, out=self.C)

    kernel_only = step

    def units_per_step(self):
        return (self.E * self.N * self.K // 2 + self.E * self.N * self.K // 16 + self.T * self.K * 2
                + self.R * self.N * 2)

    kernel_units = units_per_step

    def flops_per_step(self):
        return 2.0 * self.R * self.N * self.K

    def e2e_step(self, i):
        self.tok.copy_(self.tok_pin, non_blocking=True)
        self.step(i)
        self.C_host.copy_(self.C, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    def oracle_prepare(self, rows):
        self.o_rows = rows
        self.o_tok = self.tok_host.float().numpy()
        self.o_w = workloads.expert_weight(self.seed, 0, self.N, self.K)

    def oracle_step(self):
        import oracle
        r = self.rt_h[self.offs_h[0]:self.offs_h[0] + 64]
        qa = oracle.quantize_nvfp4(self.o_tok, rows=r)
        qb = oracle.quantize_nvfp4(self.o_w, rows=np.arange(self.o_rows))
        oracle.gemm_w4a4_nvfp4(*qa, *qb)

    def oracle_units(self):
        return 64 * self.K * 2 + self.o_rows * self.K // 2 + self.o_rows * self.K // 16 + 64 * self.o_rows * 2

    def oracle_sample_text(self):
        return (f"64 routed rows of expert 0 x its first {self.o_rows} weight rows: quantize both + FP64 GEMM")

    oracle_grain = 128


WORKLOADS = {"decode": Decode, "decode_nvfp4": DecodeNvfp4, "prefill": Prefill, "moe": Moe,
             "moe_fused": MoeFused,
             "grouped": Grouped, "quantize": QuantizeNvfp4, "quantize_rne": QuantizeNvfp4Rne,
             "fp8_blockwise": Fp8Blockwise, "w4a8": W4a8}
DTYPES = {"decode": "bf16 (exact int4 values) x bf16 -> fp32",
          "decode_nvfp4": "bf16 (exact e2m1 x e4m3 values) x bf16 -> fp32",
          "quantize": "bf16 -> e2m1 + e4m3 (fp32 arithmetic)", "quantize_rne": "bf16 -> e2m1 + e4m3 (fp32 arithmetic)",
          "prefill": "e2m1 x e2m1 -> fp32",
          "moe": "e2m1 x e2m1 -> fp32", "moe_fused": "e2m1 x e2m1 -> fp32", "grouped": "e2m1 x e2m1 -> fp32",
          "fp8_blockwise": "e4m3 x e4m3 -> fp32 (block-promoted)",
          "w4a8": "e4m3 x int4 (exact e4m3) -> fp32 (block-promoted)"}


def scale_units(x, unit):
    return x / 1e9 if unit == "GB/s" else x / 1e12


def time_oracle(wl, seconds: float):
    """Time the oracle as it stands on a sample sized to about ``seconds``."""
    rows = wl.oracle_grain
    wl.oracle_prepare(rows)
    t0 = time.perf_counter()
    wl.oracle_step()
    t1 = time.perf_counter() - t0
    reps = max(1, int(seconds / max(t1, 1e-6)))
    t0 = time.perf_counter()
    for _ in range(reps):
        wl.oracle_step()
    el = time.perf_counter() - t0
    val = scale_units(wl.oracle_units() * reps / el, wl.unit)
    return {"value": val, "unit": wl.unit, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{wl.oracle_sample_text()}; {reps} repetitions in {el:.1f} s; numpy "
                      f"elementwise on 1 thread, FP64 matmul on the BLAS threads"}


def chunk_for(K: int) -> int:
    for g in range(min(K, 100), 0, -1):
        if K % g == 0:
            return g
    return 1


def run_reference(args, dist):
    if dist.world > 1 and dist.rank != 0:
        return
    wl = WORKLOADS[args.workload]()
    wl_setup_host(wl, args.seed)
    K = args.steps or wl.default_steps
    W = max(3, args.warmup)
    # size the per-step sample so that the whole run takes about --reference-seconds
    # (two minutes by default)
    wl.oracle_prepare(wl.oracle_grain)
    t0 = time.perf_counter()
    wl.oracle_step()
    t1 = time.perf_counter() - t0
    grains = max(1, int(args.reference_seconds / max((K + W) * t1, 1e-9)))
    wl.oracle_prepare(wl.oracle_grain * min(grains, 64))
    for _ in range(W):
        wl.oracle_step()
    t0 = time.perf_counter()
    for _ in range(K):
        wl.oracle_step()
    el = time.perf_counter() - t0
    val = scale_units(wl.oracle_units() * K / el, wl.unit)
    cfg = wl.config()
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": wl.unit, "n_gpus": args.gpus,
            "steps": K, "warmup": W, "ms_per_step": el / K * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
            "cpu_baseline": {"kind": "oracle", "cores": os.cpu_count(), "value": val, "unit": wl.unit,
                             "sample": wl.oracle_sample_text() + " per step"},
            "e2e": {"value": val, "unit": wl.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def peak_text(wl):
    r = getattr(wl, "tensor_over_bf16", FP4_OVER_BF16)
    return f"bf16_tflops_sustained x {r:g} (nominal {'FP8' if r == 2.0 else 'FP4'}:BF16)"


def library_peak(fmt: str, dev, n: int = 8192, reps: int = 10, seconds: float = 1.5):
    """Dense tensor-core peaks of this GPU for ``fmt`` ("nvfp4" or "fp8"),
    measured the way the bf16 peaks are: a library GEMM (torch._scaled_mm on
    cuBLASLt) of n x n x n, as a burst (the best of ``reps`` groups of 5
    back-to-back launches, CUDA events) and sustained (back to back for
    ``seconds``, the rate over the last two thirds, under the power cap).  Returns
    (burst TFLOP/s, sustained TFLOP/s, description), or (None, None, why) when
    the library path is missing."""
    try:
        g = torch.Generator(device=dev).manual_seed(0)
        if fmt == "nvfp4":
            a = torch.randint(0, 256, (n, n // 2), device=dev, dtype=torch.uint8, generator=g)
            b = torch.randint(0, 256, (n, n // 2), device=dev, dtype=torch.uint8, generator=g)
            a, b = a.view(torch.float4_e2m1fn_x2), b.view(torch.float4_e2m1fn_x2)
            sa = torch.ones(n * (n // 16), device=dev).to(torch.float8_e4m3fn)  # tensor-core layout
            sb = torch.ones(n * (n // 16), device=dev).to(torch.float8_e4m3fn)
            what = "NVFP4 (E2M1, E4M3 block scales of 16)"
        else:
            a = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
            b = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
            sa = sb = torch.ones((), device=dev)
            what = "FP8 E4M3 (per-tensor scales)"
        run = lambda: torch._scaled_mm(a, b.t(), sa, sb, out_dtype=torch.bfloat16)
        flop = 2.0 * n ** 3
        for _ in range(5):
            run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        best = float("inf")
        for _ in range(reps):  # short back-to-back groups: clocks up, power cap not yet reached
            e0.record()
            for _ in range(5):
                run()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) / 1e3 / 5)
        burst = flop / best / 1e12
        per = max(1, int(seconds / 3 / best))  # launches per third
        for _ in range(per):
            run()
        e0.record()
        for _ in range(2 * per):
            run()
        e1.record()
        torch.cuda.synchronize()
        sustained = flop * 2 * per / (e0.elapsed_time(e1) / 1e3) / 1e12
        del a, b
        torch.cuda.empty_cache()
        return burst, sustained, (f"measured live: torch._scaled_mm {what} {n}^3 (cuBLASLt), "
                                  f"burst = best of {reps} groups of 5 launches, sustained = back to back "
                                  f"for {seconds:g} s")
    except Exception as e:  # no FP4/FP8 library path in this torch build
        return None, None, f"library {fmt} GEMM unavailable ({type(e).__name__})"


def wl_setup_host(wl, seed):
    """Host-only inputs for the oracle arm (no GPU needed)."""
    if isinstance(wl, Decode):
        wl.w_host = workloads.int4_weights(wl.N, wl.K, seed)
        wl.A_host = {M: workloads.to_bf16(workloads.normal(workloads.rng_for(seed, 1), (M, wl.K), 1.0))
                     for M in wl.Ms}
    elif isinstance(wl, QuantizeNvfp4):
        wl.x_host = workloads.prefill_activations(seed, wl.M, wl.K).float().numpy()
    elif isinstance(wl, Fp8Blockwise):
        wl.a_host, wl.b_host = workloads.prefill(seed)
        wl.M, wl.K = wl.a_host.shape
        wl.N = wl.b_host.shape[0]
    elif isinstance(wl, Grouped):
        tok, _, offs, rt = workloads.grouped(seed, T=wl.T, E=wl.E, N=wl.N, K=wl.K, top_k=wl.top,
                                             experts=False)
        wl.tok_host, wl.offs_h, wl.rt_h, wl.seed = tok, offs, rt, seed
    else:
        a, b = workloads.prefill(seed) if isinstance(wl, Prefill) else workloads.moe(seed)
        wl.a_host, wl.b_host = a, b
        wl.M, wl.K = a.shape
        wl.N = b.shape[0]


SEEDS = {"decode": workloads.SEED_BASE + 2, "decode_nvfp4": workloads.SEED_BASE + 2,
         "moe": workloads.SEED_BASE + 3, "moe_fused": workloads.SEED_BASE + 3,
         "prefill": workloads.SEED_BASE + 4, "grouped": workloads.SEED_BASE + 5,
         "quantize": workloads.SEED_BASE + 4, "quantize_rne": workloads.SEED_BASE + 4,
         "fp8_blockwise": workloads.SEED_BASE + 4, "w4a8": workloads.SEED_BASE + 4}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (default: per workload)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode")
    ap.add_argument("--seed", type=int, default=None)
    ap.add_argument("--oracle-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=120.0,
                    help="--impl reference: about how long the whole run takes")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shape", default=None,
                    help="M,N,K override (a smaller case of the same code path, e.g. for profiling)")
    args = ap.parse_args()
    if args.seed is None:
        args.seed = SEEDS[args.workload]
    dist = Dist()
    if args.impl == "reference":
        run_reference(args, dist)
        return

    dist.init(use_gpu=True)
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    import int4_gemm_gb300 as q4
    q4.load()
    wl = WORKLOADS[args.workload]()
    shape = tuple(int(v) for v in args.shape.split(",")) if args.shape else None
    wl.setup(q4, dev, args.seed, shape)
    K = args.steps or wl.default_steps
    W = max(3, args.warmup)
    # a tensor-bound kernel's roofline peak: the library GEMM of its type,
    # measured here before the timed steps
    lib_peaks = (library_peak(getattr(wl, "tensor_fmt", "nvfp4"), dev) if wl.bound == "tensor"
                 else (None, None, ""))
    for i in range(W):
        wl.step(i)
    torch.cuda.synchronize()
    if q4.sync_status() != 0:
        raise RuntimeError("a kernel reported an error during warm-up")

    # the timed steps run as CUDA-graph replays of G steps each (K / G replays)
    G = chunk_for(K)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(G):
            wl.step(i)
    graph.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else dist.local)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(K // G):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    dist.barrier()
    clk = clocks.stop()
    t = dist.max(e0.elapsed_time(e1) / 1e3)
    total_units = dist.sum(wl.units_per_step() * K)
    value = scale_units(total_units / t, wl.unit)
    status = q4.sync_status()
    if status != 0:
        raise RuntimeError(f"a kernel reported status {status} during the timed steps")

    # the dominant kernel alone, in the same graph form
    pk, src = peaks()
    lib_src = ""
    if wl.bound == "hbm":
        peak, punit = pk["hbm_gbs"], "GB/s"
    else:
        punit = "TFLOP/s"
        # the kernel below runs hundreds of launches back to back: the
        # library's sustained rate is its peak (the burst rate is reported too)
        peak, lib_src = lib_peaks[1], lib_peaks[2]
        if peak is None:  # nominal ratio to the measured bf16 peak, said so below
            peak = pk["bf16_tflops_sustained"] * getattr(wl, "tensor_over_bf16", FP4_OVER_BF16)
    kg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(kg):
        for i in range(G):
            wl.kernel_only(i)
    kg.replay()
    torch.cuda.synchronize()
    # at least 200 launches of the kernel, whatever the step count
    reps = max(K // G // 2, -(-200 // (G * wl.kernel_launches)))
    e0.record()
    for _ in range(reps):
        kg.replay()
    e1.record()
    torch.cuda.synchronize()
    launches = reps * G * wl.kernel_launches
    avg_s = e0.elapsed_time(e1) / 1e3 / launches
    per_launch = wl.kernel_units() / wl.kernel_launches
    achieved = scale_units(per_launch / avg_s, punit)
    roofline = {"bound": wl.bound, "achieved": achieved, "peak": peak, "unit": punit,
                "frac": achieved / peak, "traffic": NCU_TRAFFIC.get(args.workload),
                "kernel": wl.kernel, "avg_launch_us": avg_s * 1e6,
                "peak_burst": lib_peaks[0],
                "peak_source": (f"{src} (hbm_gbs)" if punit == "GB/s" else
                                lib_src if lib_src.startswith("measured") else
                                f"{src} ({peak_text(wl)}); {lib_src}")}

    if wl.bound == "hbm" and getattr(wl, "read_probe", False):
        # context for the fraction: a bare read of the same bytes per launch
        nb = per_launch
        rp = read_probe_rate(q4, dev, nb)
        roofline["read_probe"] = {
            "gbs": rp, "bytes_per_launch": int(nb), "frac_of_peak": rp / peak,
            "kernel_over_probe": achieved / rp,
            "what": "the library's bare 16-byte-load read (q4_read_probe) of the same bytes per "
                    "launch, launches back to back in a CUDA graph over rotating buffers > 2 x L2"}

    # end to end through the public API: host buffers, copies inside the timed region
    n_e2e = min(K, 2000 if wl.unit == "GB/s" else 50)
    for i in range(3):
        wl.e2e_step(i)
    dist.barrier()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        wl.e2e_step(i)
    t_e2e = dist.max(time.perf_counter() - t0)
    e2e_val = scale_units(dist.sum(wl.units_per_step() * n_e2e) / t_e2e, wl.unit)

    cpu = None
    if dist.rank == 0 and not args.no_cpu_baseline:
        cpu = time_oracle(wl, args.oracle_seconds)

    if dist.rank == 0:
        cfg = wl.config()
        cfg["parallelism"] = f"replicas x{dist.world}" if dist.world > 1 else "single GPU"
        line = {"metric": METRIC, "value": value, "unit": wl.unit, "n_gpus": dist.world, "steps": K,
                "warmup": W, "ms_per_step": t / K * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": DTYPES[args.workload], "data": "synthetic", "config": cfg,
                "tflops": scale_units(dist.sum(wl.flops_per_step() * K) / t, "TFLOP/s"),
                "roofline": roofline, "cpu_baseline": cpu,
                "e2e": {"value": e2e_val, "unit": wl.unit, "h2d_bytes_per_step": wl.h2d,
                        "d2h_bytes_per_step": wl.d2h, "steps": n_e2e},
                "gpu_launches": K * wl.launches_per_step, "clocks": clk,
                "timing": f"CUDA events on the launching stream around {K // G} replays of a "
                          f"{G}-step CUDA graph"}
        print(json.dumps(line), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
