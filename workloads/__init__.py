"""Seeded synthetic inputs for the block-scaled 4-bit quantize + GEMM workloads.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
benchmark.  It only draws random numbers and lays them out; it contains none of
the quantization or GEMM arithmetic.  Every tensor is drawn in float32 with
numpy's PCG64 generator and, where the workload says bf16, rounded to bf16 by
torch's CPU cast (round to nearest even).

Workloads (sizes as stated for the five decode / prefill / MoE shapes):

* ``tiny``    NVFP4 W4A4: A 16x512, B 256x512 fp32, N(0, 0.02) with 0.1% of the
               entries replaced by +-U(0.5, 2); the eight-weight worked row
               (drpranayjha.com "LLM quantization", "A worked example in INT8,
               INT4 and FP4") is planted at A[0, 0:8] with A[0, 8:16] = 0.
* ``decode``  W4A16: A bf16 M in {1, 4, 16} x 8192 ~ N(0, 1); W 8192x8192
               ~ N(0, 0.02) plus 0.1% outliers.
* ``moe``     MXFP4 W4A4: A bf16 256x7168 ~ N(0, 1) with 0.5% of the channels
               scaled x20; B 2048x7168 ~ N(0, 0.02).
* ``prefill`` NVFP4 W4A4: A bf16 8192x8192 ~ N(0, 1), 0.5% channels x20;
               B 28672x8192 ~ N(0, 0.02).
* ``grouped`` 64 experts of 2048x7168 ~ N(0, 0.02); 4096 bf16 tokens ~ N(0, 1);
               top-8 routing over seeded logits N(0,1) + b_e, b_e = 0.2 N(0,1),
               with expert 63 biased by -1e4 so that it receives no rows.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "WORKED_ROW", "SEED_BASE", "rng_for", "normal", "add_entry_outliers",
    "scale_channels", "to_bf16", "tiny", "decode", "moe", "prefill", "prefill_activations",
    "grouped",
    "route_top_k", "nvfp4_pair", "mxfp4_pair", "int4_weights",
]

# The eight weights of the worked example (drpranayjha.com "LLM quantization",
# section "A worked example in INT8, INT4 and FP4").
WORKED_ROW = np.array([0.12, -0.45, 0.03, 0.88, -0.27, 0.51, -0.09, 0.34], dtype=np.float32)

SEED_BASE = 1000


def rng_for(seed: int, tag: int) -> np.random.Generator:
    """An independent PCG64 stream per (seed, tensor tag)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(tag)])))


def normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def add_entry_outliers(rng: np.random.Generator, x: np.ndarray, frac: float = 1e-3,
                       lo: float = 0.5, hi: float = 2.0) -> np.ndarray:
    """Replace round(frac * numel) entries, chosen uniformly without replacement,
    by a random sign times U(lo, hi).  Works in place on a float32 array."""
    flat = x.reshape(-1)
    count = int(round(frac * flat.size))
    if count == 0:
        return x
    pos = rng.choice(flat.size, size=count, replace=False)
    sign = np.where(rng.integers(0, 2, size=count) == 1, 1.0, -1.0)
    mag = rng.uniform(lo, hi, size=count)
    flat[pos] = (sign * mag).astype(np.float32)
    return x


def scale_channels(rng: np.random.Generator, x: np.ndarray, frac: float = 5e-3,
                   factor: float = 20.0) -> np.ndarray:
    """Multiply round(frac * K) whole input channels (columns) by ``factor``."""
    k = x.shape[-1]
    count = int(round(frac * k))
    if count:
        ch = rng.choice(k, size=count, replace=False)
        x[..., ch] *= np.float32(factor)
    return x


def to_bf16(x: np.ndarray):
    """Round a float32 array to a torch bf16 CPU tensor (RNE)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


# ---------------------------------------------------------------------------
# Operand generators at arbitrary shapes (tests use small ragged shapes)
# ---------------------------------------------------------------------------

def nvfp4_pair(M: int, N: int, K: int, seed: int, a_std: float = 0.02,
               entry_outliers: bool = True, channel_outliers: bool = False,
               worked_row: bool = False):
    """float32 A [M, K] and B [N, K] for an NVFP4 / MXFP4 W4A4 problem."""
    a = normal(rng_for(seed, 1), (M, K), a_std)
    b = normal(rng_for(seed, 2), (N, K), 0.02)
    if entry_outliers:
        add_entry_outliers(rng_for(seed, 3), a)
        add_entry_outliers(rng_for(seed, 4), b)
    if channel_outliers:
        scale_channels(rng_for(seed, 5), a)
    if worked_row and M > 0 and K >= 16:
        a[0, 0:8] = WORKED_ROW
        a[0, 8:16] = 0.0
    return a, b


def mxfp4_pair(M: int, N: int, K: int, seed: int):
    """A ~ N(0,1) with 0.5% channels x20, B ~ N(0, 0.02) (float32)."""
    a = normal(rng_for(seed, 1), (M, K), 1.0)
    scale_channels(rng_for(seed, 5), a)
    b = normal(rng_for(seed, 2), (N, K), 0.02)
    return a, b


def int4_weights(N: int, K: int, seed: int) -> np.ndarray:
    w = normal(rng_for(seed, 2), (N, K), 0.02)
    add_entry_outliers(rng_for(seed, 4), w)
    return w


# ---------------------------------------------------------------------------
# The five named workloads
# ---------------------------------------------------------------------------

def tiny(seed: int = SEED_BASE + 1):
    """A [16, 512], B [256, 512] float32 (worked row planted in A)."""
    return nvfp4_pair(16, 256, 512, seed, worked_row=True)


def decode(M: int, seed: int = SEED_BASE + 2, N: int = 8192, K: int = 8192):
    """bf16 activations [M, K] (torch) and float32 weights [N, K] (numpy)."""
    a = normal(rng_for(seed, 1), (M, K), 1.0)
    return to_bf16(a), int4_weights(N, K, seed)


def moe(seed: int = SEED_BASE + 3, M: int = 256, N: int = 2048, K: int = 7168):
    """bf16 A [M, K] (torch) and float32 B [N, K] (numpy)."""
    a, b = mxfp4_pair(M, N, K, seed)
    return to_bf16(a), b


def prefill_activations(seed: int = SEED_BASE + 4, M: int = 8192, K: int = 8192):
    """The prefill activations alone: bf16 [M, K] (torch), N(0, 1) with 0.5% of
    the channels scaled by 20."""
    a = normal(rng_for(seed, 1), (M, K), 1.0)
    scale_channels(rng_for(seed, 5), a)
    return to_bf16(a)


def prefill(seed: int = SEED_BASE + 4, M: int = 8192, N: int = 28672, K: int = 8192):
    """bf16 A [M, K] (torch) and float32 B [N, K] (numpy)."""
    a = prefill_activations(seed, M, K)
    b = normal(rng_for(seed, 2), (N, K), 0.02)
    return a, b


def route_top_k(T: int, E: int, top_k: int, seed: int, bias_std: float = 0.2,
                empty_expert: int | None = -1):
    """Seeded routing: logits N(0,1)[T, E] + b_e; the top-k experts per token
    (ties go to the lower expert id).  Softmax is monotone, so ranking the
    logits ranks the softmax probabilities.  Returns (expert_offsets [E+1],
    row_token [T*top_k]) with rows grouped by expert and, within an expert,
    in ascending token order."""
    rng = rng_for(seed, 7)
    bias = rng.standard_normal(E) * bias_std
    if empty_expert is not None and E > 0:
        bias[empty_expert] = -1e4
    logits = rng.standard_normal((T, E)) + bias[None, :]
    order = np.argsort(-logits, axis=1, kind="stable")[:, :top_k]
    experts = order.reshape(-1)
    tokens = np.repeat(np.arange(T, dtype=np.int64), top_k)
    perm = np.lexsort((tokens, experts))
    counts = np.bincount(experts, minlength=E)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return offsets, tokens[perm].astype(np.int32)


def grouped(seed: int = SEED_BASE + 5, T: int = 4096, E: int = 64, N: int = 2048,
            K: int = 7168, top_k: int = 8, experts: bool = True):
    """bf16 tokens [T, K] (torch), float32 expert weights [E, N, K] (numpy, or
    None when ``experts`` is False), expert offsets and the routed token ids."""
    tok = to_bf16(normal(rng_for(seed, 1), (T, K), 1.0))
    w = None
    if experts:
        w = np.empty((E, N, K), dtype=np.float32)
        for e in range(E):
            w[e] = normal(rng_for(seed, 100 + e), (N, K), 0.02)
    offsets, row_token = route_top_k(T, E, top_k, seed)
    return tok, w, offsets, row_token


def expert_weight(seed: int, e: int, N: int, K: int) -> np.ndarray:
    """Expert e's float32 weight, drawn exactly as :func:`grouped` draws it."""
    return normal(rng_for(seed, 100 + e), (N, K), 0.02)
