"""Seeded synthetic inputs for the canvas sampler.

This module only draws random inputs; it holds none of the sampler's arithmetic, so the
CUDA path (through the Python binding) and the fp64 oracle under ``oracle/`` can both take
their inputs from it without sharing any of the method.

The workloads follow the shapes of the DiffusionGemma pages: a canvas of 256 token slots
("A diffusion language model refines 256 tokens in 12 steps", sokufu.com article) and a
vocabulary of 262k (= 262,144) entries ("Sampling", technical report section 6). No
dataset is read: embeddings and hidden states are drawn from fixed distributions.

Input recipes (all generators are numpy PCG64, so every array is identical on x86 and Arm):

* ``E`` ~ N(0, 1/d) per element, rounded to bf16 (round-to-nearest-even) unless the
  workload is fp32.
* ``peaked`` hidden states: H_i = c_i * ln(V) * E[t_i] + xi_i with c_i ~ U[0.5, 4],
  xi_i ~ N(0, I_d) and t_i uniform in [0, V); rounded to bf16. The logit of t_i is then
  about c_i ln V while the other logits are about N(0, 1), so the probability of t_i is
  about 1 / (1 + 1.65 V^(1 - c_i)) and the confidences spread over (0, 1).
* ``target3`` hidden states (tiny fp32 case): H_i = 3 sqrt(d) E[t_i] + N(0, 1).
* ``standin`` loops draw W ~ N(0, 1/(2d)) in bf16, shape [d, 2d]; the hidden states are then
  computed inside the loop from the previous self-conditioning vector and the canvas.
* canvas tokens uniform in [0, V); lock mask, step counters and done flags start at 0.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

CANVAS_LEN = 256


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    L: int
    V: int
    d: int
    dtype: str  # "bf16" or "fp32": storage type of E and H
    seed: int  # data seed
    philox_seed: int  # seed of the sampler's counter-based generator
    h_mode: str  # "target3", "peaked" or "standin"
    steps: int = 1  # denoising steps the workload runs
    max_steps: int = 48
    top_k: int = 0
    T: tuple = (1.0, 1.0)  # per-sequence temperature: fixed value or U[lo, hi]
    tau: tuple = (0.9, 0.9)  # per-sequence lock threshold: fixed value or U[lo, hi]
    notes: str = field(default="", compare=False)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_fp32_b1_v4096_d256", 1, 256, 4096, 256, "fp32", seed=0, philox_seed=1,
                 h_mode="target3", steps=1, T=(1.0, 1.0), tau=(0.9, 0.9)),
        Workload("loop8_bf16_b1_v32768_d1024", 1, 256, 32768, 1024, "bf16", seed=7, philox_seed=7,
                 h_mode="peaked", steps=8, T=(1.0, 1.0), tau=(0.9, 0.9)),
        Workload("step_bf16_b1_v262144_d2816", 1, 256, 262144, 2816, "bf16", seed=11, philox_seed=11,
                 h_mode="peaked", steps=1, T=(1.0, 1.0), tau=(0.85, 0.85)),
        Workload("step_bf16_b8_v262144_d2816", 8, 256, 262144, 2816, "bf16", seed=23, philox_seed=23,
                 h_mode="peaked", steps=1, T=(0.7, 1.0), tau=(0.8, 0.95)),
        Workload("loop48_topk64_bf16_b4_v262144_d2816", 4, 256, 262144, 2816, "bf16", seed=42,
                 philox_seed=42, h_mode="standin", steps=48, top_k=64, T=(1.0, 1.0),
                 tau=(0.9, 0.9)),
    ]
}

# The workload the bench times: one sampler step over a B=1 canvas at the pages' vocabulary.
BENCH_WORKLOAD = "step_bf16_b1_v262144_d2816"


def scaled(w: Workload, *, V: int | None = None, d: int | None = None, B: int | None = None,
           L: int | None = None, name: str | None = None) -> Workload:
    """The same recipe at other sizes (for parity cases the oracle finishes quickly)."""
    V = w.V if V is None else V
    d = w.d if d is None else d
    B = w.B if B is None else B
    L = w.L if L is None else L
    tag = "" if L == w.L else f"_L{L}"
    return replace(w, V=V, d=d, B=B, L=L, name=name or f"{w.name}@B{B}_V{V}_d{d}{tag}")


# --------------------------------------------------------------------------------------
# bf16 storage helpers (bit patterns in uint16; numpy has no bf16 dtype)
# --------------------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------------------

_CHUNK_ROWS = 4096


def _rng(seed: int, tag: int, chunk: int = 0) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(tag), int(chunk)])


def _threads() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        n = os.cpu_count() or 1
    return max(1, min(16, n))


def gen_embeddings(w: Workload) -> np.ndarray:
    """E [V, d]: N(0, 1/d); bf16 bits (uint16) or float32 for fp32 workloads.

    Rows are drawn in fixed chunks of 4096, each from its own seeded stream, so the result
    does not depend on the number of threads used."""
    V, d = w.V, w.d
    out = np.empty((V, d), dtype=np.float32 if w.dtype == "fp32" else np.uint16)
    scale = np.float32(1.0 / math.sqrt(d))
    nchunks = (V + _CHUNK_ROWS - 1) // _CHUNK_ROWS

    def work(c):
        r0, r1 = c * _CHUNK_ROWS, min(V, (c + 1) * _CHUNK_ROWS)
        x = _rng(w.seed, 1, c).standard_normal((r1 - r0, d), dtype=np.float32)
        x *= scale
        out[r0:r1] = x if w.dtype == "fp32" else f32_to_bf16_bits(x)

    if nchunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def embeddings_f32(w: Workload, E: np.ndarray) -> np.ndarray:
    return E if w.dtype == "fp32" else bf16_bits_to_f32(E)


def gen_hidden(w: Workload, E: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """H [B, L, d] for fixed-H workloads, and the target tokens t [B, L] it points at."""
    B, L, V, d = w.B, w.L, w.V, w.d
    rng = _rng(w.seed, 2)
    t = rng.integers(0, V, size=(B, L), dtype=np.int64)
    Et = embeddings_f32(w, E[t.reshape(-1)]).reshape(B, L, d)
    xi = rng.standard_normal((B, L, d), dtype=np.float32)
    if w.h_mode == "target3":
        H = np.float32(3.0 * math.sqrt(d)) * Et + xi
        return (H.astype(np.float32) if w.dtype == "fp32" else f32_to_bf16_bits(H)), t.astype(np.int32)
    if w.h_mode in ("peaked", "standin"):
        c = rng.uniform(0.5, 4.0, size=(B, L, 1)).astype(np.float32)
        H = c * np.float32(math.log(V)) * Et + xi
        return (H.astype(np.float32) if w.dtype == "fp32" else f32_to_bf16_bits(H)), t.astype(np.int32)
    raise ValueError(w.h_mode)


def gen_standin_weight(w: Workload) -> np.ndarray:
    """W [d, 2d] bf16 bits, N(0, 1/(2d)): the stand-in for the model's hidden-state provider."""
    d = w.d
    x = _rng(w.seed, 3).standard_normal((d, 2 * d), dtype=np.float32)
    x *= np.float32(1.0 / math.sqrt(2 * d))
    return f32_to_bf16_bits(x)


def gen_sequence_params(w: Workload) -> tuple[np.ndarray, np.ndarray]:
    rng = _rng(w.seed, 4)
    lo, hi = w.T
    T = np.full(w.B, lo, np.float32) if lo == hi else rng.uniform(lo, hi, w.B).astype(np.float32)
    lo, hi = w.tau
    tau = np.full(w.B, lo, np.float32) if lo == hi else rng.uniform(lo, hi, w.B).astype(np.float32)
    return T, tau


def gen_canvas(w: Workload) -> np.ndarray:
    return _rng(w.seed, 5).integers(0, w.V, size=(w.B, w.L), dtype=np.int64).astype(np.int32)


def make_inputs(w: Workload | str, *, with_E: bool = True) -> dict:
    """All inputs of a workload as numpy arrays (E may be skipped and passed in later)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    E = gen_embeddings(w)
    T, tau = gen_sequence_params(w)
    inp = {
        "workload": w,
        "T": T,
        "tau": tau,
        "canvas": gen_canvas(w),
        "lock": np.zeros((w.B, w.L), np.uint8),
        "step": np.zeros(w.B, np.int32),
        "done": np.zeros(w.B, np.uint8),
        "seed": int(w.philox_seed),
    }
    if w.h_mode == "standin":
        inp["W"] = gen_standin_weight(w)
        inp["H"] = None
    else:
        inp["H"], inp["targets"] = gen_hidden(w, E)
    if with_E:
        inp["E"] = E
    return inp
