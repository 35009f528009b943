"""Seeded synthetic inputs for the batched decode step.

This module only draws random numbers and lays them out in the canonical byte
formats the library and the oracle both consume.  It holds none of the decode
step's arithmetic (no dequantisation, no matmul, no normalisation), so that the
CUDA path and the CPU oracle can share their inputs without sharing any code.

Workload shapes follow the two model families the batched-decode pages run:
a tiny one-layer model small enough for a pure fp64 oracle, and a
Llama-3-8B-shaped dense model (32 layers, hidden 4096, 32 query / 8 KV heads
of 128, SwiGLU FFN 14336, vocabulary 128256).  All weights are Q8_0: blocks of
32 consecutive input-dimension values of one output row, stored as a
little-endian fp16 scale ``d`` followed by 32 int8 quants (34 bytes), so that
``value = q * d``.  Quants are uniform over the integers in [-127, 127]; scales
are ``fp16(|z| / 127)`` with ``z ~ N(0, 0.02^2)``.  Norm weights are fp32 ones
(the workloads' own weights); ``norm_weights`` draws non-unit ones, different
for every layer, for extra parity cases.  Pre-filled KV rows are fp16 draws of
N(0, 1).

Every tensor has its own substream, keyed by ``(seed, name)``, so any piece can
be regenerated on its own (the oracle regenerates only the sessions it checks).
"""
from __future__ import annotations

import os
import zlib
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

Q8_BLOCK = 32          # values per Q8_0 block
Q8_BLOCK_BYTES = 34    # fp16 scale + 32 int8 quants


@dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float
    rms_eps: float

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def matrix_shapes(self) -> dict[str, tuple[int, int]]:
        """(rows, cols) of every per-layer Q8_0 matrix, in [out][in] order."""
        return {
            "attn_q": (self.q_dim, self.hidden),
            "attn_k": (self.kv_dim, self.hidden),
            "attn_v": (self.kv_dim, self.hidden),
            "attn_output": (self.hidden, self.q_dim),
            "ffn_gate": (self.ffn, self.hidden),
            "ffn_up": (self.ffn, self.hidden),
            "ffn_down": (self.hidden, self.ffn),
        }

    def weight_bytes(self) -> int:
        """Q8_0 bytes of every matrix read once per step (embedding rows excluded)."""
        per_layer = sum(r * c for r, c in self.matrix_shapes().values())
        total = per_layer * self.n_layers + self.vocab * self.hidden  # + lm_head
        return total * Q8_BLOCK_BYTES // Q8_BLOCK


TINY = ModelShape("tiny-1L-h256", 1, 256, 4, 2, 64, 768, 512, 10000.0, 1e-5)
# 128-wide heads (the Q8_0 KV cache's head size), 2 layers, 4 query heads per KV head.
TINY_HD128 = ModelShape("tiny-2L-h256-hd128", 2, 256, 4, 1, 128, 768, 512, 10000.0, 1e-5)
# A vocabulary of 32000 (1000 row groups of the lm_head, which no whole number of
# groups per SM covers evenly), so the head runs on the stream schedule, as at
# the 8B shape, while the rest of the model stays tiny.
TINY_WIDE_VOCAB = ModelShape("tiny-1L-h256-v32000", 1, 256, 4, 2, 64, 768, 32000, 10000.0, 1e-5)
LLAMA3_8B = ModelShape("llama3-8b-shaped", 32, 4096, 32, 8, 128, 14336, 128256, 500000.0, 1e-5)


def substream(seed: int, *names) -> np.random.Generator:
    """An independent generator for one named tensor under a run seed."""
    key = [int(seed) & 0xFFFFFFFF] + [zlib.crc32(str(n).encode()) for n in names]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(key)))


def q8_0_matrix(seed: int, name: str, rows: int, cols: int) -> np.ndarray:
    """Canonical Q8_0 bytes, uint8 [rows][cols/32][34]."""
    if cols % Q8_BLOCK:
        raise ValueError(f"{name}: cols={cols} is not a multiple of {Q8_BLOCK}")
    rng = substream(seed, name)
    nb = cols // Q8_BLOCK
    qs = rng.integers(-127, 128, size=(rows, nb, Q8_BLOCK), dtype=np.int8)
    z = rng.standard_normal(size=(rows, nb)) * 0.02
    d = (np.abs(z) / 127.0).astype(np.float16)
    out = np.empty((rows, nb, Q8_BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = d.view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 2:] = qs.view(np.uint8)
    return out


def q8_0_from_parts(d: np.ndarray, qs: np.ndarray) -> np.ndarray:
    """Lay out given fp16 scales [rows][nb] and int8 quants [rows][nb][32] as canonical Q8_0."""
    d = np.asarray(d, dtype=np.float16)
    qs = np.asarray(qs, dtype=np.int8)
    rows, nb = d.shape
    out = np.empty((rows, nb, Q8_BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = d.view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 2:] = qs.view(np.uint8).reshape(rows, nb, Q8_BLOCK)
    return out


def q8_0_split(m: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Inverse of q8_0_from_parts: (fp16 scales [rows][nb], int8 quants [rows][nb][32])."""
    d = np.ascontiguousarray(m[:, :, 0:2]).view(np.float16)[:, :, 0]
    qs = np.ascontiguousarray(m[:, :, 2:]).view(np.int8)
    return d, qs


def model_weights(shape: ModelShape, seed: int = 0, threads: int | None = None) -> dict:
    """All weights of a model: Q8_0 matrices plus fp32 norm weights (ones).

    Keys: ``tok_embd``, ``output``, ``output_norm`` and, per layer ``l``,
    ``blk.{l}.{attn_q,attn_k,attn_v,attn_output,ffn_gate,ffn_up,ffn_down,attn_norm,ffn_norm}``.
    """
    jobs = [("tok_embd", shape.vocab, shape.hidden), ("output", shape.vocab, shape.hidden)]
    for l in range(shape.n_layers):
        for m, (r, c) in shape.matrix_shapes().items():
            jobs.append((f"blk.{l}.{m}", r, c))
    threads = threads or min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(threads) as ex:
        mats = list(ex.map(lambda j: q8_0_matrix(seed, *j), jobs))
    w = {name: m for (name, _, _), m in zip(jobs, mats)}
    w["output_norm"] = np.ones(shape.hidden, dtype=np.float32)
    for l in range(shape.n_layers):
        w[f"blk.{l}.attn_norm"] = np.ones(shape.hidden, dtype=np.float32)
        w[f"blk.{l}.ffn_norm"] = np.ones(shape.hidden, dtype=np.float32)
    return w


def norm_weights(shape: ModelShape, seed: int = 0, spread: float = 0.1) -> dict:
    """Non-unit fp32 norm weights, ``1 + spread * N(0, 1)``, one seeded vector per
    (layer, norm) and one for the output norm, all different.

    Keys as in ``model_weights``; ``dict(model_weights(...), **norm_weights(...))``
    gives the same matrices with these norms (a parity case beside the
    workloads' unit norms, so that a kernel dropping the weight, or reading the
    wrong layer's, cannot pass)."""
    def draw(name):
        z = substream(seed, "norm", name).standard_normal(shape.hidden)
        return (1.0 + spread * z).astype(np.float32)

    w = {"output_norm": draw("output_norm")}
    for l in range(shape.n_layers):
        w[f"blk.{l}.attn_norm"] = draw(f"blk.{l}.attn_norm")
        w[f"blk.{l}.ffn_norm"] = draw(f"blk.{l}.ffn_norm")
    return w


def normal_fp16(rng: np.random.Generator, shape) -> np.ndarray:
    """fp16 draws of N(0,1), returned as their uint16 bit patterns."""
    return rng.standard_normal(size=shape, dtype=np.float32).astype(np.float16).view(np.uint16)


def kv_prefill(shape: ModelShape, seed: int, session: int, length: int,
               threads: int | None = None) -> tuple[np.ndarray, np.ndarray]:
    """Pre-filled KV of one session: K and V as fp16 bits, uint16 [L][n_kv][length][hd].

    Each (session, layer) pair has its own substream, so a session's KV does not
    depend on how many other sessions exist.
    """
    L, nkv, hd = shape.n_layers, shape.n_kv_heads, shape.head_dim
    k = np.empty((L, nkv, length, hd), dtype=np.uint16)
    v = np.empty((L, nkv, length, hd), dtype=np.uint16)

    def fill(l):
        rng = substream(seed, "kv", session, l)
        k[l] = normal_fp16(rng, (nkv, length, hd))
        v[l] = normal_fp16(rng, (nkv, length, hd))

    threads = threads or min(16, os.cpu_count() or 1)
    if L > 1 and length * nkv * hd > (1 << 16):
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(L)))
    else:
        for l in range(L):
            fill(l)
    return k, v


def tokens(seed: int, name: str, n: int, vocab: int) -> np.ndarray:
    """int32 tokens uniform over [0, vocab)."""
    return substream(seed, "tokens", name).integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def activations_fp16(seed: int, name: str, m: int, k: int) -> np.ndarray:
    """fp16 activations ~N(0,1) as uint16 bits [m][k] (isolated mmvq workload)."""
    return normal_fp16(substream(seed, "act", name), (m, k))


def ragged_lengths(seed: int, name: str, n: int, lo: int, hi: int) -> np.ndarray:
    """int32 lengths uniform over the integers in [lo, hi] (ragged attention workload)."""
    return substream(seed, "len", name).integers(lo, hi + 1, size=n, dtype=np.int64).astype(np.int32)


def f32_normal(seed: int, name: str, shape) -> np.ndarray:
    """fp32 draws of N(0,1) (new q/k/v rows of the isolated attention workload)."""
    return substream(seed, "f32", name).standard_normal(size=shape, dtype=np.float32)


# ---------------------------------------------------------------------------
# The workloads, as data.  Sizes and mixes follow the configurations the decode
# path is measured on; the names say what each one is.
# ---------------------------------------------------------------------------
TINY_CASE = dict(shape=TINY, sessions=2, prefill=(17, 40), steps=4, seed=0)
MMVQ_CASE = dict(matrices=((4096, 4096), (14336, 4096)), rows_m=(1, 2, 4, 8, 16), seed=0)
TINY_KV_Q8_CASE = dict(shape=TINY_HD128, sessions=3, prefill=(17, 64, 70), steps=6, seed=0)
RAGGED_ATTN_CASE = dict(n_heads=32, n_kv_heads=8, head_dim=128, sessions=8, max_ctx=32768, seed=0)
DENSE_8B_CASE = dict(shape=LLAMA3_8B, batch=(1, 2, 4, 8, 16), prefill=1238, capacity=2048,
                     steps=128, seed=0)
LONG_CTX_8B_CASE = dict(shape=LLAMA3_8B, sessions=8, capacity=32768, prefill_base=25704,
                        prefill_stagger=1000, steps=64, seed=0)
