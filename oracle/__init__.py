"""CPU oracle of the batched decode step (ctypes wrapper around kd_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library, and the library never imports it.

Every function is a thin marshalling layer over the C file, which states what
it computes and which passage of the pages each part follows.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "kd_oracle.c"
_LIB = _HERE / "liboracle.so"
_lib = None


def build(force: bool = False) -> Path:
    """Compile kd_oracle.c into liboracle.so next to it (gcc, OpenMP, no fast-math)."""
    if _LIB.exists() and not force and _LIB.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB
    base = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
            str(_SRC), "-o", str(_LIB) + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)  # serial fallback
    os.replace(str(_LIB) + ".tmp", _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = C.CDLL(str(_LIB))
        _declare(_lib)
    return _lib


_u8p = C.POINTER(C.c_uint8)
_f32p = C.POINTER(C.c_float)
_f64p = C.POINTER(C.c_double)
_u16p = C.POINTER(C.c_uint16)
_i32p = C.POINTER(C.c_int32)


class KdoConfig(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("hidden", C.c_int32), ("n_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn", C.c_int32),
                ("vocab", C.c_int32), ("rope_theta", C.c_double), ("rms_eps", C.c_double),
                ("kv_q8_0", C.c_int32)]


class KdoWeights(C.Structure):
    _fields_ = [("tok_embd", _u8p), ("output", _u8p), ("output_norm", _f32p),
                ("wq", C.POINTER(_u8p)), ("wk", C.POINTER(_u8p)), ("wv", C.POINTER(_u8p)),
                ("wo", C.POINTER(_u8p)), ("w_gate", C.POINTER(_u8p)), ("w_up", C.POINTER(_u8p)),
                ("w_down", C.POINTER(_u8p)), ("attn_norm", C.POINTER(_f32p)),
                ("ffn_norm", C.POINTER(_f32p))]


def _declare(L):
    L.kdo_half_to_double.argtypes = [C.c_uint16]
    L.kdo_half_to_double.restype = C.c_double
    L.kdo_double_to_half.argtypes = [C.c_double]
    L.kdo_double_to_half.restype = C.c_uint16
    L.kdo_q8_0_dequant_row.argtypes = [_u8p, C.c_int32, _f64p]
    L.kdo_matvec_q8_0.argtypes = [_u8p, C.c_int32, C.c_int32, _f64p, _f64p]
    L.kdo_rmsnorm_f16.argtypes = [_f64p, _f32p, C.c_int32, C.c_double, _f64p]
    L.kdo_rope_neox.argtypes = [_f64p, C.c_int32, C.c_int32, C.c_double]
    L.kdo_attention_head.argtypes = [_f64p, _u16p, _u16p, C.c_int32, C.c_int32, C.c_int64,
                                     C.c_double, _f64p]
    L.kdo_q8_0_quantize_f32.argtypes = [_f32p, C.c_int32, _u8p]
    L.kdo_attention_head_q8.argtypes = [_f64p, _u8p, _u8p, C.c_int32, C.c_int32, C.c_int64, C.c_double, _f64p]
    L.kdo_silu.argtypes = [C.c_double]
    L.kdo_silu.restype = C.c_double
    L.kdo_argmax_f32.argtypes = [_f32p, C.c_int32]
    L.kdo_argmax_f32.restype = C.c_int32
    L.kdo_philox4x64_10.argtypes = [C.POINTER(C.c_uint64), C.POINTER(C.c_uint64), C.POINTER(C.c_uint64)]
    L.kdo_gumbel_perturbed.argtypes = [C.c_float, C.c_int32, C.c_float, C.c_uint64, C.c_uint64]
    L.kdo_gumbel_perturbed.restype = C.c_float
    L.kdo_sample_f32.argtypes = [_f32p, C.c_int32, C.c_float, C.c_uint64, C.c_uint64]
    L.kdo_sample_f32.restype = C.c_int32
    L.kdo_session_step.argtypes = [C.POINTER(KdoConfig), C.POINTER(KdoWeights), C.c_int32,
                                   C.c_int32, C.c_void_p, C.c_void_p, C.c_int32, _f32p, _f32p]
    L.kdo_session_step.restype = C.c_int32
    L.kdo_layer_step.argtypes = [C.POINTER(KdoConfig), C.POINTER(KdoWeights), C.c_int32, C.c_int32,
                                 C.c_void_p, C.c_void_p, C.c_int32, _f64p]
    L.kdo_layer_step.restype = C.c_int32
    L.kdo_decode_step.argtypes = [C.POINTER(KdoConfig), C.POINTER(KdoWeights), C.c_int32,
                                  _i32p, _i32p, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.c_int32,
                                  _f32p, _f32p, _i32p]
    L.kdo_decode_step.restype = C.c_int32


def _p(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(t)


# ---------------------------------------------------------------------------
# Single functions (used by the pins)
# ---------------------------------------------------------------------------
def half_to_double(h: int) -> float:
    return lib().kdo_half_to_double(int(h))


def double_to_half(x: float) -> int:
    return int(lib().kdo_double_to_half(float(x)))


def q8_0_dequant_row(row: np.ndarray, cols: int) -> np.ndarray:
    row = np.ascontiguousarray(row, dtype=np.uint8).reshape(-1)
    out = np.empty(cols, dtype=np.float64)
    lib().kdo_q8_0_dequant_row(_p(row, _u8p), cols, _p(out, _f64p))
    return out


def matvec_q8_0(W: np.ndarray, x: np.ndarray) -> np.ndarray:
    rows, nb, _ = W.shape
    W = np.ascontiguousarray(W)
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(rows, dtype=np.float64)
    lib().kdo_matvec_q8_0(_p(W, _u8p), rows, nb * 32, _p(x, _f64p), _p(y, _f64p))
    return y


def rmsnorm_f16(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty_like(x)
    lib().kdo_rmsnorm_f16(_p(x, _f64p), _p(w, _f32p), x.size, eps, _p(out, _f64p))
    return out


def rope_neox(u: np.ndarray, pos: int, theta: float) -> np.ndarray:
    u = np.array(u, dtype=np.float64, copy=True)
    lib().kdo_rope_neox(_p(u, _f64p), u.size, int(pos), float(theta))
    return u


def attention_head(q: np.ndarray, K16: np.ndarray, V16: np.ndarray) -> np.ndarray:
    """q [hd] float64; K16/V16 uint16 fp16 bits [t_kv][hd]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K16 = np.ascontiguousarray(K16, dtype=np.uint16)
    V16 = np.ascontiguousarray(V16, dtype=np.uint16)
    t, hd = K16.shape
    out = np.empty(hd, dtype=np.float64)
    lib().kdo_attention_head(_p(q, _f64p), _p(K16, _u16p), _p(V16, _u16p), t, hd, hd,
                             1.0 / np.sqrt(hd), _p(out, _f64p))
    return out


def q8_0_quantize_f32(x: np.ndarray) -> np.ndarray:
    """Canonical Q8_0 blocks (uint8 [n/32][34]) of fp32 values, quantised in fp32."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.empty((x.size // 32, 34), dtype=np.uint8)
    lib().kdo_q8_0_quantize_f32(_p(x, _f32p), x.size, _p(out, _u8p))
    return out


def attention_head_q8(q: np.ndarray, Kq: np.ndarray, Vq: np.ndarray) -> np.ndarray:
    """q [hd] float64; Kq/Vq uint8 Q8_0 rows [t_kv][hd/32][34]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    Kq = np.ascontiguousarray(Kq, dtype=np.uint8)
    Vq = np.ascontiguousarray(Vq, dtype=np.uint8)
    t = Kq.shape[0]
    hd = q.size
    out = np.empty(hd, dtype=np.float64)
    lib().kdo_attention_head_q8(_p(q, _f64p), _p(Kq, _u8p), _p(Vq, _u8p), t, hd, (hd // 32) * 34,
                                1.0 / np.sqrt(hd), _p(out, _f64p))
    return out


def silu(y: float) -> float:
    return lib().kdo_silu(float(y))


def argmax_f32(v: np.ndarray) -> int:
    v = np.ascontiguousarray(v, dtype=np.float32)
    return int(lib().kdo_argmax_f32(_p(v, _f32p), v.size))


def philox4x64_10(counter, key) -> list:
    """The four 64-bit words of the Philox4x64-10 block at `counter` (4 words) under `key` (2 words)."""
    c = (C.c_uint64 * 4)(*[int(x) for x in counter])
    k = (C.c_uint64 * 2)(*[int(x) for x in key])
    o = (C.c_uint64 * 4)()
    lib().kdo_philox4x64_10(c, k, o)
    return list(o)


def gumbel_perturbed(logit: float, v: int, temperature: float, seed: int, counter: int) -> float:
    return float(lib().kdo_gumbel_perturbed(float(logit), int(v), float(temperature), int(seed), int(counter)))


def sample_f32(logits: np.ndarray, temperature: float, seed: int, counter: int) -> int:
    """One temperature draw over an fp32 logit row (temperature <= 0: the greedy argmax)."""
    v = np.ascontiguousarray(logits, dtype=np.float32)
    return int(lib().kdo_sample_f32(_p(v, _f32p), v.size, float(temperature), int(seed), int(counter)))


# ---------------------------------------------------------------------------
# The model
# ---------------------------------------------------------------------------
class OracleModel:
    """Holds references to the host weights (canonical Q8_0) of one model."""

    def __init__(self, shape, weights: dict, kv_q8_0: bool = False):
        self.shape = shape
        self.w = weights
        self.kv_q8_0 = bool(kv_q8_0)
        s = shape
        self.cfg = KdoConfig(s.n_layers, s.hidden, s.n_heads, s.n_kv_heads, s.head_dim,
                             s.ffn, s.vocab, s.rope_theta, s.rms_eps, 1 if kv_q8_0 else 0)
        L = s.n_layers

        def arr(key, t):
            a = weights[key]
            assert a.flags["C_CONTIGUOUS"]
            return _p(a, t)

        def table(name, t):
            return (t * L)(*[arr(f"blk.{l}.{name}", t) for l in range(L)])

        self._tables = {n: table(n, _u8p) for n in
                        ("attn_q", "attn_k", "attn_v", "attn_output", "ffn_gate", "ffn_up",
                         "ffn_down")}
        self._tables["attn_norm"] = table("attn_norm", _f32p)
        self._tables["ffn_norm"] = table("ffn_norm", _f32p)
        t = self._tables
        self.cw = KdoWeights(arr("tok_embd", _u8p), arr("output", _u8p), arr("output_norm", _f32p),
                             t["attn_q"], t["attn_k"], t["attn_v"], t["attn_output"],
                             t["ffn_gate"], t["ffn_up"], t["ffn_down"], t["attn_norm"],
                             t["ffn_norm"])

    def new_cache(self, cap: int, k_prefill=None, v_prefill=None):
        """A session's KV cache, optionally pre-filled from fp16 bits [L][n_kv][n][hd]:
        fp16 [L][n_kv][cap][hd] (uint16 bits), or with kv_q8_0 Q8_0 rows
        [L][n_kv][cap][hd/32][34] (the pre-filled rows quantised from their fp16 values)."""
        s = self.shape
        if not self.kv_q8_0:
            k = np.zeros((s.n_layers, s.n_kv_heads, cap, s.head_dim), dtype=np.uint16)
            v = np.zeros_like(k)
            if k_prefill is not None:
                n = k_prefill.shape[2]
                k[:, :, :n] = k_prefill
                v[:, :, :n] = v_prefill
            return k, v
        nb = s.head_dim // 32
        k = np.zeros((s.n_layers, s.n_kv_heads, cap, nb, 34), dtype=np.uint8)
        v = np.zeros_like(k)
        if k_prefill is not None:
            n = k_prefill.shape[2]
            for src, dst in ((k_prefill, k), (v_prefill, v)):
                f = np.ascontiguousarray(src).view(np.float16).astype(np.float32)
                dst[:, :, :n] = q8_0_quantize_f32(f).reshape(s.n_layers, s.n_kv_heads, n, nb, 34)
        return k, v

    def layer_step(self, layer: int, pos: int, cache, cap: int, x: np.ndarray) -> np.ndarray:
        """One layer of one session: x (fp64 [hidden]) updated in place; cache = (k, v)."""
        k, v = cache
        s = self.shape
        row = (s.head_dim // 32) * 34 if self.kv_q8_0 else 2 * s.head_dim
        off = layer * s.n_kv_heads * cap * row
        kp = C.c_void_p(k.ctypes.data + off)
        vp = C.c_void_p(v.ctypes.data + off)
        rc = lib().kdo_layer_step(C.byref(self.cfg), C.byref(self.cw), layer, pos, kp, vp, cap,
                                  _p(x, _f64p))
        if rc != 0:
            raise ValueError(f"oracle layer step rejected its inputs (rc={rc})")
        return x

    def step(self, tokens, positions, caches, cap: int, want_hidden: bool = False):
        """One batched step.  caches: list of (k, v) per session, updated in place.

        Returns (logits [B][vocab] f32, argmax [B] i32, hidden [B][L+1][H] f32 or None).
        """
        s = self.shape
        B = len(tokens)
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        pos = np.ascontiguousarray(positions, dtype=np.int32)
        kp = (C.c_void_p * B)(*[c[0].ctypes.data for c in caches])
        vp = (C.c_void_p * B)(*[c[1].ctypes.data for c in caches])
        logits = np.empty((B, s.vocab), dtype=np.float32)
        am = np.empty(B, dtype=np.int32)
        hidden = np.empty((B, s.n_layers + 1, s.hidden), dtype=np.float32) if want_hidden else None
        rc = lib().kdo_decode_step(C.byref(self.cfg), C.byref(self.cw), B, _p(tok, _i32p),
                                   _p(pos, _i32p), kp, vp, cap, _p(logits, _f32p),
                                   _p(hidden, _f32p) if want_hidden else None, _p(am, _i32p))
        if rc != 0:
            raise ValueError(f"oracle step rejected its inputs (rc={rc})")
        return logits, am, hidden
