"""Python binding of libkd.so, the batched multi-session decode step for GB300.

Argument marshalling only: every function here has the name of the C entry
point it calls (include/kd.h), converts numpy arrays / torch tensors / streams
into pointers, and raises KdError on a non-zero status.  All the step's work
runs in the library's CUDA kernels; there is no fallback path.  PyTorch is used
only to hand over device memory and streams.
"""
from __future__ import annotations

import ctypes as C
from pathlib import Path

import numpy as np

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libkd.so"

KD_MAX_BATCH = 16
KD_ATTN_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024
KD_FLAG_NO_GRAPH = 1
KD_FLAG_SCHEDULE_STREAM = 2
KD_FLAG_SCHEDULE_GROUP = 4
KD_FLAG_FUSED_NORM = 32
KD_FLAG_UNFUSED = 64
KD_FLAG_KV_Q8_0 = 128
STATUS = {0: "KD_OK", -1: "KD_ERR_INVALID_ARG", -2: "KD_ERR_OOM", -3: "KD_ERR_CUDA",
          -4: "KD_ERR_NO_FREE_SLOT", -5: "KD_ERR_BAD_SESSION", -6: "KD_ERR_POSITION",
          -7: "KD_ERR_BATCH", -8: "KD_ERR_UNSUPPORTED", -9: "KD_ERR_DEVICE"}


class KdError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.name = STATUS.get(status, str(status))


class KdConfig(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("hidden", C.c_int32), ("n_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn", C.c_int32),
                ("vocab", C.c_int32), ("rope_theta", C.c_float), ("rms_eps", C.c_float),
                ("max_sessions", C.c_int32), ("max_ctx", C.c_int32), ("flags", C.c_int32)]


_vp = C.c_void_p
_vpp = C.POINTER(C.c_void_p)
_fp = C.POINTER(C.c_float)
_fpp = C.POINTER(_fp)


class KdWeights(C.Structure):
    _fields_ = [("tok_embd", _vp), ("output", _vp), ("output_norm", _fp),
                ("wq", _vpp), ("wk", _vpp), ("wv", _vpp), ("wo", _vpp),
                ("w_gate", _vpp), ("w_up", _vpp), ("w_down", _vpp),
                ("attn_norm", _fpp), ("ffn_norm", _fpp)]


class KdSampleParams(C.Structure):
    _fields_ = [("temperature", C.c_float), ("reserved", C.c_uint32), ("seed", C.c_uint64), ("counter", C.c_uint64)]


def sample_params(temperatures, seeds, counters):
    """A host array of kd_sample_params from per-row temperatures, seeds and counters."""
    t = list(np.asarray(temperatures, dtype=np.float32).reshape(-1))
    arr = (KdSampleParams * len(t))()
    for i, (tt, sd, ct) in enumerate(zip(t, seeds, counters)):
        arr[i] = KdSampleParams(float(tt), 0, int(sd), int(ct))
    return arr


_lib = None


def lib():
    """Load libkd.so.  It must have been built (build.build()); nothing else will run."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise ImportError(f"{LIB_PATH} is missing: build it with session_decode_step_gb300.build.build()")
        L = C.CDLL(str(LIB_PATH))
        i32, i32p = C.c_int32, C.POINTER(C.c_int32)
        sig = {
            "kd_model_load": [C.POINTER(KdConfig), C.POINTER(KdWeights), C.POINTER(_vp)],
            "kd_model_free": [_vp],
            "kd_session_bind": [_vp, i32p],
            "kd_session_free": [_vp, i32],
            "kd_session_load_kv": [_vp, i32, _vp, _vp, i32, _vp],
            "kd_session_length": [_vp, i32, i32p],
            "kd_decode_step": [_vp, i32p, i32p, i32p, i32, _vp, _vp, _vp],
            "kd_debug_capture_hidden": [_vp, _vp],
            "kd_debug_layer": [_vp, i32, i32p, i32p, i32, _vp, _vp, _vp],
            "kd_device_status": [_vp, i32p],
            "kd_debug_inject_wait_timeout": [_vp, i32],
            "kd_q8_matrix_status": [_vp, i32p],
            "kd_attn_device_status": [_vp, i32p, _vp],
            "kd_profile_enable": [_vp, i32],
            "kd_profile_read": [_vp, i32p, C.POINTER(C.c_double)],
            "kd_profile_timeline": [_vp, _vp, i32, i32p],
            "kd_q8_matrix_create": [_vp, i32, i32, C.POINTER(_vp)],
            "kd_q8_matrix_free": [_vp],
            "kd_mmvq": [_vp, _vp, i32, _vp, _vp],
            "kd_argmax": [_vp, i32, i32, _vp, _vp, _vp],
            "kd_sample": [_vp, i32, i32, _vp, _vp, _vp, _vp],
            "kd_decode_step_sampled": [_vp, i32p, i32p, i32p, i32, _vp, _vp, _vp, _vp],
            "kd_mmvq_schedule": [i32, i32, i32, i32p, i32p, i32p],
            "kd_attn_append_decode": [_vp, _vp, _vp, _vp, _vp, i32p, i32p, i32, i32, i32, i32, i32,
                                      i32, _vp, _vp, C.c_size_t, _vp],
            "kd_attn_append_decode_noalloc": [_vp, _vp, _vp, _vp, _vp, i32p, i32p, i32, i32, i32, i32, i32,
                                              i32, _vp, _vp],
            "kd_kv_q8_quantize": [_vp, C.c_int64, _vp, _vp, _vp],
            "kd_debug_fail_alloc": [i32, i32p],
            "kd_attn_append_decode_q8": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, i32p, i32p, i32, i32, i32, i32, i32,
                                         _vp, _vp, C.c_size_t, _vp],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = C.c_int32
        L.kd_last_error.argtypes = []
        L.kd_last_error.restype = C.c_char_p
        L.kd_attn_workspace_bytes.argtypes = [i32, i32, i32, i32]
        L.kd_attn_workspace_bytes.restype = C.c_size_t
        _lib = L
    return _lib


def kd_last_error() -> str:
    return lib().kd_last_error().decode()


def _check(status: int):
    if status != 0:
        raise KdError(status, kd_last_error())


def _ptr(obj):
    """Address of a numpy array, a torch tensor, an int, or None."""
    if obj is None:
        return None
    if isinstance(obj, int):
        return obj
    if isinstance(obj, np.ndarray):
        if not obj.flags["C_CONTIGUOUS"]:
            raise ValueError("arrays passed to libkd must be C-contiguous")
        return obj.ctypes.data
    if hasattr(obj, "data_ptr"):
        if not obj.is_contiguous():
            raise ValueError("tensors passed to libkd must be contiguous")
        return obj.data_ptr()
    raise TypeError(f"cannot take the address of {type(obj)}")


def _stream(stream):
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _i32(a, n=None):
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int32).reshape(-1))
    if n is not None and arr.size != n:
        raise ValueError(f"expected {n} entries, got {arr.size}")
    return arr


# ----------------------------------------------------------------- model ---
def make_config(shape, max_sessions: int, max_ctx: int, flags: int = 0) -> KdConfig:
    """A kd_config for a model shape (anything with the ModelShape fields)."""
    return KdConfig(shape.n_layers, shape.hidden, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                    shape.ffn, shape.vocab, shape.rope_theta, shape.rms_eps, max_sessions, max_ctx,
                    flags)


def kd_model_load(cfg: KdConfig, weights: dict):
    """Load a model from host weights keyed like the synthetic generator's output."""
    L = cfg.n_layers

    def mats(name):
        return (_vp * L)(*[_ptr(weights[f"blk.{l}.{name}"]) for l in range(L)])

    keep = []  # arrays converted here must outlive the call

    def f32(a):
        a = np.ascontiguousarray(a, dtype=np.float32)
        keep.append(a)
        return C.cast(_ptr(a), _fp)

    def norms(name):
        return (_fp * L)(*[f32(weights[f"blk.{l}.{name}"]) for l in range(L)])
    w = KdWeights(_ptr(weights["tok_embd"]), _ptr(weights["output"]),
                  f32(weights["output_norm"]),
                  mats("attn_q"), mats("attn_k"), mats("attn_v"), mats("attn_output"),
                  mats("ffn_gate"), mats("ffn_up"), mats("ffn_down"),
                  norms("attn_norm"), norms("ffn_norm"))
    h = _vp()
    _check(lib().kd_model_load(C.byref(cfg), C.byref(w), C.byref(h)))
    return h


def kd_model_free(m):
    _check(lib().kd_model_free(m))


def kd_session_bind(m) -> int:
    out = C.c_int32()
    _check(lib().kd_session_bind(m, C.byref(out)))
    return out.value


def kd_session_free(m, session_id: int):
    _check(lib().kd_session_free(m, int(session_id)))


def kd_session_load_kv(m, session_id: int, k, v, length: int, stream=None):
    """k, v: [n_layers][n_kv][length][head_dim] fp16 (numpy uint16/float16 or a torch tensor)."""
    _check(lib().kd_session_load_kv(m, int(session_id), _ptr(k), _ptr(v), int(length), _stream(stream)))


def kd_session_length(m, session_id: int) -> int:
    out = C.c_int32()
    _check(lib().kd_session_length(m, int(session_id), C.byref(out)))
    return out.value


def kd_decode_step(m, session_ids, tokens, positions, logits_out=None, argmax_out=None, stream=None):
    """One batched step.  logits_out / argmax_out: device tensors (float32 [B][V], int32 [B]) or None."""
    ids = _i32(session_ids)
    B = ids.size
    tok, pos = _i32(tokens, B), _i32(positions, B)
    i32p = C.POINTER(C.c_int32)
    _check(lib().kd_decode_step(m, ids.ctypes.data_as(i32p), tok.ctypes.data_as(i32p),
                                pos.ctypes.data_as(i32p), B, _ptr(logits_out), _ptr(argmax_out),
                                _stream(stream)))


def kd_decode_step_sampled(m, session_ids, tokens, positions, params, logits_out=None, token_out=None, stream=None):
    """One batched step with device temperature sampling: params from sample_params(); token_out a
    device int32 [B] tensor (required)."""
    ids = _i32(session_ids)
    B = ids.size
    tok, pos = _i32(tokens, B), _i32(positions, B)
    if len(params) != B:
        raise ValueError(f"expected {B} sampling parameter rows, got {len(params)}")
    i32p = C.POINTER(C.c_int32)
    _check(lib().kd_decode_step_sampled(m, ids.ctypes.data_as(i32p), tok.ctypes.data_as(i32p),
                                        pos.ctypes.data_as(i32p), B, C.cast(params, _vp), _ptr(logits_out),
                                        _ptr(token_out), _stream(stream)))


def kd_debug_capture_hidden(m, buf):
    _check(lib().kd_debug_capture_hidden(m, _ptr(buf)))


def kd_debug_layer(m, layer: int, session_ids, positions, x_in, x_out, stream=None):
    ids = _i32(session_ids)
    pos = _i32(positions, ids.size)
    i32p = C.POINTER(C.c_int32)
    _check(lib().kd_debug_layer(m, int(layer), ids.ctypes.data_as(i32p), pos.ctypes.data_as(i32p), ids.size,
                                _ptr(x_in), _ptr(x_out), _stream(stream)))


def kd_device_status(m) -> int:
    out = C.c_int32()
    _check(lib().kd_device_status(m, C.byref(out)))
    return out.value


KERNEL_CLASSES = ("embed", "rmsnorm", "qkv", "attn_split", "attn_combine", "wo", "gate_up", "down",
                  "lm_head", "argmax")


def kd_debug_inject_wait_timeout(m, kernel_class: str):
    """Make one bounded wait of the next step's first `kernel_class` launch run out
    (a test of the device fault path; nothing faults or hangs)."""
    _check(lib().kd_debug_inject_wait_timeout(m, KERNEL_CLASSES.index(kernel_class)))


def kd_profile_enable(m, on: bool = True):
    _check(lib().kd_profile_enable(m, 1 if on else 0))


KD_TIMELINE_CTAS = 1024


def kd_profile_timeline(m, buf, max_launches: int = 0):
    """Turn the per-CTA timeline on (buf: device uint64 [max_launches][KD_TIMELINE_CTAS][4],
    zeroed) or off (buf None).  Returns the kernel class name of each launch index."""
    n = int(max_launches) if buf is not None else 0
    cls = (C.c_int32 * max(n, 1))()
    _check(lib().kd_profile_timeline(m, _ptr(buf), n, cls if n else None))
    return [KERNEL_CLASSES[c] if c >= 0 else None for c in cls[:n]]


def kd_profile_read(m) -> dict:
    """{kernel class: (launches, total ms)} since the previous read."""
    n = len(KERNEL_CLASSES)
    launches = (C.c_int32 * n)()
    ms = (C.c_double * n)()
    _check(lib().kd_profile_read(m, launches, ms))
    return {k: (launches[i], ms[i]) for i, k in enumerate(KERNEL_CLASSES)}


# -------------------------------------------------------------- op level ---
def kd_q8_matrix_create(q8_0: np.ndarray):
    """q8_0: canonical uint8 [rows][cols/32][34] in host memory."""
    rows, nb, _ = q8_0.shape
    h = _vp()
    _check(lib().kd_q8_matrix_create(_ptr(np.ascontiguousarray(q8_0)), rows, nb * 32, C.byref(h)))
    return h


def kd_q8_matrix_free(w):
    _check(lib().kd_q8_matrix_free(w))


def kd_mmvq(w, x, m: int, y, stream=None):
    _check(lib().kd_mmvq(w, _ptr(x), int(m), _ptr(y), _stream(stream)))


def kd_q8_matrix_status(w) -> int:
    out = C.c_int32()
    _check(lib().kd_q8_matrix_status(w, C.byref(out)))
    return out.value


KD_ARGMAX_WORKSPACE_BYTES = 256


def kd_mmvq_schedule(rows: int, cols: int, num_sms: int):
    """(mode, warps, share) the library picks for a rows x cols Q8_0 matrix on num_sms SMs
    (host only): mode 1 = group, 0 = stream."""
    mode, warps, share = C.c_int32(), C.c_int32(), C.c_int32()
    _check(lib().kd_mmvq_schedule(int(rows), int(cols), int(num_sms), C.byref(mode), C.byref(warps), C.byref(share)))
    return mode.value, warps.value, share.value


def kd_argmax(logits, B: int, V: int, out, workspace, stream=None):
    """logits: device fp32 [B][V]; out: device int32 [B]; workspace: KD_ARGMAX_WORKSPACE_BYTES of device memory."""
    _check(lib().kd_argmax(_ptr(logits), int(B), int(V), _ptr(out), _ptr(workspace), _stream(stream)))


KD_SAMPLE_WORKSPACE_BYTES = 1024


def kd_sample(logits, B: int, V: int, params, out, workspace, stream=None):
    """logits: device fp32 [B][V]; params: sample_params(...) of B rows; out: device int32 [B];
    workspace: KD_SAMPLE_WORKSPACE_BYTES of device memory."""
    if len(params) != B:
        raise ValueError(f"expected {B} sampling parameter rows, got {len(params)}")
    _check(lib().kd_sample(_ptr(logits), int(B), int(V), C.cast(params, _vp), _ptr(out), _ptr(workspace),
                           _stream(stream)))


def kd_attn_workspace_bytes(B: int, n_heads: int, head_dim: int, cap: int) -> int:
    return int(lib().kd_attn_workspace_bytes(B, n_heads, head_dim, cap))


def kd_attn_append_decode(q, k_new, v_new, k_cache, v_cache, slots, positions, n_heads, n_kv_heads,
                          head_dim, n_slots, cap, out, workspace, stream=None):
    sl = _i32(slots)
    B = sl.size
    ps = _i32(positions, B)
    i32p = C.POINTER(C.c_int32)
    nbytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else workspace.nbytes
    _check(lib().kd_attn_append_decode(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                       sl.ctypes.data_as(i32p), ps.ctypes.data_as(i32p), B, n_heads,
                                       n_kv_heads, head_dim, n_slots, cap, _ptr(out), _ptr(workspace),
                                       nbytes, _stream(stream)))


def kd_debug_fail_alloc(nth: int) -> int:
    """Arm (nth >= 1) or disarm (0) the allocation-failure switch of the next
    kd_model_load; returns the number of allocations the last load made."""
    out = C.c_int32()
    _check(lib().kd_debug_fail_alloc(int(nth), C.byref(out)))
    return out.value


def kd_kv_q8_quantize(src, quants, scales, stream=None):
    """Rows of 128 fp32 values (device [rows][128]) into Q8_0 quants (uint8
    [rows][128], q + 128) and fp16 block scales ([rows][4], as int16/uint16 bits)."""
    rows = src.numel() // 128
    _check(lib().kd_kv_q8_quantize(_ptr(src), rows, _ptr(quants), _ptr(scales), _stream(stream)))


def kd_attn_append_decode_q8(q, k_new, v_new, k_quants, k_scales, v_quants, v_scales, slots, positions, n_heads,
                             n_kv_heads, n_slots, cap, out, workspace, stream=None):
    """kd_attn_append_decode over a Q8_0 cache of head_dim 128 (see include/kd.h)."""
    sl = _i32(slots)
    B = sl.size
    ps = _i32(positions, B)
    i32p = C.POINTER(C.c_int32)
    nbytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else workspace.nbytes
    _check(lib().kd_attn_append_decode_q8(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_quants), _ptr(k_scales),
                                          _ptr(v_quants), _ptr(v_scales), sl.ctypes.data_as(i32p),
                                          ps.ctypes.data_as(i32p), B, n_heads, n_kv_heads, n_slots, cap, _ptr(out),
                                          _ptr(workspace), nbytes, _stream(stream)))


def kd_attn_device_status(workspace=None, stream=None) -> int:
    """Fault word of the last attention call given `workspace` (None: the last
    allocation-free call on the current device)."""
    out = C.c_int32()
    _check(lib().kd_attn_device_status(_ptr(workspace), C.byref(out), _stream(stream)))
    return out.value


def kd_attn_append_decode_noalloc(q, k_new, v_new, k_cache, v_cache, slots, positions, n_heads, n_kv_heads,
                                  head_dim, n_slots, cap, out, stream=None):
    """kd_attn_append_decode with its scratch in the library's fixed device array
    (no workspace argument, no allocation); see include/kd.h for the limits."""
    sl = _i32(slots)
    B = sl.size
    ps = _i32(positions, B)
    i32p = C.POINTER(C.c_int32)
    _check(lib().kd_attn_append_decode_noalloc(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                               sl.ctypes.data_as(i32p), ps.ctypes.data_as(i32p), B, n_heads,
                                               n_kv_heads, head_dim, n_slots, cap, _ptr(out), _stream(stream)))
