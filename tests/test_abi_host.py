"""The C-ABI library without a GPU: it builds, loads, exports every declared
symbol, and rejects bad arguments on the host before touching CUDA."""
import ctypes as C
import os
import re
import subprocess

import numpy as np
import pytest

import session_decode_step_gb300 as kd
import synth
from session_decode_step_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kd.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(kd_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 15, names
    out = subprocess.run(["nm", "-D", "--defined-only", str(kd.LIB_PATH)], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (kd_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared in kd.h but not exported: {missing}"
    for n in names:
        assert hasattr(lib, n)


def test_null_arguments_are_rejected(lib):
    assert lib.kd_model_load(None, None, None) == -1
    assert "null" in kd.kd_last_error()
    assert lib.kd_model_free(None) == -1
    assert lib.kd_session_bind(None, None) == -1
    assert lib.kd_session_free(None, 0) == -1
    assert lib.kd_decode_step(None, None, None, None, 1, None, None, None) == -1
    assert lib.kd_mmvq(None, None, 1, None, None) == -1
    assert lib.kd_q8_matrix_create(None, 32, 128, None) == -1
    out = C.c_int32()
    assert lib.kd_session_length(None, 0, C.byref(out)) == -1
    assert lib.kd_device_status(None, C.byref(out)) == -1


def test_unsupported_model_shapes_fail_before_cuda(lib):
    good = kd.make_config(synth.TINY, 2, 64)
    w = kd.KdWeights()
    h = C.c_void_p()
    for field, value in [("hidden", 200), ("hidden", 131072 + 128), ("head_dim", 96), ("n_kv_heads", 3),
                         ("ffn", 100), ("vocab", 500)]:
        cfg = kd.make_config(synth.TINY, 2, 64)
        setattr(cfg, field, value)
        st = lib.kd_model_load(C.byref(cfg), C.byref(w), C.byref(h))
        assert st in (-8, -1), (field, st)
    for field in ("n_layers", "max_sessions", "max_ctx"):
        cfg = kd.make_config(synth.TINY, 2, 64)
        setattr(cfg, field, 0)
        assert lib.kd_model_load(C.byref(cfg), C.byref(w), C.byref(h)) == -1
    # the Q8_0 KV cache needs 128-wide heads and an even slot capacity
    for shape, cap in ((synth.TINY, 64), (synth.TINY_HD128, 63)):
        cfg = kd.make_config(shape, 2, cap, kd.KD_FLAG_KV_Q8_0)
        assert lib.kd_model_load(C.byref(cfg), C.byref(w), C.byref(h)) == -8, (shape.name, cap)
    # a valid config with null weights is rejected on the host too
    assert lib.kd_model_load(C.byref(good), C.byref(w), C.byref(h)) == -1
    assert not h.value


def test_argmax_argument_checks(lib):
    fake = C.c_void_p(1 << 20)  # never dereferenced: every check runs on the host first
    assert lib.kd_argmax(None, 1, 8, fake, fake, None) == -1
    assert lib.kd_argmax(fake, 0, 8, fake, fake, None) == -7
    assert lib.kd_argmax(fake, 17, 8, fake, fake, None) == -7
    assert lib.kd_argmax(fake, 1, 6, fake, fake, None) == -1
    assert lib.kd_argmax(C.c_void_p((1 << 20) + 4), 1, 8, fake, fake, None) == -1
    assert "aligned" in kd.kd_last_error()


def test_op_level_argument_checks(lib):
    m = synth.q8_0_matrix(0, "abi", 48, 128)  # 48 rows: not a multiple of 32
    h = C.c_void_p()
    assert lib.kd_q8_matrix_create(m.ctypes.data, 48, 128, C.byref(h)) == -8
    assert lib.kd_q8_matrix_create(m.ctypes.data, 32, 96, C.byref(h)) == -8
    i32p = C.POINTER(C.c_int32)
    slots = np.zeros(2, np.int32)
    pos = np.zeros(2, np.int32)
    dummy = 1 << 20
    st = lib.kd_attn_append_decode(dummy, dummy, dummy, dummy, dummy, slots.ctypes.data_as(i32p),
                                   pos.ctypes.data_as(i32p), 17, 32, 8, 128, 4, 64, dummy, dummy, 1 << 30,
                                   None)
    assert st == -7  # B > 16
    st = lib.kd_attn_append_decode(dummy, dummy, dummy, dummy, dummy, slots.ctypes.data_as(i32p),
                                   pos.ctypes.data_as(i32p), 2, 32, 8, 96, 4, 64, dummy, dummy, 1 << 30,
                                   None)
    assert st == -8  # head_dim 96 unsupported
    st = lib.kd_attn_append_decode(dummy, dummy, dummy, dummy, dummy, slots.ctypes.data_as(i32p),
                                   pos.ctypes.data_as(i32p), 2, 32, 8, 128, 4, 64, dummy, dummy, 16, None)
    assert st == -1  # workspace too small
    st = lib.kd_attn_append_decode(dummy, dummy, dummy, dummy, dummy, slots.ctypes.data_as(i32p),
                                   pos.ctypes.data_as(i32p), 2, 32, 8, 128, 4, 64, dummy, dummy, 1 << 30,
                                   None)
    assert st == -5  # slot 0 repeated


def test_fail_alloc_switch_host_side(lib):
    out = C.c_int32(-7)
    assert lib.kd_debug_fail_alloc(-1, C.byref(out)) == -1
    assert lib.kd_debug_fail_alloc(3, C.byref(out)) == 0 and out.value >= 0
    # a load refused before it allocates anything leaves the switch armed; disarm it
    cfg = kd.make_config(synth.TINY, 2, 64)
    cfg.head_dim = 96
    h = C.c_void_p()
    assert lib.kd_model_load(C.byref(cfg), C.byref(kd.KdWeights()), C.byref(h)) in (-8, -1)
    assert lib.kd_debug_fail_alloc(0, None) == 0


def test_kv_q8_argument_checks(lib):
    i32p = C.POINTER(C.c_int32)
    slots = np.array([0, 1], np.int32)
    pos = np.zeros(2, np.int32)
    d = 1 << 20
    big = 1 << 30

    def call(B=2, nh=32, nkv=8, n_slots=4, cap=64, ws=big, sl=slots, ps=pos, q=d):
        return lib.kd_attn_append_decode_q8(q, d, d, d, d, d, d, sl.ctypes.data_as(i32p), ps.ctypes.data_as(i32p),
                                            B, nh, nkv, n_slots, cap, d, d, ws, None)
    assert call(B=17) == -7
    assert call(nh=24, nkv=8) == -8        # group 3
    assert call(nh=32, nkv=2) == -8        # group 16
    assert call(cap=63) == -1              # odd capacity
    assert call(ws=16) == -1               # workspace too small
    assert call(q=d + 4) == -1             # not 16-byte aligned
    assert call(sl=np.array([0, 0], np.int32)) == -5
    assert call(sl=np.array([0, 4], np.int32)) == -5
    assert call(ps=np.array([0, 64], np.int32)) == -6
    assert lib.kd_kv_q8_quantize(None, 4, d, d, None) == -1
    assert lib.kd_kv_q8_quantize(d, 0, d, d, None) == -1


def test_attention_workspace_size():
    n = kd.kd_attn_workspace_bytes(8, 32, 128, 32768)
    assert n == 256 + 8 * 32 * 512 * 132 * 4  # 64-key splits, 16-byte aligned records
    assert kd.kd_attn_workspace_bytes(0, 32, 128, 10) == 0


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    monkeypatch.setattr(kd, "LIB_PATH", tmp_path / "libkd.so")
    monkeypatch.setattr(kd, "_lib", None)
    with pytest.raises(ImportError):
        kd.lib()
