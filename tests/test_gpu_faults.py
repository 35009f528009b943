"""The device fault path, on the tiny model, through the C ABI.

Every wait a kernel does on a copy or on another warp is bounded (about half a
second); when one runs out the kernel sets the model's fault word, lets its
issued copies land and returns, and kd_device_status reports KD_ERR_DEVICE.  The
debug hook kd_debug_inject_wait_timeout makes one such wait run out on purpose:
one barrier of the chosen kernel expects a few bytes more than its copies
deliver.  Nothing faults or hangs; the GPU context stays usable.

Checked for every kernel class with bounded waits, on both projection
schedules: the faulted step is reported, and the next step (rewound to the same
positions) matches the oracle before the host has cleared anything -- so a
kernel that gave up left no state (arrival counters, ring barriers) that spoils
later launches -- and again after the status call.

Also the host side of failure: a model load that runs out of memory at any one
of its allocations (kd_debug_fail_alloc) fails closed with KD_ERR_OOM, returns
the device memory it took, and leaves the next load and step working."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

LOGIT_TOL = 5e-2
CAP = 64
LENS = (17, 40)


@pytest.fixture(scope="module")
def tiny():
    shape = synth.TINY
    return shape, synth.model_weights(shape, 0)


def run_step(kd, m, ids, tok, pos, V):
    lg = torch.empty(len(ids), V, device="cuda", dtype=torch.float32)
    am = torch.empty(len(ids), device="cuda", dtype=torch.int32)
    kd.kd_decode_step(m, ids, tok, pos, lg, am)
    torch.cuda.synchronize()
    return lg.cpu().numpy()


# flags 0: schedules as chosen (every tiny projection on the group schedule);
# flags 2: every projection on the stream schedule, whose split row groups meet
# through arrival counters in global memory.
@pytest.mark.parametrize("flags,cls", [
    (0, "qkv"), (0, "attn_split"), (0, "wo"), (0, "gate_up"), (0, "down"), (0, "lm_head"),
    (2, "qkv"), (2, "down"), (2, "lm_head"),
])
def test_bounded_wait_runs_out_is_reported_and_recovered(kdlib, tiny, flags, cls):
    kd = kdlib
    shape, w = tiny
    m = kd.kd_model_load(kd.make_config(shape, 4, CAP, flags), w)
    try:
        ids = []
        for i, n in enumerate(LENS):
            k, v = synth.kv_prefill(shape, 0, i, n)
            sid = kd.kd_session_bind(m)
            kd.kd_session_load_kv(m, sid, k, v, n)
            ids.append(sid)
        om = oracle.OracleModel(shape, w)
        caches = [om.new_cache(CAP, *synth.kv_prefill(shape, 0, i, n)) for i, n in enumerate(LENS)]
        tok = synth.tokens(0, "faults", len(LENS), shape.vocab)
        pos = list(LENS)
        ref, _, _ = om.step(tok, pos, caches, CAP)

        kd.kd_debug_inject_wait_timeout(m, cls)
        run_step(kd, m, ids, tok, pos, shape.vocab)  # the faulted step (its outputs are not valid)
        # rewound to the same positions, before anything is cleared on the host
        got = run_step(kd, m, ids, tok, pos, shape.vocab)
        assert np.abs(got - ref).max() <= LOGIT_TOL, (cls, float(np.abs(got - ref).max()))
        with pytest.raises(kd.KdError) as e:
            kd.kd_device_status(m)
        assert e.value.name == "KD_ERR_DEVICE"
        assert kd.kd_device_status(m) == 0  # read and cleared
        got = run_step(kd, m, ids, tok, pos, shape.vocab)
        assert np.abs(got - ref).max() <= LOGIT_TOL, cls
        assert kd.kd_device_status(m) == 0
    finally:
        kd.kd_model_free(m)


# 10 sessions: every projection runs its two-tile kernel (two 8-session MMA
# column tiles per warp), whose give-up path differs from the one-tile kernel's.
@pytest.mark.parametrize("cls", ["qkv", "wo", "gate_up", "down", "lm_head"])
def test_bounded_wait_runs_out_in_the_two_tile_kernels(kdlib, tiny, cls):
    kd = kdlib
    shape, w = tiny
    lens = [17 + 3 * i for i in range(10)]
    m = kd.kd_model_load(kd.make_config(shape, 12, CAP), w)
    try:
        ids = []
        for i, n in enumerate(lens):
            k, v = synth.kv_prefill(shape, 0, i, n)
            sid = kd.kd_session_bind(m)
            kd.kd_session_load_kv(m, sid, k, v, n)
            ids.append(sid)
        om = oracle.OracleModel(shape, w)
        caches = [om.new_cache(CAP, *synth.kv_prefill(shape, 0, i, n)) for i, n in enumerate(lens)]
        tok = synth.tokens(0, "faults-10", len(lens), shape.vocab)
        ref, _, _ = om.step(tok, lens, caches, CAP)
        kd.kd_debug_inject_wait_timeout(m, cls)
        run_step(kd, m, ids, tok, lens, shape.vocab)  # the faulted step
        got = run_step(kd, m, ids, tok, lens, shape.vocab)
        assert np.abs(got - ref).max() <= LOGIT_TOL, (cls, float(np.abs(got - ref).max()))
        with pytest.raises(kd.KdError) as e:
            kd.kd_device_status(m)
        assert e.value.name == "KD_ERR_DEVICE"
        assert kd.kd_device_status(m) == 0
    finally:
        kd.kd_model_free(m)


def test_inject_refuses_classes_without_waits(kdlib, tiny):
    kd = kdlib
    shape, w = tiny
    m = kd.kd_model_load(kd.make_config(shape, 2, CAP), w)
    try:
        for cls in ("embed", "rmsnorm", "attn_combine", "argmax"):
            with pytest.raises(kd.KdError) as e:
                kd.kd_debug_inject_wait_timeout(m, cls)
            assert e.value.name == "KD_ERR_INVALID_ARG"
    finally:
        kd.kd_model_free(m)


def test_op_level_fault_words_read_clean(kdlib):
    """The op-level calls' fault words are readable and zero after healthy calls."""
    kd = kdlib
    W = synth.q8_0_matrix(0, "fault-word", 64, 256)
    h = kd.kd_q8_matrix_create(W)
    try:
        x = torch.from_numpy(synth.activations_fp16(0, "fault-word", 2, 256).view(np.int16)).cuda()
        y = torch.empty(2, 64, device="cuda", dtype=torch.float32)
        kd.kd_mmvq(h, x, 2, y)
        assert kd.kd_q8_matrix_status(h) == 0
    finally:
        kd.kd_q8_matrix_free(h)
    nh, nkv, hd, cap, B = 8, 2, 64, 128, 2
    q = torch.randn(B, nh, hd, device="cuda")
    kn, vn = torch.randn(B, nkv, hd, device="cuda"), torch.randn(B, nkv, hd, device="cuda")
    kc = torch.zeros(B, nkv, cap, hd, device="cuda", dtype=torch.float16)
    vc = torch.zeros_like(kc)
    out = torch.empty(B, nh * hd, device="cuda", dtype=torch.float16)
    ws = torch.empty(kd.kd_attn_workspace_bytes(B, nh, hd, cap), device="cuda", dtype=torch.uint8)
    slots, pos = np.arange(B, dtype=np.int32), np.array([0, 5], np.int32)
    kd.kd_attn_append_decode(q, kn, vn, kc, vc, slots, pos, nh, nkv, hd, B, cap, out, ws)
    assert kd.kd_attn_device_status(ws) == 0


def test_model_load_fails_closed_at_every_allocation(kdlib, tiny):
    kd = kdlib
    shape, w = tiny
    cfg = kd.make_config(shape, 2, CAP)
    m = kd.kd_model_load(cfg, w)  # a complete load first: its kernels' modules are resident after it
    kd.kd_model_free(m)
    n = kd.kd_debug_fail_alloc(0)
    assert n >= 20, n
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for k in range(1, n + 1):
        kd.kd_debug_fail_alloc(k)
        with pytest.raises(kd.KdError) as e:
            kd.kd_model_load(cfg, w)
        assert e.value.name == "KD_ERR_OOM", (k, e.value)
        assert abs(torch.cuda.mem_get_info()[0] - free0) <= (2 << 20), k  # nothing left allocated
    # disarmed (one-shot): the next load and a step work and match the oracle
    m = kd.kd_model_load(cfg, w)
    try:
        assert kd.kd_debug_fail_alloc(0) == n
        ids = []
        for i, L0 in enumerate(LENS):
            k_, v_ = synth.kv_prefill(shape, 0, i, L0)
            sid = kd.kd_session_bind(m)
            kd.kd_session_load_kv(m, sid, k_, v_, L0)
            ids.append(sid)
        torch.cuda.synchronize()
        om = oracle.OracleModel(shape, w)
        caches = [om.new_cache(CAP, *synth.kv_prefill(shape, 0, i, L0)) for i, L0 in enumerate(LENS)]
        tok = synth.tokens(0, "fail-alloc", len(LENS), shape.vocab)
        got = run_step(kd, m, ids, tok, list(LENS), shape.vocab)
        ref, _, _ = om.step(tok, list(LENS), caches, CAP)
        assert np.abs(got - ref).max() <= LOGIT_TOL
        assert kd.kd_device_status(m) == 0
    finally:
        kd.kd_model_free(m)
