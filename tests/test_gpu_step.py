"""The whole batched decode step through the C ABI, on the tiny model.

Workload: the tiny oracle model (1 layer, hidden 256, 4/2 heads of 64, FFN 768,
vocab 512, RoPE theta 1e4, Q8_0 weights as generated), B = 2 sessions with 17
and 40 pre-filled fp16 positions, 4 greedy steps, seed 0.

Gates: teacher-forced logits within 5e-2 (max abs) of the oracle and per-layer
hidden states within 1e-3 relative L2 -- with the workload's unit norm weights
and with seeded non-unit ones, different for every layer and norm; every
session's greedy stream and logits bit-identical to its isolated B = 1 run;
graph replay identical to the direct launch train."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

LOGIT_TOL = 5e-2
HIDDEN_REL_L2 = 1e-3


def load(kd, shape, w, max_sessions, cap, flags=0):
    return kd.kd_model_load(kd.make_config(shape, max_sessions, cap, flags), w)


def bind_prefilled(kd, m, shape, lens, seed=0, first_session=0):
    ids = []
    for i, n in enumerate(lens):
        k, v = synth.kv_prefill(shape, seed, first_session + i, n)
        sid = kd.kd_session_bind(m)
        kd.kd_session_load_kv(m, sid, k, v, n)
        ids.append(sid)
    return ids


def gpu_step(kd, m, ids, tok, pos, V):
    B = len(ids)
    lg = torch.empty(B, V, device="cuda", dtype=torch.float32)
    am = torch.empty(B, device="cuda", dtype=torch.int32)
    kd.kd_decode_step(m, ids, tok, pos, lg, am)
    torch.cuda.synchronize()
    return lg.cpu().numpy(), am.cpu().numpy()


@pytest.fixture(scope="module")
def tiny():
    shape = synth.TINY
    return shape, synth.model_weights(shape, 0)


# 0: schedules chosen per matrix; 2 / 4: every projection forced onto the
# stream / group schedule (the tiny model alone would only exercise one of them);
# 32: the RMSNorm folded into the q|k|v and gate|up activation load.
# norms: the workload's unit norm weights, or seeded non-unit ones (1 + 0.1 N(0,1),
# a different vector for every layer's two norms and the output norm), so that a
# kernel that dropped the weight or read another layer's would fail.
@pytest.mark.parametrize("norms", ["unit", "seeded"])
@pytest.mark.parametrize("flags", [0, 2, 4, 32])
def test_tiny_teacher_forced_against_oracle(kdlib, tiny, flags, norms):
    kd = kdlib
    shape, w = tiny
    if norms == "seeded":
        w = dict(w, **synth.norm_weights(shape, 7))
    case = synth.TINY_CASE
    cap = 64
    m = load(kd, shape, w, 4, cap, flags)
    try:
        lens = list(case["prefill"])
        ids = bind_prefilled(kd, m, shape, lens)
        om = oracle.OracleModel(shape, w)
        caches = [om.new_cache(cap, *synth.kv_prefill(shape, 0, i, n)) for i, n in enumerate(lens)]
        B, L, H = len(lens), shape.n_layers, shape.hidden
        hid = torch.empty(L + 1, B, H, device="cuda", dtype=torch.float32)
        kd.kd_debug_capture_hidden(m, hid)
        tok = synth.tokens(0, "tiny-steps", B, shape.vocab)
        for step in range(case["steps"]):
            pos = [n + step for n in lens]
            lg, am = gpu_step(kd, m, ids, tok, pos, shape.vocab)
            ref, ref_am, ref_h = om.step(tok, pos, caches, cap, want_hidden=True)
            assert np.abs(lg - ref).max() <= LOGIT_TOL, (step, float(np.abs(lg - ref).max()))
            gh = hid.cpu().numpy()
            for b in range(B):
                for l in range(L + 1):
                    rel = np.linalg.norm(gh[l, b] - ref_h[b, l]) / np.linalg.norm(ref_h[b, l])
                    assert rel <= HIDDEN_REL_L2, (step, b, l, rel)
            for b in range(B):
                assert kd.kd_session_length(m, ids[b]) == pos[b] + 1
            tok = ref_am  # teacher forcing: the oracle's greedy token feeds the next step
        assert kd.kd_device_status(m) == 0
    finally:
        kd.kd_model_free(m)


def test_tiny_first_position_and_last_slot_position(kdlib, tiny):
    """The degenerate ends of a slot in one ragged batch, teacher-forced against
    the oracle: a fresh session decoding from position 0 (one key, a single
    split, the KV append at the slot's first row) beside a session that decodes
    up to the slot's last position (cap - 1), where the next position is refused."""
    kd = kdlib
    shape, w = tiny
    cap, steps = 64, 4
    lens = [0, cap - steps]
    m = load(kd, shape, w, 4, cap)
    try:
        fresh = kd.kd_session_bind(m)
        (full,) = bind_prefilled(kd, m, shape, [lens[1]], first_session=1)
        ids = [fresh, full]
        om = oracle.OracleModel(shape, w)
        caches = [om.new_cache(cap), om.new_cache(cap, *synth.kv_prefill(shape, 0, 1, lens[1]))]
        B, L, H = 2, shape.n_layers, shape.hidden
        hid = torch.empty(L + 1, B, H, device="cuda", dtype=torch.float32)
        kd.kd_debug_capture_hidden(m, hid)
        tok = synth.tokens(0, "tiny-ends", B, shape.vocab)
        for step in range(steps):
            pos = [n + step for n in lens]
            lg, _ = gpu_step(kd, m, ids, tok, pos, shape.vocab)
            ref, ref_am, ref_h = om.step(tok, pos, caches, cap, want_hidden=True)
            assert np.abs(lg - ref).max() <= LOGIT_TOL, (step, float(np.abs(lg - ref).max()))
            gh = hid.cpu().numpy()
            for b in range(B):
                for l in range(L + 1):
                    rel = np.linalg.norm(gh[l, b] - ref_h[b, l]) / np.linalg.norm(ref_h[b, l])
                    assert rel <= HIDDEN_REL_L2, (step, b, l, rel)
            tok = ref_am
        assert kd.kd_session_length(m, full) == cap
        kd.kd_debug_capture_hidden(m, None)
        with pytest.raises(kd.KdError) as e:  # the slot is full
            kd.kd_decode_step(m, [full], tok[1:], np.array([cap], np.int32), None, None)
        assert e.value.name == "KD_ERR_POSITION"
        assert kd.kd_device_status(m) == 0
    finally:
        kd.kd_model_free(m)


def greedy_stream(kd, m, ids, lens, tok0, steps, V):
    tok = np.array(tok0, np.int32)
    toks, logits = [], []
    for s in range(steps):
        lg, am = gpu_step(kd, m, ids, tok, [n + s for n in lens], V)
        toks.append(am.copy())
        logits.append(lg.copy())
        tok = am
    return np.array(toks), np.array(logits)


# graph replay (auto schedules), kernel-by-kernel launches, each schedule forced,
# and the folded norm
@pytest.mark.parametrize("flags", [0, 1, 2, 4, 32])
def test_tiny_batch_invariance(kdlib, tiny, flags):
    kd = kdlib
    shape, w = tiny
    cap, steps = 64, 8
    lens = [17, 40, 3, 9, 25]
    tok0 = synth.tokens(0, "tiny-inv", len(lens), shape.vocab)
    m = load(kd, shape, w, 8, cap, flags)
    try:
        ids = bind_prefilled(kd, m, shape, lens)
        batch_t, batch_l = greedy_stream(kd, m, ids, lens, tok0, steps, shape.vocab)
        for b in range(len(lens)):
            kd.kd_session_free(m, ids[b])
        for b in range(len(lens)):
            (sid,) = bind_prefilled(kd, m, shape, [lens[b]], first_session=b)
            t1, l1 = greedy_stream(kd, m, [sid], [lens[b]], tok0[b:b + 1], steps, shape.vocab)
            assert np.array_equal(t1[:, 0], batch_t[:, b]), b
            assert np.array_equal(l1[:, 0].view(np.uint32), batch_l[:, b].view(np.uint32)), b
            kd.kd_session_free(m, sid)
    finally:
        kd.kd_model_free(m)


def test_tiny_graph_equals_direct_and_rewind(kdlib, tiny):
    kd = kdlib
    shape, w = tiny
    cap, lens = 64, [17, 40]
    tok = synth.tokens(0, "tiny-gd", 2, shape.vocab)
    out = []
    for flags in (0, 1):
        m = load(kd, shape, w, 4, cap, flags)
        try:
            ids = bind_prefilled(kd, m, shape, lens)
            a = gpu_step(kd, m, ids, tok, lens, shape.vocab)
            gpu_step(kd, m, ids, tok[::-1].copy(), [n + 1 for n in lens], shape.vocab)
            # rewind both sessions to their first decode position: same inputs, same bits
            b = gpu_step(kd, m, ids, tok, lens, shape.vocab)
            assert np.array_equal(a[0].view(np.uint32), b[0].view(np.uint32))
            assert kd.kd_session_length(m, ids[0]) == lens[0] + 1
            out.append(a[0])
        finally:
            kd.kd_model_free(m)
    assert np.array_equal(out[0].view(np.uint32), out[1].view(np.uint32))


def test_tiny_errors_change_no_state(kdlib, tiny):
    kd = kdlib
    shape, w = tiny
    m = load(kd, shape, w, 2, 32)
    try:
        a = kd.kd_session_bind(m)
        b = kd.kd_session_bind(m)
        with pytest.raises(kd.KdError) as e:
            kd.kd_session_bind(m)
        assert e.value.name == "KD_ERR_NO_FREE_SLOT"
        cases = [
            (dict(session_ids=[a, a], tokens=[1, 2], positions=[0, 0]), "KD_ERR_BAD_SESSION"),
            (dict(session_ids=[a, 7], tokens=[1, 2], positions=[0, 0]), "KD_ERR_BAD_SESSION"),
            (dict(session_ids=[a], tokens=[shape.vocab], positions=[0]), "KD_ERR_INVALID_ARG"),
            (dict(session_ids=[a], tokens=[-1], positions=[0]), "KD_ERR_INVALID_ARG"),
            (dict(session_ids=[a], tokens=[1], positions=[1]), "KD_ERR_POSITION"),
            (dict(session_ids=[a], tokens=[1], positions=[-1]), "KD_ERR_POSITION"),
            (dict(session_ids=list(range(17)), tokens=[1] * 17, positions=[0] * 17), "KD_ERR_BATCH"),
            (dict(session_ids=[], tokens=[], positions=[]), "KD_ERR_BATCH"),
        ]
        for kw, name in cases:
            with pytest.raises(kd.KdError) as e:
                kd.kd_decode_step(m, **kw)
            assert e.value.name == name, (kw, e.value)
        assert kd.kd_session_length(m, a) == 0 and kd.kd_session_length(m, b) == 0
        kd.kd_decode_step(m, [a, b], [1, 2], [0, 0])
        assert kd.kd_session_length(m, a) == 1
        with pytest.raises(kd.KdError) as e:  # capacity 32: position 32 is out of range
            kd.kd_session_load_kv(m, a, None, None, 33)
        assert e.value.name == "KD_ERR_POSITION"
        kd.kd_session_free(m, a)
        with pytest.raises(kd.KdError):
            kd.kd_session_length(m, a)
        assert kd.kd_session_bind(m) == a  # lowest free slot, length 0 again
        assert kd.kd_session_length(m, a) == 0
        assert kd.kd_device_status(m) == 0
    finally:
        kd.kd_model_free(m)


def test_tiny_fused_norm_bitwise_equals_norm_kernel(kdlib, tiny):
    """The RMSNorm folded into the q|k|v and gate|up activation load gives the
    same bits as the unfused train (the norm as a kernel of its own, then the
    projection reading its fp16 output): logits and every layer's hidden state,
    over several steps, with seeded non-unit norm weights."""
    kd = kdlib
    shape, w = tiny
    w = dict(w, **synth.norm_weights(shape, 5))
    cap, lens = 64, [17, 40, 3]
    tok0 = synth.tokens(0, "tiny-fuse", len(lens), shape.vocab)
    runs = []
    for flags in (0, 32):
        m = load(kd, shape, w, 4, cap, flags)
        try:
            ids = bind_prefilled(kd, m, shape, lens)
            B, L, H = len(lens), shape.n_layers, shape.hidden
            hid = torch.empty(L + 1, B, H, device="cuda", dtype=torch.float32)
            kd.kd_debug_capture_hidden(m, hid)
            tok, out = tok0.copy(), []
            for step in range(4):
                lg, am = gpu_step(kd, m, ids, tok, [n + step for n in lens], shape.vocab)
                out.append((lg.view(np.uint32).copy(), hid.cpu().numpy().view(np.uint32).copy()))
                tok = am
            runs.append(out)
        finally:
            kd.kd_model_free(m)
    for step, ((l0, h0), (l1, h1)) in enumerate(zip(*runs)):
        assert np.array_equal(l0, l1), step
        assert np.array_equal(h0, h1), step


def test_tiny_batch_above_16_runs_in_groups(kdlib, tiny):
    """B = 37 > 16: the step runs as groups of 16, 16 and 5 rows on the same
    kernels.  Every session's greedy tokens and logit bits, and its hidden states
    (captured across the groups), equal its run alone at B = 1."""
    kd = kdlib
    shape, w = tiny
    cap, steps, B = 64, 3, 37
    lens = [(5 * i + 3) % 50 for i in range(B)]
    tok0 = synth.tokens(0, "tiny-chunks", B, shape.vocab)
    m = load(kd, shape, w, 40, cap)
    try:
        L, H = shape.n_layers, shape.hidden
        ids = bind_prefilled(kd, m, shape, lens)
        hid = torch.empty(L + 1, B, H, device="cuda", dtype=torch.float32)
        kd.kd_debug_capture_hidden(m, hid)
        gpu_step(kd, m, ids, tok0, lens, shape.vocab)
        batch_hidden = hid.cpu().numpy().view(np.uint32).copy()
        kd.kd_debug_capture_hidden(m, None)
        batch_t, batch_l = greedy_stream(kd, m, ids, lens, tok0, steps, shape.vocab)  # rewinds to lens
        for sid in ids:
            kd.kd_session_free(m, sid)
        one = torch.empty(L + 1, 1, H, device="cuda", dtype=torch.float32)
        for b in range(B):
            (sid,) = bind_prefilled(kd, m, shape, [lens[b]], first_session=b)
            kd.kd_debug_capture_hidden(m, one)
            gpu_step(kd, m, [sid], tok0[b:b + 1], [lens[b]], shape.vocab)
            assert np.array_equal(one.cpu().numpy().view(np.uint32)[:, 0], batch_hidden[:, b]), b
            kd.kd_debug_capture_hidden(m, None)
            t1, l1 = greedy_stream(kd, m, [sid], [lens[b]], tok0[b:b + 1], steps, shape.vocab)
            assert np.array_equal(t1[:, 0], batch_t[:, b]), b
            assert np.array_equal(l1[:, 0].view(np.uint32), batch_l[:, b].view(np.uint32)), b
            kd.kd_session_free(m, sid)
        assert kd.kd_device_status(m) == 0
    finally:
        kd.kd_model_free(m)


def test_tiny_fused_epilogues_bitwise_equal_unfused_train(kdlib, tiny):
    """Each fusion of the step against its unfused sequence, bit for bit: RoPE and
    the KV append in the q|k|v epilogue, SwiGLU in the gate|up epilogue, the
    residual add and the next norm's sums of squares in the o-proj and down
    epilogues, and layer 0's attention norm in the embedding kernel
    (KD_FLAG_UNFUSED runs them as kernels of their own after plain
    projections, with the group schedule's summation order).  Logits, every
    hidden state and the appended cache rows (through later steps' attention),
    several steps, seeded norm weights."""
    kd = kdlib
    shape, w = tiny
    w = dict(w, **synth.norm_weights(shape, 9))
    cap, lens = 64, [17, 40, 3]
    tok0 = synth.tokens(0, "tiny-unfused", len(lens), shape.vocab)
    runs = []
    for flags in (0, 64):
        m = load(kd, shape, w, 4, cap, flags)
        try:
            ids = bind_prefilled(kd, m, shape, lens)
            B, L, H = len(lens), shape.n_layers, shape.hidden
            hid = torch.empty(L + 1, B, H, device="cuda", dtype=torch.float32)
            kd.kd_debug_capture_hidden(m, hid)
            tok, out = tok0.copy(), []
            for step in range(5):
                lg, am = gpu_step(kd, m, ids, tok, [n + step for n in lens], shape.vocab)
                out.append((lg.view(np.uint32).copy(), hid.cpu().numpy().view(np.uint32).copy()))
                tok = am
            runs.append(out)
            assert kd.kd_device_status(m) == 0
        finally:
            kd.kd_model_free(m)
    for step, ((l0, h0), (l1, h1)) in enumerate(zip(*runs)):
        assert np.array_equal(h0, h1), step
        assert np.array_equal(l0, l1), step


@pytest.mark.parametrize("flags", [0, 1])
def test_tiny_measured_steps(kdlib, tiny, flags):
    """kd_profile_enable: measured steps (every kernel launched from the host and
    bracketed by two events) give the same bits as unmeasured ones, graph-replayed
    or not, and kd_profile_read counts every launch of every class with a
    positive device time, then resets."""
    kd = kdlib
    shape, w = tiny
    cap, lens, steps = 64, [17, 40], 3
    m = load(kd, shape, w, 4, cap, flags)
    try:
        ids = bind_prefilled(kd, m, shape, lens)
        tok = synth.tokens(0, "tiny-prof", len(lens), shape.vocab)
        ref = [gpu_step(kd, m, ids, tok, [n + s for n in lens], shape.vocab)[0] for s in range(steps)]
        kd.kd_profile_enable(m, True)
        kd.kd_profile_read(m)
        got = [gpu_step(kd, m, ids, tok, [n + s for n in lens], shape.vocab)[0] for s in range(steps)]
        prof = kd.kd_profile_read(m)
        kd.kd_profile_enable(m, False)
        after = gpu_step(kd, m, ids, tok, lens, shape.vocab)[0]
        for a, b in zip(ref, got):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        assert np.array_equal(after.view(np.uint32), ref[0].view(np.uint32))
        L = shape.n_layers
        # the embedding kernel forms layer 0's attention norm (2L norm launches:
        # L - 1 attention norms, L FFN norms, the output norm)
        want = {"embed": 1, "rmsnorm": 2 * L, "qkv": L, "attn_split": L, "attn_combine": L, "wo": L,
                "gate_up": L, "down": L, "lm_head": 1, "argmax": 1}
        for k, per_step in want.items():
            n, ms = prof[k]
            assert n == per_step * steps, (k, n)
            assert ms > 0.0, k
        assert all(v == (0, 0.0) for v in kd.kd_profile_read(m).values())
        assert kd.kd_device_status(m) == 0
    finally:
        kd.kd_model_free(m)
