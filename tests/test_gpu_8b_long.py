"""The 8B-shaped decode step at long context through the C ABI.

Workload (the long-context multi-tenant case): the Llama-3-8B-shaped model with
random Q8_0 weights, B = 8 sessions in slots of 32768 positions each, pre-filled
with seeded N(0, 1) fp16 KV to 25704 + 1000 i positions (i = 0 .. 7, staggered),
64 greedy steps.

Gates:
- at the first step, the logits of the shortest and the longest session within
  5e-2 of the fp64 oracle (which runs each alone at its own length), and layers
  0, 16 and 31 of both within 1e-3 relative L2 when fed the oracle's input;
- the longest session teacher-forced through all 64 steps: at the last one it
  writes and attends the slot's last position (32767, a full last split), where
  its logits must be within 5e-2 of the oracle's and its hidden states within
  the end-to-end bound;
- every session's 64-step greedy stream (tokens, and the logit bits of sampled
  steps) in the B = 8 batch equal to its run alone (B = 1) from the same start.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SHAPE = synth.LLAMA3_8B
CASE = synth.LONG_CTX_8B_CASE
S, CAP, STEPS = CASE["sessions"], CASE["capacity"], CASE["steps"]
LENS = [CASE["prefill_base"] + CASE["prefill_stagger"] * i for i in range(S)]
CHECKED = (0, S - 1)  # the shortest and the longest session
LOGIT_TOL = 5e-2
HIDDEN_REL_L2 = 1e-3


@pytest.fixture(scope="module")
def long_model(kdlib):
    kd = kdlib
    assert LENS[-1] + STEPS <= CAP
    w = synth.model_weights(SHAPE, CASE["seed"])
    m = kd.kd_model_load(kd.make_config(SHAPE, S, CAP), w)
    ids, keep = [], {}
    try:
        for i, n in enumerate(LENS):
            k, v = synth.kv_prefill(SHAPE, CASE["seed"], 1000 + i, n)
            sid = kd.kd_session_bind(m)
            kd.kd_session_load_kv(m, sid, k, v, n)
            torch.cuda.synchronize()  # the copy reads k, v until the stream reaches it
            ids.append(sid)
            if i in CHECKED:
                keep[i] = (k, v)
        yield kd, m, w, ids, keep
    finally:
        kd.kd_model_free(m)


def test_8b_long_context_against_oracle(long_model):
    kd, m, w, ids, keep = long_model
    V, H, L = SHAPE.vocab, SHAPE.hidden, SHAPE.n_layers
    tok0 = synth.tokens(CASE["seed"], "8b-long", S, V)
    lg = torch.empty(S, V, device="cuda", dtype=torch.float32)
    kd.kd_decode_step(m, ids, tok0, LENS, lg, None)
    got = lg.cpu().numpy()
    om = oracle.OracleModel(SHAPE, w)
    ref_h = {}
    for i in CHECKED:
        cache = om.new_cache(CAP, *keep[i])
        ref, _, h = om.step(tok0[i:i + 1], [LENS[i]], [cache], CAP, want_hidden=True)
        err = float(np.abs(got[i] - ref[0]).max())
        assert err <= LOGIT_TOL, (i, err)
        ref_h[i] = h[0]
        del cache
    x_out = torch.empty(len(CHECKED), H, device="cuda", dtype=torch.float32)
    sids = [ids[i] for i in CHECKED]
    for l in (0, L // 2, L - 1):
        x_in = torch.from_numpy(np.ascontiguousarray(np.stack([ref_h[i][l] for i in CHECKED]))).cuda()
        kd.kd_debug_layer(m, l, sids, [LENS[i] for i in CHECKED], x_in, x_out)
        out = x_out.cpu().numpy()
        for j, i in enumerate(CHECKED):
            want = ref_h[i][l + 1]
            rel = float(np.linalg.norm(out[j] - want) / np.linalg.norm(want))
            assert rel <= HIDDEN_REL_L2, (l, i, rel)
    assert kd.kd_device_status(m) == 0


HIDDEN_REL_L2_END_TO_END = 1e-2  # as in test_gpu_8b.py (see the sensitivity test)


def test_8b_long_context_last_position_against_oracle(long_model):
    kd, m, w, ids, keep = long_model
    V, H, L = SHAPE.vocab, SHAPE.hidden, SHAPE.n_layers
    i = S - 1
    assert LENS[i] + STEPS == CAP  # the last step decodes position CAP - 1
    tok0 = synth.tokens(CASE["seed"], "8b-long-tf", S, V)
    om = oracle.OracleModel(SHAPE, w)
    cache = om.new_cache(CAP, *keep[i])
    tok = tok0[i:i + 1].copy()
    toks = []
    for s in range(STEPS):  # the oracle alone, from its own greedy tokens
        lg, am, h = om.step(tok, [LENS[i] + s], [cache], CAP, want_hidden=s == STEPS - 1)
        toks.append(int(tok[0]))
        tok = am.copy()
    ref_lg, ref_h = lg[0], h[0]
    del cache
    hid = torch.empty(L + 1, S, H, device="cuda", dtype=torch.float32)
    lgd = torch.empty(S, V, device="cuda", dtype=torch.float32)
    amd = torch.empty(S, device="cuda", dtype=torch.int32)
    tok = tok0.copy()
    try:
        for s in range(STEPS):
            tok[i] = toks[s]
            kd.kd_debug_capture_hidden(m, hid if s == STEPS - 1 else None)
            kd.kd_decode_step(m, ids, tok, [n + s for n in LENS], lgd, amd)
            tok = amd.cpu().numpy()
        got, gh = lgd.cpu().numpy()[i], hid.cpu().numpy()[:, i]
    finally:
        kd.kd_debug_capture_hidden(m, None)
    assert kd.kd_session_length(m, ids[i]) == CAP
    err = float(np.abs(got - ref_lg).max())
    assert err <= LOGIT_TOL, err
    for l in range(L + 1):
        rel = float(np.linalg.norm(gh[l] - ref_h[l]) / np.linalg.norm(ref_h[l]))
        assert rel <= HIDDEN_REL_L2_END_TO_END, (l, rel)
    assert kd.kd_device_status(m) == 0


def greedy(kd, m, ids, starts, tok0, steps):
    B = len(ids)
    tok = np.array(tok0, np.int32)
    toks = np.empty((steps, B), np.int32)
    sampled = {}
    lg = torch.empty(B, SHAPE.vocab, device="cuda", dtype=torch.float32)
    am = torch.empty(B, device="cuda", dtype=torch.int32)
    for s in range(steps):
        kd.kd_decode_step(m, ids, tok, [p + s for p in starts], lg, am)
        tok = am.cpu().numpy()
        toks[s] = tok
        if s % 16 == 0 or s == steps - 1:
            sampled[s] = lg.cpu().numpy().view(np.uint32).copy()
    return toks, sampled


def test_8b_long_context_batch_invariance(long_model):
    kd, m, w, ids, keep = long_model
    tok0 = synth.tokens(CASE["seed"], "8b-long-greedy", S, SHAPE.vocab)
    toks, sampled = greedy(kd, m, ids, LENS, tok0, STEPS)
    for i in range(S):
        # the same session alone, rewound to the same start
        t1, s1 = greedy(kd, m, [ids[i]], [LENS[i]], tok0[i:i + 1], STEPS)
        assert np.array_equal(t1[:, 0], toks[:, i]), i
        for s in sampled:
            assert np.array_equal(s1[s][0], sampled[s][i]), (i, s)
    assert kd.kd_device_status(m) == 0
