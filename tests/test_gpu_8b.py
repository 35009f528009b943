"""The 8B-shaped decode step through the C ABI.

Workload: a Llama-3-8B-shaped dense model with random Q8_0 weights (32 layers,
hidden 4096, 32/8 heads of 128, FFN 14336, vocab 128256), every session's slot
pre-filled with 1238 random fp16 positions (capacity 2048), seed 0.

Gates:
- teacher-forced logits within 5e-2 of the fp64 oracle for 4 of the 8 sessions
  of a B = 8 batch at steps 0, 1, 63 and 127, and every layer's output within
  1e-3 relative L2 of the oracle's when the layer is fed the oracle's input to it
  (through the step's own RMSNorm kernel);
- every session's greedy stream (tokens and logit bits) at B = 2, 4, 8, 16 equal
  to its isolated B = 1 run, over 128 steps.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SHAPE = synth.LLAMA3_8B
CASE = synth.DENSE_8B_CASE
PREFILL, CAP = CASE["prefill"], CASE["capacity"]


@pytest.fixture(scope="module")
def model8b(kdlib):
    kd = kdlib
    w = synth.model_weights(SHAPE, 0)
    m = kd.kd_model_load(kd.make_config(SHAPE, 16, CAP), w)
    kv = {}

    def prefill(i):
        if i not in kv:
            kv[i] = synth.kv_prefill(SHAPE, 0, i, PREFILL)
        return kv[i]

    yield kd, m, w, prefill
    kd.kd_model_free(m)


def bind(kd, m, prefill, sessions):
    ids = []
    for i in sessions:
        sid = kd.kd_session_bind(m)
        k, v = prefill(i)
        kd.kd_session_load_kv(m, sid, k, v, PREFILL)
        ids.append(sid)
    return ids


def free(kd, m, ids):
    for sid in ids:
        kd.kd_session_free(m, sid)


# End to end, the hidden states of this random-weight model are sensitive to the
# fp16 rounding points themselves: the oracle moves by > 1e-3 (relative L2) at
# depth when one norm weight is nudged by 2^-20 (tests/test_oracle_sensitivity.py).
# So 1e-3 is checked per layer (each layer fed the oracle's input to that layer);
# end to end the hidden states are held to a bound above that sensitivity.
HIDDEN_REL_L2 = 1e-3
HIDDEN_REL_L2_END_TO_END = 1e-2


CHECKED = (0, 2, 5, 7)        # sessions of the B = 8 batch compared with the oracle
SAMPLED = (0, 1, 63, 127)     # steps at which they are compared


def oracle_stream(om, prefill, b, tok0, steps, cap):
    """Session b run alone by the oracle for `steps` greedy steps from its own
    argmax (teacher forcing): its input tokens, and its logits and hidden
    states at the sampled steps."""
    cache = om.new_cache(cap, *prefill(b))
    tok = np.array([tok0], np.int32)
    toks, logits, hidden = [], {}, {}
    for s in range(steps):
        lg, am, h = om.step(tok, [PREFILL + s], [cache], cap, want_hidden=s in SAMPLED)
        toks.append(int(tok[0]))
        if s in SAMPLED:
            logits[s], hidden[s] = lg[0], h[0]
        tok = am.copy()
    return toks, logits, hidden


def test_8b_teacher_forced_against_oracle(model8b):
    """Teacher forcing over the workload's 128 steps: the checked sessions' inputs
    are the oracle's own greedy tokens; the other rows follow the GPU's.  At the
    sampled steps the checked rows' logits must be within 5e-2 of the oracle's and
    their hidden states within the end-to-end bound."""
    kd, m, w, prefill = model8b
    B, L, H, V = 8, SHAPE.n_layers, SHAPE.hidden, SHAPE.vocab
    steps = CASE["steps"]
    cap = PREFILL + steps
    om = oracle.OracleModel(SHAPE, w)
    tok0 = synth.tokens(0, "8b-steps", B, V)
    ref = {b: oracle_stream(om, prefill, b, int(tok0[b]), steps, cap) for b in CHECKED}
    ids = bind(kd, m, prefill, range(B))
    hid = torch.empty(L + 1, B, H, device="cuda", dtype=torch.float32)
    lg = torch.empty(B, V, device="cuda", dtype=torch.float32)
    am = torch.empty(B, device="cuda", dtype=torch.int32)
    try:
        tok = tok0.copy()
        for step in range(steps):
            for b in CHECKED:
                tok[b] = ref[b][0][step]
            kd.kd_debug_capture_hidden(m, hid if step in SAMPLED else None)
            kd.kd_decode_step(m, ids, tok, [PREFILL + step] * B, lg, am)
            torch.cuda.synchronize()
            if step in SAMPLED:
                got, gh = lg.cpu().numpy(), hid.cpu().numpy()
                for b in CHECKED:
                    err = float(np.abs(got[b] - ref[b][1][step]).max())
                    assert err <= 5e-2, (step, b, err)
                    for l in range(L + 1):
                        want = ref[b][2][step][l]
                        rel = np.linalg.norm(gh[l, b] - want) / np.linalg.norm(want)
                        assert rel <= HIDDEN_REL_L2_END_TO_END, (step, b, l, rel)
            tok = am.cpu().numpy()
        assert kd.kd_device_status(m) == 0
    finally:
        kd.kd_debug_capture_hidden(m, None)
        free(kd, m, ids)


def test_8b_each_layer_against_oracle(model8b):
    kd, m, w, prefill = model8b
    L, H = SHAPE.n_layers, SHAPE.hidden
    sessions = (1, 6)
    om = oracle.OracleModel(SHAPE, w)
    tok = synth.tokens(0, "8b-layers", len(sessions), SHAPE.vocab)
    ref_h = []
    for j, b in enumerate(sessions):
        c = om.new_cache(PREFILL + 1, *prefill(b))
        _, _, h = om.step(tok[j:j + 1], [PREFILL], [c], PREFILL + 1, want_hidden=True)
        ref_h.append(h[0])
    ref_h = np.stack(ref_h, axis=1)  # [L+1][B][H]
    ids = bind(kd, m, prefill, sessions)
    try:
        x_out = torch.empty(len(sessions), H, device="cuda", dtype=torch.float32)
        worst = 0.0
        for l in range(L):
            x_in = torch.from_numpy(np.ascontiguousarray(ref_h[l])).cuda()
            kd.kd_debug_layer(m, l, ids, [PREFILL] * len(sessions), x_in, x_out)
            got = x_out.cpu().numpy()
            for j in range(len(sessions)):
                rel = np.linalg.norm(got[j] - ref_h[l + 1, j]) / np.linalg.norm(ref_h[l + 1, j])
                worst = max(worst, rel)
                assert rel <= HIDDEN_REL_L2, (l, sessions[j], rel)
        assert kd.kd_device_status(m) == 0
        print(f"worst per-layer relative L2: {worst:.3e}")
    finally:
        free(kd, m, ids)


def greedy(kd, m, ids, tok0, steps):
    B = len(ids)
    tok = np.array(tok0, np.int32)
    toks = np.empty((steps, B), np.int32)
    logits = []
    lg = torch.empty(B, SHAPE.vocab, device="cuda", dtype=torch.float32)
    am = torch.empty(B, device="cuda", dtype=torch.int32)
    for s in range(steps):
        kd.kd_decode_step(m, ids, tok, [PREFILL + s] * B, lg, am)
        tok = am.cpu().numpy()
        toks[s] = tok
        if s % 16 == 0 or s == steps - 1:
            logits.append(lg.cpu().numpy().view(np.uint32).copy())
    return toks, logits


def test_8b_batch_invariance_of_greedy_streams(model8b):
    kd, m, w, prefill = model8b
    steps = CASE["steps"]
    tok0 = synth.tokens(0, "8b-greedy", 16, SHAPE.vocab)
    alone = {}
    for i in range(16):
        ids = bind(kd, m, prefill, [i])
        alone[i] = greedy(kd, m, ids, tok0[i:i + 1], steps)
        free(kd, m, ids)
    for B in (2, 4, 8, 16):
        ids = bind(kd, m, prefill, range(B))
        toks, logits = greedy(kd, m, ids, tok0[:B], steps)
        free(kd, m, ids)
        for i in range(B):
            assert np.array_equal(toks[:, i], alone[i][0][:, 0]), (B, i)
            for a, b in zip(logits, alone[i][1]):
                assert np.array_equal(a[i], b[0]), (B, i)
    assert kd.kd_device_status(m) == 0
