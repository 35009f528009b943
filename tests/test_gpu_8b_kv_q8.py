"""The 8B-shaped decode step at long context with the Q8_0 KV cache.

Workload: the long-context multi-tenant case (Llama-3-8B-shaped, random Q8_0
weights, B = 8 sessions in slots of 32768 positions, pre-filled with seeded
N(0, 1) fp16 KV to 25704 + 1000 i positions) with KD_FLAG_KV_Q8_0: the pre-filled
rows and every appended row held as Q8_0 (136 bytes a head row).

Gates: at the first step the logits of the shortest and the longest session
within 5e-2 of the fp64 oracle over the same Q8_0 cache, and layers 0, 16 and 31
of both within 1e-3 relative L2 when fed the oracle's input; every session's
16-step greedy stream (tokens and logit bits) in the batch equal to its run alone."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SHAPE = synth.LLAMA3_8B
CASE = synth.LONG_CTX_8B_CASE
S, CAP = CASE["sessions"], CASE["capacity"]
LENS = [CASE["prefill_base"] + CASE["prefill_stagger"] * i for i in range(S)]
CHECKED = (0, S - 1)
STEPS = 16
LOGIT_TOL = 5e-2
HIDDEN_REL_L2 = 1e-3


@pytest.fixture(scope="module")
def q8_model(kdlib):
    kd = kdlib
    w = synth.model_weights(SHAPE, CASE["seed"])
    m = kd.kd_model_load(kd.make_config(SHAPE, S, CAP, kd.KD_FLAG_KV_Q8_0), w)
    ids, keep = [], {}
    try:
        for i, n in enumerate(LENS):
            k, v = synth.kv_prefill(SHAPE, CASE["seed"], 1000 + i, n)
            sid = kd.kd_session_bind(m)
            kd.kd_session_load_kv(m, sid, k, v, n)
            torch.cuda.synchronize()
            ids.append(sid)
            if i in CHECKED:
                keep[i] = (k, v)
        yield kd, m, w, ids, keep
    finally:
        kd.kd_model_free(m)


def test_8b_kv_q8_against_oracle(q8_model):
    kd, m, w, ids, keep = q8_model
    V, H, L = SHAPE.vocab, SHAPE.hidden, SHAPE.n_layers
    tok0 = synth.tokens(CASE["seed"], "8b-long", S, V)
    lg = torch.empty(S, V, device="cuda", dtype=torch.float32)
    kd.kd_decode_step(m, ids, tok0, LENS, lg, None)
    got = lg.cpu().numpy()
    om = oracle.OracleModel(SHAPE, w, kv_q8_0=True)
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


def greedy(kd, m, ids, starts, tok0, steps):
    B = len(ids)
    tok = np.array(tok0, np.int32)
    toks = np.empty((steps, B), np.int32)
    lgs = []
    lg = torch.empty(B, SHAPE.vocab, device="cuda", dtype=torch.float32)
    am = torch.empty(B, device="cuda", dtype=torch.int32)
    for s in range(steps):
        kd.kd_decode_step(m, ids, tok, [p + s for p in starts], lg, am)
        tok = am.cpu().numpy()
        toks[s] = tok
        if s % 4 == 3:
            lgs.append(lg.cpu().numpy().view(np.uint32).copy())
    return toks, lgs


def test_8b_kv_q8_batch_invariance(q8_model):
    kd, m, w, ids, keep = q8_model
    tok0 = synth.tokens(CASE["seed"], "8b-long-greedy", S, SHAPE.vocab)
    toks, lgs = greedy(kd, m, ids, LENS, tok0, STEPS)
    for i in (0, 3, S - 1):
        t1, l1 = greedy(kd, m, [ids[i]], [LENS[i]], tok0[i:i + 1], STEPS)
        assert np.array_equal(t1[:, 0], toks[:, i]), i
        for a, b in zip(l1, lgs):
            assert np.array_equal(a[0], b[i]), i
    assert kd.kd_device_status(m) == 0
