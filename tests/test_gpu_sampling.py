"""Device temperature sampling (Gumbel-max over Philox4x64-10), through the C ABI.

- kd_sample against the oracle's sampler on the same seeded fp32 logit rows (the
  lm_head's width, 128256), over many (temperature, seed, counter) rows: the same
  token, or -- where the oracle's two best perturbed values lie within a few fp32
  ulps, which libm's and CUDA's logf may order differently -- a near-tie.
- kd_decode_step_sampled on the tiny model: each session's sampled token stream
  and logit bits at B = 5 equal its run alone (the draw does not depend on the
  batch), greedy rows equal kd_decode_step's pick, and the first step's draws
  agree with the oracle's sampler applied to the oracle's logits (up to near-ties).
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def near_tie(logits_row, T, seed, ctr, got, want, ulps=8):
    zg = oracle.gumbel_perturbed(logits_row[got], got, T, seed, ctr)
    zw = oracle.gumbel_perturbed(logits_row[want], want, T, seed, ctr)
    return zw - zg <= ulps * np.spacing(np.float32(abs(zw)))


def test_sample_matches_oracle_on_lm_head_rows(kdlib):
    kd = kdlib
    B, V = 16, 128256
    x = synth.f32_normal(0, "sample-logits", (B, V)) * np.float32(3.0)
    x[3, 1000:1010] = np.nan  # NaN logits are never drawn
    xt = torch.from_numpy(x).cuda()
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = torch.zeros(kd.KD_SAMPLE_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    temps = [0.0, 0.25, 0.5, 0.7, 1.0, 1.0, 1.3, 2.0, 4.0, 0.9, 0.6, 1.1, -1.0, 0.8, 1.5, 3.0]
    checked, ties = 0, 0
    for rep in range(4):
        seeds = [1000 * rep + b for b in range(B)]
        ctrs = [7 * rep + 3 * b for b in range(B)]
        kd.kd_sample(xt, B, V, kd.sample_params(temps, seeds, ctrs), out, ws)
        got = out.cpu().numpy()
        for b in range(B):
            want = oracle.sample_f32(x[b], temps[b], seeds[b], ctrs[b])
            checked += 1
            if got[b] != want:
                assert temps[b] > 0 and near_tie(x[b], temps[b], seeds[b], ctrs[b], got[b], want), (rep, b, got[b], want)
                ties += 1
            if temps[b] <= 0:
                assert got[b] == oracle.argmax_f32(x[b])
    assert ties <= 2, ties
    assert checked == 64


def test_sample_draws_vary_with_counter_and_respect_temperature(kdlib):
    """Many counters at once on small rows: the draws' frequencies follow
    softmax(logits / T) (a chi-square test of the device draws themselves)."""
    kd = kdlib
    scipy_stats = pytest.importorskip("scipy.stats")
    V = 8
    logits = np.array([0.5, -1.0, 1.5, 0.0, 2.0, -0.5, 1.0, 0.2], np.float32)
    B = 16
    xt = torch.from_numpy(np.tile(logits, (B, 1))).cuda()
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = torch.zeros(kd.KD_SAMPLE_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    T = 0.9
    draws = []
    for rep in range(400):
        kd.kd_sample(xt, B, V, kd.sample_params([T] * B, [42] * B, [rep * B + b for b in range(B)]), out, ws)
        draws.append(out.cpu().numpy())
    d = np.concatenate(draws)
    p = np.exp(logits.astype(np.float64) / T)
    p /= p.sum()
    assert scipy_stats.chisquare(np.bincount(d, minlength=V), p * d.size).pvalue > 1e-4


@pytest.fixture(scope="module")
def tiny():
    shape = synth.TINY
    return shape, synth.model_weights(shape, 0)


def bind(kd, m, shape, lens, first=0):
    ids = []
    for i, n in enumerate(lens):
        k, v = synth.kv_prefill(shape, 0, first + i, n)
        sid = kd.kd_session_bind(m)
        kd.kd_session_load_kv(m, sid, k, v, n)
        ids.append(sid)
    return ids


def sampled_stream(kd, m, ids, lens, tok0, params_of, steps, V):
    B = len(ids)
    tok = np.array(tok0, np.int32)
    toks, lgs = [], []
    lg = torch.empty(B, V, device="cuda", dtype=torch.float32)
    out = torch.empty(B, device="cuda", dtype=torch.int32)
    for s in range(steps):
        kd.kd_decode_step_sampled(m, ids, tok, [n + s for n in lens], params_of(s), lg, out)
        tok = out.cpu().numpy()
        toks.append(tok.copy())
        lgs.append(lg.cpu().numpy().view(np.uint32).copy())
    return np.array(toks), np.array(lgs)


def test_sampled_step_is_batch_invariant_and_matches_oracle(kdlib, tiny):
    kd = kdlib
    shape, w = tiny
    cap, steps = 64, 6
    lens = [17, 40, 3, 9, 25]
    temps = [0.8, 0.0, 1.3, 0.5, 2.0]
    seeds = [11, 22, 33, 44, 55]
    tok0 = synth.tokens(0, "tiny-sample", len(lens), shape.vocab)
    m = kd.kd_model_load(kd.make_config(shape, 8, cap), w)
    try:
        ids = bind(kd, m, shape, lens)
        # first step: the draws against the oracle's sampler on the oracle's logits
        lg = torch.empty(len(ids), shape.vocab, device="cuda", dtype=torch.float32)
        out = torch.empty(len(ids), device="cuda", dtype=torch.int32)
        kd.kd_decode_step_sampled(m, ids, tok0, lens, kd.sample_params(temps, seeds, [0] * 5), lg, out)
        got = out.cpu().numpy()
        om = oracle.OracleModel(shape, w)
        caches = [om.new_cache(cap, *synth.kv_prefill(shape, 0, i, n)) for i, n in enumerate(lens)]
        ref, _, _ = om.step(tok0, lens, caches, cap)
        for b in range(len(lens)):
            want = oracle.sample_f32(ref[b], temps[b], seeds[b], 0)
            if got[b] != want:  # the logits agree to ~1e-7 here; only a near-tie may flip
                zg = oracle.gumbel_perturbed(ref[b][got[b]], int(got[b]), temps[b], seeds[b], 0)
                zw = oracle.gumbel_perturbed(ref[b][want], want, temps[b], seeds[b], 0)
                assert temps[b] > 0 and zw - zg < 1e-4, (b, got[b], want)
        # greedy rows equal kd_decode_step's pick
        am = torch.empty(len(ids), device="cuda", dtype=torch.int32)
        kd.kd_decode_step(m, ids, tok0, lens, None, am)
        assert am.cpu().numpy()[1] == got[1]
        # batch invariance of the sampled streams (counters: the step index)
        params_of = lambda s: kd.sample_params(temps, seeds, [s] * 5)
        batch_t, batch_l = sampled_stream(kd, m, ids, lens, tok0, params_of, steps, shape.vocab)
        for sid in ids:
            kd.kd_session_free(m, sid)
        for b in range(len(lens)):
            (sid,) = bind(kd, m, shape, [lens[b]], first=b)
            one = lambda s: kd.sample_params([temps[b]], [seeds[b]], [s])
            t1, l1 = sampled_stream(kd, m, [sid], [lens[b]], tok0[b:b + 1], one, steps, shape.vocab)
            assert np.array_equal(t1[:, 0], batch_t[:, b]), b
            assert np.array_equal(l1[:, 0], batch_l[:, b]), b
            kd.kd_session_free(m, sid)
        assert len(set(batch_t[:, 4].tolist())) > 1  # a hot row does not repeat one token
        assert kd.kd_device_status(m) == 0
    finally:
        kd.kd_model_free(m)
