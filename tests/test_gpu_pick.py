"""The pick fused into the lm_head launch, through the C ABI.

When the lm_head runs on the stream schedule, its store epilogue also makes each
row's pick (greedy argmax, or Gumbel-max sampling with the row's temperature,
seed and counter), merging per-CTA best keys and finishing in the last CTA; no
pick kernel runs.  The pick kernels alone are pinned to the oracle elsewhere
(argmax edge cases, the oracle's sampler); here the fused pick must give the
same token, bit for bit, as those kernels applied to the logits the same step
stored.

Workload: a tiny model with a 32000-entry vocabulary (1000 row groups: the
stream schedule, as at the 8B shape), B = 1, 5, 8, 12, 16 sessions with
pre-filled fp16 positions, three fed-back steps each.  Ties: the same model
with the lm_head's second half a copy of its first, so every logit appears
twice, 16000 rows apart (in other CTAs); the lower index must win.  NaN: a NaN
in the output norm makes every logit NaN; every pick must be -1."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SHAPE = synth.TINY_WIDE_VOCAB
CAP = 64


@pytest.fixture(scope="module")
def weights():
    return dict(synth.model_weights(SHAPE, 0), **synth.norm_weights(SHAPE, 13))


def bind(kd, m, lens):
    ids = []
    for i, n in enumerate(lens):
        k, v = synth.kv_prefill(SHAPE, 0, i, n)
        sid = kd.kd_session_bind(m)
        kd.kd_session_load_kv(m, sid, k, v, n)
        ids.append(sid)
    return ids


def picks_of(kd, lg, B, sp=None):
    """The standalone pick kernels on stored logits, 16 rows per call; sp: the
    rows' (temperatures, seeds, counters) for sampling, or None."""
    got = []
    for r0 in range(0, B, 16):
        r1 = min(B, r0 + 16)
        out = torch.empty(r1 - r0, dtype=torch.int32, device="cuda")
        rows = lg[r0:r1].contiguous()
        if sp is None:
            ws = torch.zeros(kd.KD_ARGMAX_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
            kd.kd_argmax(rows, r1 - r0, SHAPE.vocab, out, ws)
        else:
            ws = torch.zeros(kd.KD_SAMPLE_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
            params = kd.sample_params(*(list(x[r0:r1]) for x in sp))
            kd.kd_sample(rows, r1 - r0, SHAPE.vocab, params, out, ws)
        got.append(out.cpu().numpy())
    return np.concatenate(got)


def run_and_compare(kd, m, B, sampled):
    lens = [3 + (7 * b) % 40 for b in range(B)]
    ids = bind(kd, m, lens)
    tok = synth.tokens(0, "pick", B, SHAPE.vocab)
    lg = torch.empty(B, SHAPE.vocab, device="cuda", dtype=torch.float32)
    out = torch.empty(B, device="cuda", dtype=torch.int32)
    temps = [(0.0 if b % 4 == 1 else 0.5 + 0.25 * b) for b in range(B)]
    try:
        for step in range(3):
            pos = [n + step for n in lens]
            if sampled:
                sp = (temps, [100 + b for b in range(B)], [step * 7 + b for b in range(B)])
                kd.kd_decode_step_sampled(m, ids, tok, pos, kd.sample_params(*sp), lg, out)
                want = picks_of(kd, lg, B, sp)
            else:
                kd.kd_decode_step(m, ids, tok, pos, lg, out)
                want = picks_of(kd, lg, B)
            got = out.cpu().numpy()
            assert np.array_equal(got, want), (B, sampled, step, got, want)
            tok = got
        assert kd.kd_device_status(m) == 0
        return got
    finally:
        for sid in ids:
            kd.kd_session_free(m, sid)


@pytest.mark.parametrize("B", [1, 5, 8, 12, 16])
def test_fused_pick_equals_the_pick_kernels(kdlib, weights, B):
    kd = kdlib
    m = kd.kd_model_load(kd.make_config(SHAPE, 16, CAP), weights)
    try:
        run_and_compare(kd, m, B, sampled=False)
        run_and_compare(kd, m, B, sampled=True)
        # the launch train has no pick kernel: the lm_head launch made the pick
        kd.kd_profile_enable(m, True)
        kd.kd_profile_read(m)
        run_and_compare(kd, m, B, sampled=False)
        prof = kd.kd_profile_read(m)
        kd.kd_profile_enable(m, False)
        assert prof["argmax"][0] == 0 and prof["lm_head"][0] == 3, prof
    finally:
        kd.kd_model_free(m)


def test_fused_pick_first_step_matches_oracle(kdlib, weights):
    """The first greedy step's tokens against the oracle's logits (up to a
    near-tie of the two best logits)."""
    kd = kdlib
    B = 5
    lens = [3 + (7 * b) % 40 for b in range(B)]
    tok = synth.tokens(0, "pick", B, SHAPE.vocab)
    m = kd.kd_model_load(kd.make_config(SHAPE, 16, CAP), weights)
    try:
        ids = bind(kd, m, lens)
        lg = torch.empty(B, SHAPE.vocab, device="cuda", dtype=torch.float32)
        out = torch.empty(B, device="cuda", dtype=torch.int32)
        kd.kd_decode_step(m, ids, tok, lens, lg, out)
        got = out.cpu().numpy()
    finally:
        kd.kd_model_free(m)
    om = oracle.OracleModel(SHAPE, weights)
    caches = [om.new_cache(CAP, *synth.kv_prefill(SHAPE, 0, i, n)) for i, n in enumerate(lens)]
    ref, _, _ = om.step(tok, lens, caches, CAP)
    for b in range(B):
        want = int(np.argmax(ref[b]))
        assert got[b] == want or ref[b][want] - ref[b][got[b]] < 1e-4, (b, got[b], want)


def test_fused_pick_ties_take_the_lower_index(kdlib, weights):
    kd = kdlib
    w = dict(weights)
    head = w["output"].copy()
    half = SHAPE.vocab // 2
    head[half:] = head[:half]
    w["output"] = head
    m = kd.kd_model_load(kd.make_config(SHAPE, 16, CAP), w)
    try:
        for B in (1, 8, 16):
            got = run_and_compare(kd, m, B, sampled=False)
            assert (got < half).all(), got
    finally:
        kd.kd_model_free(m)


def test_fused_pick_all_nan_rows_give_minus_one(kdlib, weights):
    """A NaN in the output norm makes every logit NaN: the fused pick, greedy and
    sampled, returns -1 for every row, as the pick kernels do."""
    kd = kdlib
    w = dict(weights)
    on = w["output_norm"].copy()
    on[7] = np.float32(np.nan)
    w["output_norm"] = on
    B = 5
    lens = [3 + (7 * b) % 40 for b in range(B)]
    tok = synth.tokens(0, "pick-nan", B, SHAPE.vocab)
    m = kd.kd_model_load(kd.make_config(SHAPE, 16, CAP), w)
    try:
        ids = bind(kd, m, lens)
        lg = torch.empty(B, SHAPE.vocab, device="cuda", dtype=torch.float32)
        out = torch.empty(B, device="cuda", dtype=torch.int32)
        kd.kd_decode_step(m, ids, tok, lens, lg, out)
        assert torch.isnan(lg).all()
        assert (out.cpu().numpy() == -1).all()
        assert (picks_of(kd, lg, B) == -1).all()
        sp = ([0.7] * B, list(range(B)), [0] * B)
        kd.kd_decode_step_sampled(m, ids, tok, lens, kd.sample_params(*sp), lg, out)
        assert (out.cpu().numpy() == -1).all()
        assert (picks_of(kd, lg, B, sp) == -1).all()
        assert kd.kd_device_status(m) == 0
    finally:
        kd.kd_model_free(m)


def test_fused_pick_in_groups_of_16(kdlib, weights):
    """B = 20 runs as groups of 16 and 4 rows: each group's lm_head makes its
    rows' picks, equal to the pick kernels on the logits the step stored."""
    kd = kdlib
    m = kd.kd_model_load(kd.make_config(SHAPE, 24, CAP), weights)
    try:
        run_and_compare(kd, m, 20, sampled=False)
        run_and_compare(kd, m, 20, sampled=True)
    finally:
        kd.kd_model_free(m)
