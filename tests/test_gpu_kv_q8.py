"""The Q8_0 KV cache (KD_FLAG_KV_Q8_0) on the GPU against the CPU oracle.

Workloads:
- the quantiser: seeded fp32 rows of 128 with per-row magnitudes from 1e-3 to 1e3,
  an all-zero block, exact halves (x / d = k + 1/2) and values at +-max;
- the isolated attention with 128-wide heads over Q8_0 rows: groups 1, 2, 4, 8,
  ragged attended lengths around the 64-key split boundaries, and the long-context
  configuration (32 query / 8 KV heads, B = 8, lengths uniform in [1, 32768]);
  the history is quantised by the oracle from seeded N(0, 1) rows scaled per row
  by U(0.05, 4), the rows nothing should read hold NaN scales;
- the whole step on the 2-layer hd-128 tiny model, three sessions pre-filled to
  17, 64 and 70 positions, 6 teacher-forced steps, seeded non-unit norms.

Gates: quantised bytes (the appended rows included) bit-identical to the oracle's;
attention outputs within one fp16 ulp + 1e-4 of the fp64 oracle; one key gives its
dequantised value exactly; step logits within 5e-2 and hidden states within 1e-3
relative L2; every session's stream in the batch bit-identical to its run alone."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

HD = 128


def assert_close_fp16(got16, ref):
    got = got16.astype(np.float64)
    tol = 2.0 ** -10 * np.abs(ref) + 1e-4
    err = np.abs(got - ref)
    assert np.all(err <= tol), float((err / tol).max())


def oracle_blocks(x):
    """The oracle's Q8_0 rows [..][4][34] of fp32 rows [..][128]."""
    x = np.ascontiguousarray(x, np.float32)
    return oracle.q8_0_quantize_f32(x).reshape(*x.shape[:-1], HD // 32, 34)


def to_planes(blocks):
    """Q8_0 rows [..][4][34] -> the device's planes: quants (q + 128, uint8 [..][128])
    and fp16 scale bits (uint16 [..][4])."""
    b = np.ascontiguousarray(blocks, np.uint8)
    q = (b[..., 2:].view(np.int8).astype(np.int16) + 128).astype(np.uint8).reshape(*b.shape[:-2], HD)
    sc = np.ascontiguousarray(b[..., 0:2]).view(np.uint16).reshape(*b.shape[:-2], HD // 32)
    return q, sc


def test_quantizer_bytes_equal_oracle(kdlib):
    kd = kdlib
    rng = synth.substream(0, "kv-q8-quant")
    rows = 4099
    x = rng.standard_normal((rows, HD), dtype=np.float32)
    x *= np.float32(10.0) ** rng.uniform(-3, 3, (rows, 1)).astype(np.float32)
    x[7, 32:64] = 0.0                                      # an all-zero block
    x[8, :32] = np.arange(32, dtype=np.float32) - 15.5     # d = 16.5/127: many near-halves
    x[9, :32] = 0.0
    x[9, 0], x[9, 1], x[9, 2] = 127.0, 2.5, -2.5           # d = 1: exact halves
    x[10, 96:] = -np.abs(x[10, 96:])                       # every value of the block negative
    want_q, want_s = to_planes(oracle_blocks(x))
    src = torch.from_numpy(x).cuda()
    q = torch.empty(rows, HD, dtype=torch.uint8, device="cuda")
    s = torch.empty(rows, HD // 32, dtype=torch.int16, device="cuda")
    kd.kd_kv_q8_quantize(src, q, s)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), want_q)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), want_s)


def make_case(seed, B, nh, nkv, lens, n_slots, cap):
    """Slots, the oracle's Q8_0 history rows per (slot, kv head), the device planes
    (unfilled rows: arbitrary quants, NaN scales), q and the new k, v rows."""
    rng = np.random.default_rng(seed)
    slots = rng.permutation(n_slots)[:B].astype(np.int32)
    planes = {}
    for name in ("k", "v"):
        planes[name] = (np.full((n_slots, nkv, cap, HD), 0x5A, np.uint8),
                        np.full((n_slots, nkv, cap, HD // 32), 0x7E00, np.uint16))
    hist = {}
    for b in range(B):
        n = lens[b] - 1  # history rows; the step appends row n
        sub = synth.substream(seed, "attn-kv-q8", b)
        for name in ("k", "v"):
            x = sub.standard_normal((nkv, n, HD), dtype=np.float32)
            x *= sub.uniform(0.05, 4.0, (nkv, n, 1)).astype(np.float32)
            blk = oracle_blocks(x) if n else np.zeros((nkv, 0, HD // 32, 34), np.uint8)
            hist[name, b] = blk
            qp, sp = to_planes(blk)
            planes[name][0][slots[b], :, :n] = qp
            planes[name][1][slots[b], :, :n] = sp
    q = synth.f32_normal(seed, "attn-q8-q", (B, nh, HD))
    kn = synth.f32_normal(seed, "attn-q8-k", (B, nkv, HD)) * np.float32(2.0)
    vn = synth.f32_normal(seed, "attn-q8-v", (B, nkv, HD)) * np.float32(0.5)
    return slots, hist, planes, q, kn, vn


def upload(planes):
    return {k: (torch.from_numpy(qp).cuda(), torch.from_numpy(sp.view(np.int16)).cuda())
            for k, (qp, sp) in planes.items()}


def run_gpu(kd, slots, dev, q, kn, vn, pos, nh, nkv, n_slots, cap):
    B = len(slots)
    out = torch.empty(B, nh * HD, dtype=torch.int16, device="cuda")
    ws = torch.empty(kd.kd_attn_workspace_bytes(B, nh, HD, cap), dtype=torch.uint8, device="cuda")
    kd.kd_attn_append_decode_q8(torch.from_numpy(q).cuda(), torch.from_numpy(kn).cuda(),
                                torch.from_numpy(vn).cuda(), dev["k"][0], dev["k"][1], dev["v"][0], dev["v"][1],
                                slots, pos, nh, nkv, n_slots, cap, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.float16)


def oracle_attn(hist, q, kn, vn, pos, nh, nkv):
    B = q.shape[0]
    group = nh // nkv
    ref = np.empty((B, nh, HD))
    for b in range(B):
        K = np.concatenate([hist["k", b], oracle_blocks(kn[b])[:, None]], axis=1)
        V = np.concatenate([hist["v", b], oracle_blocks(vn[b])[:, None]], axis=1)
        assert K.shape[1] == pos[b] + 1
        for h in range(nh):
            ref[b, h] = oracle.attention_head_q8(q[b, h].astype(np.float64), K[h // group], V[h // group])
    return ref.reshape(B, nh * HD)


def check_appended(dev, slots, kn, vn, pos):
    for name, new in (("k", kn), ("v", vn)):
        dq = dev[name][0].cpu().numpy()
        ds = dev[name][1].cpu().numpy().view(np.uint16)
        wq, ws = to_planes(oracle_blocks(new))
        for b in range(len(slots)):
            assert np.array_equal(dq[slots[b], :, pos[b]], wq[b]), (name, b)
            assert np.array_equal(ds[slots[b], :, pos[b]], ws[b]), (name, b)


@pytest.mark.parametrize("nh,nkv,lens", [
    (32, 8, [1, 2, 63, 64, 65, 127, 128, 129]),
    (8, 8, [1, 5, 130]),
    (16, 8, [255, 257, 513]),
    (16, 2, [100, 700, 1000]),
])
def test_attention_q8_small_ragged(kdlib, nh, nkv, lens):
    kd = kdlib
    B, cap, n_slots = len(lens), 1024, len(lens) + 3
    slots, hist, planes, q, kn, vn = make_case(5, B, nh, nkv, lens, n_slots, cap)
    pos = np.array(lens, np.int32) - 1
    dev = upload(planes)
    got = run_gpu(kd, slots, dev, q, kn, vn, pos, nh, nkv, n_slots, cap)
    assert_close_fp16(got, oracle_attn(hist, q, kn, vn, pos, nh, nkv))
    check_appended(dev, slots, kn, vn, pos)


def test_attention_q8_single_key_is_dequantised_value(kdlib):
    kd = kdlib
    nh, nkv, cap = 32, 8, 16
    slots, hist, planes, q, kn, vn = make_case(9, 3, nh, nkv, [1, 1, 1], 4, cap)
    pos = np.zeros(3, np.int32)
    got = run_gpu(kd, slots, upload(planes), q * 30, kn, vn, pos, nh, nkv, 4, cap)
    deq = np.stack([[oracle.q8_0_dequant_row(r.reshape(-1), HD) for r in oracle_blocks(vn[b])] for b in range(3)])
    want = np.repeat(deq.astype(np.float16), nh // nkv, axis=1).reshape(3, nh * HD)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))


def test_attention_q8_long_context_batch_invariant(kdlib):
    kd = kdlib
    nh, nkv, cap, B = 32, 8, 32768, 8
    lens = synth.ragged_lengths(0, "attn-config", B, 1, cap)
    slots, hist, planes, q, kn, vn = make_case(0, B, nh, nkv, lens, B, cap)
    pos = lens - 1
    dev = upload(planes)
    got = run_gpu(kd, slots, dev, q, kn, vn, pos, nh, nkv, B, cap)
    assert_close_fp16(got, oracle_attn(hist, q, kn, vn, pos, nh, nkv))
    check_appended(dev, slots, kn, vn, pos)
    for b in (0, 3, 7):  # each session alone gives the same bits
        one = run_gpu(kd, slots[b:b + 1], dev, q[b:b + 1], kn[b:b + 1], vn[b:b + 1], pos[b:b + 1], nh, nkv, B, cap)
        assert np.array_equal(one[0].view(np.uint16), got[b].view(np.uint16)), b


# ---- the whole step with the Q8_0 cache ------------------------------------------
LOGIT_TOL = 5e-2
HIDDEN_REL_L2 = 1e-3


@pytest.fixture(scope="module")
def tiny128():
    case = synth.TINY_KV_Q8_CASE
    shape = case["shape"]
    w = synth.model_weights(shape, case["seed"])
    return shape, dict(w, **synth.norm_weights(shape, 3)), case


def load_bound(kd, shape, w, case, cap, flags):
    m = kd.kd_model_load(kd.make_config(shape, 4, cap, flags | kd.KD_FLAG_KV_Q8_0), w)
    ids = []
    for i, n in enumerate(case["prefill"]):
        k, v = synth.kv_prefill(shape, case["seed"], i, n)
        sid = kd.kd_session_bind(m)
        kd.kd_session_load_kv(m, sid, k, v, n)
        torch.cuda.synchronize()
        ids.append(sid)
    return m, ids


# 0: schedules as chosen; 1: direct launches instead of the graph; 2 / 4: every
# projection forced onto the stream / group schedule (both write the fp32 k, v rows
# the append quantises).
@pytest.mark.parametrize("flags", [0, 1, 2, 4])
def test_tiny_kv_q8_teacher_forced_against_oracle(kdlib, tiny128, flags):
    kd = kdlib
    shape, w, case = tiny128
    cap = 128
    lens = list(case["prefill"])
    m, ids = load_bound(kd, shape, w, case, cap, flags)
    try:
        om = oracle.OracleModel(shape, w, kv_q8_0=True)
        caches = [om.new_cache(cap, *synth.kv_prefill(shape, case["seed"], i, n)) for i, n in enumerate(lens)]
        B, L, H, V = len(lens), shape.n_layers, shape.hidden, shape.vocab
        hid = torch.empty(L + 1, B, H, device="cuda", dtype=torch.float32)
        kd.kd_debug_capture_hidden(m, hid)
        lg = torch.empty(B, V, device="cuda", dtype=torch.float32)
        am = torch.empty(B, device="cuda", dtype=torch.int32)
        tok = synth.tokens(case["seed"], "tiny-kv-q8", B, V)
        for step in range(case["steps"]):
            pos = [n + step for n in lens]
            kd.kd_decode_step(m, ids, tok, pos, lg, am)
            torch.cuda.synchronize()
            ref, ref_am, ref_h = om.step(tok, pos, caches, cap, want_hidden=True)
            err = float(np.abs(lg.cpu().numpy() - ref).max())
            assert err <= LOGIT_TOL, (step, err)
            gh = hid.cpu().numpy()
            for b in range(B):
                for l in range(L + 1):
                    rel = np.linalg.norm(gh[l, b] - ref_h[b, l]) / np.linalg.norm(ref_h[b, l])
                    assert rel <= HIDDEN_REL_L2, (step, b, l, rel)
            tok = ref_am
        assert kd.kd_device_status(m) == 0
    finally:
        kd.kd_model_free(m)


def test_tiny_kv_q8_batch_invariance(kdlib, tiny128):
    kd = kdlib
    shape, w, case = tiny128
    cap, steps = 128, case["steps"]
    lens = list(case["prefill"])
    m, ids = load_bound(kd, shape, w, case, cap, 0)
    V = shape.vocab

    def stream(sel):
        B = len(sel)
        tok = synth.tokens(case["seed"], "tiny-kv-q8-greedy", len(lens), V)[sel]
        lg = torch.empty(B, V, device="cuda", dtype=torch.float32)
        am = torch.empty(B, device="cuda", dtype=torch.int32)
        toks, lgs = [], []
        for s in range(steps):
            kd.kd_decode_step(m, [ids[i] for i in sel], tok, [lens[i] + s for i in sel], lg, am)
            tok = am.cpu().numpy()
            toks.append(tok.copy())
            lgs.append(lg.cpu().numpy().view(np.uint32).copy())
        return np.array(toks), np.array(lgs)
    try:
        toks, lgs = stream([0, 1, 2])
        for i in range(3):
            t1, l1 = stream([i])
            assert np.array_equal(t1[:, 0], toks[:, i]), i
            assert np.array_equal(l1[:, 0], lgs[:, i]), i
        assert kd.kd_device_status(m) == 0
    finally:
        kd.kd_model_free(m)


def greedy_streams(kd, m, ids, starts, tok0, steps, V, params=None):
    B = len(ids)
    tok = np.array(tok0, np.int32)
    toks, lgs = [], []
    lg = torch.empty(B, V, device="cuda", dtype=torch.float32)
    am = torch.empty(B, device="cuda", dtype=torch.int32)
    for s_ in range(steps):
        pos = [p + s_ for p in starts]
        if params is None:
            kd.kd_decode_step(m, ids, tok, pos, lg, am)
        else:
            sp = kd.sample_params([p["temperature"] for p in params], [p["seed"] for p in params], [s_] * B)
            kd.kd_decode_step_sampled(m, ids, tok, pos, sp, lg, am)
        tok = am.cpu().numpy()
        toks.append(tok.copy())
        lgs.append(lg.cpu().numpy().view(np.uint32).copy())
    return np.array(toks), np.array(lgs)


def test_tiny_kv_q8_fused_bitwise_equal_unfused_train(kdlib, tiny128):
    """The q|k|v epilogue's fp32 k, v rows and the append kernel: the fused step
    and the unfused train (plain projections, epilogues as kernels of their own)
    give the same logits, through later steps' attention over the appended rows."""
    kd = kdlib
    shape, w, case = tiny128
    lens = list(case["prefill"])
    runs = []
    for flags in (0, kd.KD_FLAG_UNFUSED):
        m, ids = load_bound(kd, shape, w, case, 128, flags)
        try:
            runs.append(greedy_streams(kd, m, ids, lens, synth.tokens(0, "q8-unfused", len(lens), shape.vocab),
                                       case["steps"], shape.vocab))
            assert kd.kd_device_status(m) == 0
        finally:
            kd.kd_model_free(m)
    assert np.array_equal(runs[0][0], runs[1][0])
    assert np.array_equal(runs[0][1], runs[1][1])


def test_tiny_kv_q8_many_sessions_and_sampling(kdlib, tiny128):
    """20 sessions (groups of 16 and 4 rows) with the Q8_0 cache, greedy and
    sampled: every session's tokens and logit bits equal its run alone."""
    kd = kdlib
    shape, w, case = tiny128
    n = 20
    lens = [5 + 5 * i for i in range(n)]
    m = kd.kd_model_load(kd.make_config(shape, n, 128, kd.KD_FLAG_KV_Q8_0), w)
    try:
        ids = []
        for i, L0 in enumerate(lens):
            k, v = synth.kv_prefill(shape, case["seed"], 100 + i, L0)
            sid = kd.kd_session_bind(m)
            kd.kd_session_load_kv(m, sid, k, v, L0)
            ids.append(sid)
        torch.cuda.synchronize()
        tok0 = synth.tokens(0, "q8-many", n, shape.vocab)
        params = [dict(temperature=0.7 + 0.1 * (i % 4), seed=1000 + i) for i in range(n)]
        for p in (None, params):
            toks, lgs = greedy_streams(kd, m, ids, lens, tok0, 3, shape.vocab, p)
            for i in (0, 7, 15, 16, 19):
                t1, l1 = greedy_streams(kd, m, [ids[i]], [lens[i]], tok0[i:i + 1], 3, shape.vocab,
                                        None if p is None else p[i:i + 1])
                assert np.array_equal(t1[:, 0], toks[:, i]), (p is None, i)
                assert np.array_equal(l1[:, 0], lgs[:, i]), (p is None, i)
        assert kd.kd_device_status(m) == 0
    finally:
        kd.kd_model_free(m)


def test_tiny_kv_q8_attention_wait_runs_out_and_recovers(kdlib, tiny128):
    """One bounded wait of the Q8_0 attention kernel made to run out: the step
    reports KD_ERR_DEVICE, and the next step (rewound) matches the oracle."""
    kd = kdlib
    shape, w, case = tiny128
    cap = 128
    lens = list(case["prefill"])
    m, ids = load_bound(kd, shape, w, case, cap, 0)
    try:
        om = oracle.OracleModel(shape, w, kv_q8_0=True)
        caches = [om.new_cache(cap, *synth.kv_prefill(shape, case["seed"], i, L0)) for i, L0 in enumerate(lens)]
        tok = synth.tokens(case["seed"], "q8-fault", len(lens), shape.vocab)
        ref, _, _ = om.step(tok, lens, caches, cap)
        lg = torch.empty(len(ids), shape.vocab, device="cuda", dtype=torch.float32)
        kd.kd_debug_inject_wait_timeout(m, "attn_split")
        kd.kd_decode_step(m, ids, tok, lens, lg, None)
        torch.cuda.synchronize()
        kd.kd_decode_step(m, ids, tok, lens, lg, None)
        torch.cuda.synchronize()
        assert float(np.abs(lg.cpu().numpy() - ref).max()) <= LOGIT_TOL
        with pytest.raises(kd.KdError) as e:
            kd.kd_device_status(m)
        assert e.value.name == "KD_ERR_DEVICE"
        assert kd.kd_device_status(m) == 0
    finally:
        kd.kd_model_free(m)
