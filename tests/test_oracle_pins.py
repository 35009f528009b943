"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these re-types an oracle formula: each compares the oracle with a
closed form, an invariant, a library routine the special case reduces to
(numpy's IEEE fp16 conversion, numpy matmul, scipy's logistic function), or a
brute-force evaluation on a tiny input.  Together they are chosen so that a
dropped term, a wrong sign, a wrong index or a transposed operand anywhere in
the oracle fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- fp16 -----
def test_half_decode_every_bit_pattern(oracle_lib):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_lib.kdo_half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_half_encode_rounds_like_ieee(oracle_lib):
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
        # exact midpoints between neighbouring halves (ties to even), incl. subnormals
        (np.arange(-3000, 3000).astype(np.float16).astype(np.float64)
         + np.nextafter(np.arange(-3000, 3000).astype(np.float16), np.float16(np.inf))
         .astype(np.float64)) / 2,
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -14 * (1 - 2.0 ** -11), np.inf, -np.inf]),
    ])
    ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle_lib.kdo_double_to_half(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)
    assert oracle.double_to_half(float("nan")) & 0x7C00 == 0x7C00


# ---------------------------------------------------------------- Q8_0 -----
def _golden_blocks():
    rows = []
    with open(os.path.join(GOLDEN, "q8_0_blocks.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if line:
                rows.append((int(line[0], 16), int(line[1]), float(line[2])))
    return rows


def test_q8_0_dequant_golden_blocks():
    for dbits, q, expect in _golden_blocks():
        blk = np.zeros(34, dtype=np.uint8)
        blk[0], blk[1] = dbits & 0xFF, dbits >> 8
        blk[2:] = np.array([q] * 32, dtype=np.int8).view(np.uint8)
        out = oracle.q8_0_dequant_row(blk, 32)
        assert np.all(out == expect), (hex(dbits), q, out[0], expect)


def test_q8_0_dequant_matches_closed_form_on_random_rows():
    m = synth.q8_0_matrix(3, "pin", 4, 256)
    d, qs = synth.q8_0_split(m)
    # about 30% of |N(0,0.02)|/127 scales are fp16 subnormals; they must not be flushed
    assert np.mean(d.astype(np.float64) < 2.0 ** -14) > 0.15
    for r in range(4):
        want = (qs[r].astype(np.float64) * d[r].astype(np.float64)[:, None]).reshape(-1)
        assert np.array_equal(oracle.q8_0_dequant_row(m[r], 256), want)


def test_matvec_against_numpy_matmul():
    m = synth.q8_0_matrix(4, "mv", 48, 96)
    d, qs = synth.q8_0_split(m)
    Wd = (qs.astype(np.float64) * d.astype(np.float64)[:, :, None]).reshape(48, 96)
    x = np.random.default_rng(5).standard_normal(96)
    y = oracle.matvec_q8_0(m, x)
    ref = Wd @ x
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-15)
    # a transposed operand or a mis-indexed block would not survive a non-square check
    x2 = np.zeros(96)
    x2[37] = 1.0
    assert np.array_equal(oracle.matvec_q8_0(m, x2), Wd[:, 37])


# ------------------------------------------------------------- RMSNorm -----
def test_rmsnorm_constant_row_closed_form():
    eps = 1e-5
    for c in (0.5, -3.0, 1e-3):
        x = np.full(64, c)
        w = np.linspace(0.5, 2.0, 64).astype(np.float32)
        want = (c / np.sqrt(c * c + eps) * w.astype(np.float64)).astype(np.float16).astype(np.float64)
        assert np.array_equal(oracle.rmsnorm_f16(x, w, eps), want)


def test_rmsnorm_uses_mean_not_sum():
    # x = (3, 4): mean(x^2) = 12.5, so with eps = 0 the outputs are 3/sqrt(12.5), 4/sqrt(12.5)
    out = oracle.rmsnorm_f16(np.array([3.0, 4.0]), np.ones(2, np.float32), 0.0)
    want = np.array([3 / math.sqrt(12.5), 4 / math.sqrt(12.5)]).astype(np.float16).astype(np.float64)
    assert np.array_equal(out, want)


def test_rmsnorm_scale_invariant():
    x = np.random.default_rng(6).standard_normal(256)
    w = np.ones(256, np.float32)
    a = oracle.rmsnorm_f16(x, w, 0.0)
    b = oracle.rmsnorm_f16(x * 8.0, w, 0.0)  # power of two: exact scaling
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- RoPE -----
def test_rope_position_zero_is_identity():
    u = np.random.default_rng(7).standard_normal(128)
    assert np.array_equal(oracle.rope_neox(u, 0, 500000.0), u)


def test_rope_neox_pairs_i_with_i_plus_half():
    hd = 128
    # frequency index 0 has w_0 = 1, so position p rotates pair (0, 64) by p radians
    e0 = np.zeros(hd)
    e0[0] = 1.0
    p = 3
    r = oracle.rope_neox(e0, p, 10000.0)
    want = np.zeros(hd)
    want[0], want[hd // 2] = math.cos(p), math.sin(p)
    assert np.allclose(r, want, atol=1e-15)
    # and the second component rotates towards -e_i
    e64 = np.zeros(hd)
    e64[hd // 2] = 1.0
    r = oracle.rope_neox(e64, p, 10000.0)
    want = np.zeros(hd)
    want[0], want[hd // 2] = -math.sin(p), math.cos(p)
    assert np.allclose(r, want, atol=1e-15)


def test_rope_frequency_schedule():
    hd, theta, p = 64, 10000.0, 5
    for i in (1, 7, 31):
        e = np.zeros(hd)
        e[i] = 1.0
        r = oracle.rope_neox(e, p, theta)
        ang = math.atan2(r[i + hd // 2], r[i])
        want = (p * theta ** (-2.0 * i / hd) + math.pi) % (2 * math.pi) - math.pi
        assert abs(ang - want) < 1e-12
        assert abs(np.linalg.norm(r) - 1.0) < 1e-14


def test_rope_relative_position_invariant():
    rng = np.random.default_rng(8)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    base = np.dot(oracle.rope_neox(q, 1000, 500000.0), oracle.rope_neox(k, 990, 500000.0))
    shifted = np.dot(oracle.rope_neox(q, 31010, 500000.0), oracle.rope_neox(k, 31000, 500000.0))
    assert abs(base - shifted) < 1e-9 * (1 + abs(base))


# ----------------------------------------------------------- attention -----
def _fp16_bits(a):
    return np.asarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def test_attention_against_two_pass_brute_force():
    rng = np.random.default_rng(9)
    for t in (1, 2, 17, 300):
        q = rng.standard_normal(64) * 2
        K = _fp16_bits(rng.standard_normal((t, 64)))
        V = _fp16_bits(rng.standard_normal((t, 64)))
        Kf = K.view(np.float16).astype(np.float64)
        Vf = V.view(np.float16).astype(np.float64)
        s = Kf @ q / math.sqrt(64)
        p = np.exp(s - s.max())
        want = (p / p.sum()) @ Vf
        assert np.allclose(oracle.attention_head(q, K, V), want, rtol=1e-12, atol=1e-14)


def test_attention_single_key_returns_its_value():
    rng = np.random.default_rng(10)
    V = _fp16_bits(rng.standard_normal((1, 128)))
    K = _fp16_bits(rng.standard_normal((1, 128)))
    out = oracle.attention_head(rng.standard_normal(128) * 50, K, V)
    assert np.array_equal(out, V.view(np.float16).astype(np.float64)[0])


def test_attention_identical_keys_average_values():
    rng = np.random.default_rng(11)
    K = np.repeat(_fp16_bits(rng.standard_normal((1, 64))), 9, axis=0)
    V = _fp16_bits(rng.standard_normal((9, 64)))
    out = oracle.attention_head(rng.standard_normal(64), K, V)
    assert np.allclose(out, V.view(np.float16).astype(np.float64).mean(0), rtol=1e-13, atol=1e-15)


# -------------------------------------------------------- SiLU, argmax -----
def test_silu_special_values_and_logistic():
    from scipy.special import expit
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12
    assert abs(oracle.silu(-40.0)) < 1e-15
    for y in np.linspace(-8, 8, 33):
        assert abs(oracle.silu(y) - y * expit(y)) < 1e-14


def test_argmax_ties_nan_and_degenerate_rows():
    v = np.array([0.5, 2.0, -1.0, 2.0, 1.0], np.float32)
    assert oracle.argmax_f32(v) == 1  # tie -> lowest index
    v = np.array([np.nan, 1.0, np.nan, 3.0, np.nan], np.float32)
    assert oracle.argmax_f32(v) == 3  # NaN never wins
    assert oracle.argmax_f32(np.full(4, np.nan, np.float32)) == -1
    assert oracle.argmax_f32(np.full(4, -np.inf, np.float32)) == 0
    big = np.random.default_rng(12).standard_normal(128256).astype(np.float32)
    big[77777] = 100.0
    assert oracle.argmax_f32(big) == 77777


# ------------------------------------------------------------ whole step ----
def _tiny(seed=0):
    shape = synth.TINY
    return shape, synth.model_weights(shape, seed)


def test_batch_equals_separate_runs():
    shape, w = _tiny()
    om = oracle.OracleModel(shape, w)
    cap = 64
    lens = (17, 40, 5)
    pre = [synth.kv_prefill(shape, 0, i, n) for i, n in enumerate(lens)]
    tok = synth.tokens(0, "pin-batch", 3, shape.vocab)
    caches = [om.new_cache(cap, *p) for p in pre]
    lg, am, hid = om.step(tok, lens, caches, cap, want_hidden=True)
    for b in range(3):
        c1 = om.new_cache(cap, *pre[b])
        lg1, am1, hid1 = om.step(tok[b:b + 1], [lens[b]], [c1], cap, want_hidden=True)
        assert np.array_equal(lg1[0], lg[b]) and am1[0] == am[b]
        assert np.array_equal(hid1[0], hid[b])
        assert np.array_equal(c1[0], caches[b][0]) and np.array_equal(c1[1], caches[b][1])


def test_step_writes_row_pos_and_ignores_rows_beyond():
    shape, w = _tiny()
    om = oracle.OracleModel(shape, w)
    cap, n = 64, 20
    kp, vp = synth.kv_prefill(shape, 0, 0, n)
    c_clean = om.new_cache(cap, kp, vp)
    c_dirty = om.new_cache(cap, kp, vp)
    nan16 = np.float16(np.nan).view(np.uint16)
    c_dirty[0][:, :, n + 1:] = nan16  # rows beyond the new token's position
    c_dirty[1][:, :, n + 1:] = nan16
    c_dirty[0][:, :, n] = nan16       # the row the step overwrites
    c_dirty[1][:, :, n] = nan16
    a = om.step([7], [n], [c_clean], cap)
    b = om.step([7], [n], [c_dirty], cap)
    assert np.array_equal(a[0], b[0])
    assert np.array_equal(c_clean[0][:, :, : n + 1], c_dirty[0][:, :, : n + 1])
    assert np.array_equal(c_clean[0][:, :, :n], kp)  # history untouched


def _dequant(m):
    d, qs = synth.q8_0_split(m)
    return (qs.astype(np.float64) * d.astype(np.float64)[:, :, None]).reshape(m.shape[0], -1)


def _f16(a):
    return np.asarray(a, np.float64).astype(np.float16).astype(np.float64)


def test_zero_mixer_and_ffn_outputs_reduce_to_head_of_embedding():
    # With W_o = 0 and W_down = 0 every layer adds exactly 0, so each hidden state is
    # the embedding row and the logits are lm_head(fp16(rmsnorm(embedding))).
    shape, w = _tiny()
    for l in range(shape.n_layers):
        for name in ("attn_output", "ffn_down"):
            m = w[f"blk.{l}.{name}"].copy()
            m[:, :, 2:] = 0
            w[f"blk.{l}.{name}"] = m
    om = oracle.OracleModel(shape, w)
    cap = 64
    c = om.new_cache(cap, *synth.kv_prefill(shape, 0, 0, 10))
    tok = 123
    lg, am, hid = om.step([tok], [10], [c], cap, want_hidden=True)
    e = _dequant(w["tok_embd"][tok:tok + 1])[0]
    for l in range(shape.n_layers + 1):
        assert np.array_equal(hid[0, l], e.astype(np.float32))
    hn = _f16(e / np.sqrt(np.mean(e * e) + shape.rms_eps))
    want = (_dequant(w["output"]) @ hn).astype(np.float32)
    assert np.allclose(lg[0], want, rtol=1e-6, atol=1e-6)
    assert am[0] == int(np.argmax(want))


def test_first_token_layer_matches_library_forward():
    # At position 0 attention over one key returns that key's value exactly, so the
    # whole layer reduces to numpy matmuls and scipy's logistic function.
    from scipy.special import expit
    shape, w = _tiny()
    om = oracle.OracleModel(shape, w)
    cap = 8
    c = om.new_cache(cap)
    tok = 77
    lg, am, hid = om.step([tok], [0], [c], cap, want_hidden=True)
    s = shape
    x = _dequant(w["tok_embd"][tok:tok + 1])[0]
    xn = _f16(x / np.sqrt(np.mean(x * x) + s.rms_eps))
    v = _dequant(w["blk.0.attn_v"]) @ xn
    group = s.n_heads // s.n_kv_heads
    att = np.concatenate([_f16(v[(h // group) * s.head_dim:(h // group + 1) * s.head_dim])
                          for h in range(s.n_heads)])
    x = (x + _dequant(w["blk.0.attn_output"]) @ att).astype(np.float32).astype(np.float64)
    z = _f16(x / np.sqrt(np.mean(x * x) + s.rms_eps))
    g, u = _dequant(w["blk.0.ffn_gate"]) @ z, _dequant(w["blk.0.ffn_up"]) @ z
    act = _f16(g * expit(g) * u)
    x = (x + _dequant(w["blk.0.ffn_down"]) @ act).astype(np.float32)
    assert np.allclose(hid[0, 1], x, rtol=1e-6, atol=1e-7)
    # the cache row 0 holds fp16(k at position 0) = fp16(W_k xn) (RoPE at 0 is the identity)
    k = _dequant(w["blk.0.attn_k"]) @ xn
    assert np.array_equal(c[0][0, :, 0].reshape(-1), k.astype(np.float16).view(np.uint16))


def test_gqa_head_mapping_and_cached_rows_brute_force():
    # Brute force of one layer's attention at a position > 0 with numpy, heads grouped
    # contiguously: q head h reads KV head h // (n_heads / n_kv_heads).
    shape, w = _tiny()
    s = shape
    om = oracle.OracleModel(shape, w)
    cap, n = 32, 11
    kp, vp = synth.kv_prefill(shape, 0, 1, n)
    c = om.new_cache(cap, kp, vp)
    tok = 5
    lg, am, hid = om.step([tok], [n], [c], cap, want_hidden=True)
    x = _dequant(w["tok_embd"][tok:tok + 1])[0]
    xn = _f16(x / np.sqrt(np.mean(x * x) + s.rms_eps))
    q = _dequant(w["blk.0.attn_q"]) @ xn
    hd, half = s.head_dim, s.head_dim // 2
    ang = n * s.rope_theta ** (-2.0 * np.arange(half) / hd)

    def rot(u):
        a, b = u[:half], u[half:]
        return np.concatenate([a * np.cos(ang) - b * np.sin(ang), a * np.sin(ang) + b * np.cos(ang)])

    Kc = c[0][0].view(np.float16).astype(np.float64)  # [n_kv][cap][hd], row n written by the step
    Vc = c[1][0].view(np.float16).astype(np.float64)
    att = []
    for h in range(s.n_heads):
        kh = h // (s.n_heads // s.n_kv_heads)
        sc = Kc[kh, : n + 1] @ rot(q[h * hd:(h + 1) * hd]) / math.sqrt(hd)
        p = np.exp(sc - sc.max())
        att.append(_f16(p @ Vc[kh, : n + 1] / p.sum()))
    x1 = (x + _dequant(w["blk.0.attn_output"]) @ np.concatenate(att)).astype(np.float32)
    # the residual after the mixer is not exposed, so compare through the FFN (as above)
    from scipy.special import expit
    x1 = x1.astype(np.float64)
    z = _f16(x1 / np.sqrt(np.mean(x1 * x1) + s.rms_eps))
    g, u = _dequant(w["blk.0.ffn_gate"]) @ z, _dequant(w["blk.0.ffn_up"]) @ z
    x2 = (x1 + _dequant(w["blk.0.ffn_down"]) @ _f16(g * expit(g) * u)).astype(np.float32)
    assert np.allclose(hid[0, 1], x2, rtol=1e-6, atol=1e-7)
