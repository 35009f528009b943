"""Pins of the oracle's Q8_0 KV cache: the quantiser and the attention over Q8_0 rows.

Quantiser (fp32; per 32-value block d = max|x| / 127 stored as fp16, q = x / d
rounded half away from zero): a block that is already q * d with max |q| = 127
and a normal fp16 d comes back unchanged, byte for byte; zeros give d = 0; the
largest value maps to +-127; every value is within d/2 (plus the fp16 rounding
of d) of its dequantised one; scaling by a power of two scales d only; x / d =
2.5 rounds to 3.  Attention over Q8_0 rows equals a numpy two-pass softmax over
the rows dequantised by the (separately pinned) Q8_0 dequantiser."""
import numpy as np

import oracle
import synth


def _blocks(d16, qs):
    """Canonical blocks from fp16 scales [n] and int8 quants [n][32]."""
    return synth.q8_0_from_parts(np.asarray(d16, np.float16)[None, :], np.asarray(qs, np.int8)[None])[0]


def test_exact_blocks_round_trip():
    rng = np.random.default_rng(0)
    for _ in range(50):
        d = np.float16(rng.uniform(1e-3, 4.0))
        qs = rng.integers(-127, 128, size=32).astype(np.int8)
        qs[rng.integers(0, 32)] = rng.choice([-127, 127])
        blk = _blocks([d], [qs])
        x = oracle.q8_0_dequant_row(blk.reshape(-1), 32).astype(np.float32)
        assert np.array_equal(oracle.q8_0_quantize_f32(x).reshape(-1), blk.reshape(-1))


def test_zero_block_and_extremes():
    z = oracle.q8_0_quantize_f32(np.zeros(32, np.float32))
    assert np.all(z == 0)
    x = np.random.default_rng(1).standard_normal(64).astype(np.float32)
    b = oracle.q8_0_quantize_f32(x)
    for k in range(2):
        qs = b[k, 2:].view(np.int8)
        j = np.argmax(np.abs(x[32 * k:32 * k + 32]))
        assert abs(int(qs[j])) == 127 and np.sign(qs[j]) == np.sign(x[32 * k + j])


def test_error_bound_and_power_of_two_scaling():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(32 * 40) * rng.uniform(0.01, 10, 32 * 40)).astype(np.float32)
    b = oracle.q8_0_quantize_f32(x)
    deq = oracle.q8_0_dequant_row(b.reshape(-1), x.size)
    for k in range(40):
        xb = x[32 * k:32 * k + 32].astype(np.float64)
        d = np.abs(xb).max() / 127
        dh = float(b[k, 0:2].view(np.float16)[0])
        assert np.all(np.abs(xb - deq[32 * k:32 * k + 32]) <= 0.5 * d + 127 * abs(d - dh) + 1e-12)
    b2 = oracle.q8_0_quantize_f32(x * np.float32(8.0))
    assert np.array_equal(b2[:, 2:], b[:, 2:])
    assert np.array_equal(b2[:, 0:2].view(np.float16).astype(np.float64), b[:, 0:2].view(np.float16).astype(np.float64) * 8)


def test_halves_round_away_from_zero():
    x = np.zeros(32, np.float32)
    x[0], x[1], x[2], x[3] = 127.0, 2.5, -2.5, 0.5  # d = 1 exactly
    qs = oracle.q8_0_quantize_f32(x)[0, 2:].view(np.int8)
    assert qs[:4].tolist() == [127, 3, -3, 1]


def test_attention_over_q8_rows_matches_two_pass_softmax():
    rng = np.random.default_rng(3)
    for t, hd in ((1, 64), (37, 128), (200, 64)):
        K = rng.standard_normal((t, hd)).astype(np.float32)
        V = rng.standard_normal((t, hd)).astype(np.float32)
        Kq = np.stack([oracle.q8_0_quantize_f32(r) for r in K])
        Vq = np.stack([oracle.q8_0_quantize_f32(r) for r in V])
        Kd = np.stack([oracle.q8_0_dequant_row(r.reshape(-1), hd) for r in Kq])
        Vd = np.stack([oracle.q8_0_dequant_row(r.reshape(-1), hd) for r in Vq])
        q = rng.standard_normal(hd)
        s = Kd @ q / np.sqrt(hd)
        p = np.exp(s - s.max())
        want = (p @ Vd) / p.sum()
        got = oracle.attention_head_q8(q, Kq, Vq)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12), (t, hd)
        if t == 1:
            assert np.allclose(got, Vd[0], rtol=1e-14, atol=0)
