"""bench.py's algorithmic bytes per step -- the numerator of every GB/s and
roofline fraction it reports -- against the byte count written out from the
model's shape (no GPU): every Q8_0 weight once (34 bytes per 32 weights), the B
embedding rows, the fp16 K and V rows each session attends (its position + 1,
all layers and KV heads) and the B new rows written."""
import pytest

import bench
import synth


def by_hand(shape, positions):
    s = shape
    qkv = (s.n_heads + 2 * s.n_kv_heads) * s.head_dim * s.hidden
    wo = s.hidden * s.n_heads * s.head_dim
    ffn = 3 * s.ffn * s.hidden
    weights = s.n_layers * (qkv + wo + ffn) + 2 * s.vocab * s.hidden  # + lm_head and embedding table
    weight_bytes = (weights - s.vocab * s.hidden) * 34 // 32          # the table is gathered, not streamed
    kv_row = s.n_layers * s.n_kv_heads * s.head_dim * 2 * 2           # K and V, fp16
    B = len(positions)
    return weight_bytes + B * (s.hidden // 32) * 34 + sum(p + 1 for p in positions) * kv_row + B * kv_row


@pytest.mark.parametrize("B", [1, 2, 4, 8, 16])
def test_8b_step_bytes(B):
    pos = [1238] * B
    assert bench.step_bytes(synth.LLAMA3_8B, pos) == by_hand(synth.LLAMA3_8B, pos)


def test_8b_weights_and_kv_row():
    s = synth.LLAMA3_8B
    # 7,504,658,432 streamed Q8_0 weights (projections and lm_head) -> 7.974 GB
    assert s.weight_bytes() == 7_504_658_432 * 34 // 32
    assert bench.kv_bytes_per_pos(s) == 131_072


def test_b8_at_1238_positions():
    # weights + 8 embedding rows + 8 x 1239 attended rows + 8 new rows written = 9.274 GB
    # (9.273 GB without the 1 MB of new rows)
    got = bench.step_bytes(synth.LLAMA3_8B, [1238] * 8)
    assert got == 7_973_699_584 + 8 * 4352 + 8 * 1239 * 131_072 + 8 * 131_072 == 9_273_968_640


def test_ragged_positions_count_each_session():
    s = synth.TINY
    pos = [0, 16, 39]
    assert bench.step_bytes(s, pos) == by_hand(s, pos)


def test_q8_0_kv_rows():
    # a Q8_0 head row: 128 quant bytes + 4 fp16 scales = 136 bytes (fp16: 256)
    s = synth.LLAMA3_8B
    assert bench.kv_bytes_per_pos(s, kv_q8=True) == 2 * 32 * 8 * 136 == 69_632
    pos = [25704, 32767]
    want = s.weight_bytes() + 2 * 4352 + (25705 + 32768) * 69_632 + 2 * 69_632
    assert bench.step_bytes(s, pos, kv_q8=True) == want
