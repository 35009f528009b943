"""Q8_0 mmvq on the GPU against the CPU oracle and against itself across m.

Workload: the isolated-mmvq configuration (4096x4096 and 14336x4096 Q8_0 weights
times fp16 activations ~N(0,1) at m = 1, 2, 4, 8, 16), the step's interleaved
gate|up shape (28672x4096), plus small shapes that span several row groups and
k-groups with ragged m."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

# fp32 accumulation of at most K/32 + 32 rounded adds (block sums in the tensor
# core, then scaled block sums), unit roundoff 2^-24, with margin for truncating
# tensor-core accumulation: |err| <= 2^-14 * sum_i |w_i x_i| per output.
REL_BOUND = 2.0 ** -14


def dequant(m):
    d, qs = synth.q8_0_split(m)
    return (qs.astype(np.float32) * d.astype(np.float32)[:, :, None]).reshape(m.shape[0], -1)


def run(kd, h, x16, rows):
    m = x16.shape[0]
    x = torch.from_numpy(x16.view(np.int16)).cuda()
    y = torch.full((m, rows), float("nan"), device="cuda", dtype=torch.float32)
    kd.kd_mmvq(h, x, m, y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def check_vs_oracle(W, x16, y):
    xf = x16.view(np.float16).astype(np.float64)
    absum = np.abs(dequant(W)).astype(np.float64) @ np.abs(xf).T  # [rows][m]
    for r in range(x16.shape[0]):
        ref = oracle.matvec_q8_0(W, xf[r])
        err = np.abs(y[r] - ref)
        bound = REL_BOUND * absum[:, r] + 1e-30
        assert np.all(err <= bound), (r, float((err / bound).max()))


# 28672 x 4096 (the interleaved gate|up shape, 896 row groups): at m <= 8 two CTAs
# per SM walking several groups each, at m = 16 one CTA per SM.
@pytest.mark.parametrize("rows,cols", [(4096, 4096), (14336, 4096), (28672, 4096)])
def test_mmvq_config_shapes_row_identity_and_oracle(kdlib, rows, cols):
    kd = kdlib
    W = synth.q8_0_matrix(0, f"mmvq-{rows}x{cols}", rows, cols)
    x16 = synth.activations_fp16(0, f"mmvq-{cols}", 16, cols)
    h = kd.kd_q8_matrix_create(W)
    try:
        y16 = run(kd, h, x16, rows)
        assert np.all(np.isfinite(y16))
        for m in (1, 2, 4, 8, 16):
            ym = run(kd, h, x16[:m], rows)
            assert np.array_equal(ym.view(np.uint32), y16[:m].view(np.uint32)), m
        for r in range(16):  # every row alone, m = 1
            y1 = run(kd, h, np.ascontiguousarray(x16[r:r + 1]), rows)
            assert np.array_equal(y1[0].view(np.uint32), y16[r].view(np.uint32)), r
        check_vs_oracle(W, x16, y16)
    finally:
        kd.kd_q8_matrix_free(h)


# 6144 x 4096 (the fused q|k|v shape): more row groups than SMs, at most twice as
# many -- one CTA per group, two per SM, for m <= 8; the 16-column kernel above.
@pytest.mark.parametrize("rows,cols", [(32, 128), (96, 384), (160, 1152), (4096, 14336), (6144, 4096)])
def test_mmvq_small_and_ragged(kdlib, rows, cols):
    kd = kdlib
    W = synth.q8_0_matrix(1, f"mmvq-s-{rows}x{cols}", rows, cols)
    x16 = synth.activations_fp16(1, f"mmvq-s-{cols}", 16, cols)
    h = kd.kd_q8_matrix_create(W)
    try:
        y16 = run(kd, h, x16, rows)
        for m in (1, 3, 8, 9, 13):
            ym = run(kd, h, x16[:m], rows)
            assert np.array_equal(ym.view(np.uint32), y16[:m].view(np.uint32)), m
        check_vs_oracle(W, x16, y16)
    finally:
        kd.kd_q8_matrix_free(h)


def test_mmvq_extreme_blocks(kdlib):
    # +-127 quants, subnormal and large scales, zero activations in some columns
    kd = kdlib
    rows, cols = 64, 256
    rng = np.random.default_rng(3)
    qs = rng.choice(np.array([-127, 127, 0, 1, -1], np.int8), size=(rows, cols // 32, 32))
    d = rng.choice(np.array([2 ** -24, 1023 * 2 ** -24, 2 ** -14, 0.5, 3.0], np.float64),
                   size=(rows, cols // 32)).astype(np.float16)
    W = synth.q8_0_from_parts(d, qs)
    x16 = synth.activations_fp16(2, "mmvq-x", 5, cols)
    x16[1] = 0
    h = kd.kd_q8_matrix_create(W)
    try:
        y = run(kd, h, x16, rows)
        assert np.all(y[1] == 0.0)
        check_vs_oracle(W, x16, y)
    finally:
        kd.kd_q8_matrix_free(h)
