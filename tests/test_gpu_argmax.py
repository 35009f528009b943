"""The greedy pick on the GPU (kd_argmax, the kernel the step ends with) against
its definition: the largest logit, ties to the lowest index, -0 equal to +0,
NaN never chosen, -1 for a row of NaN only.

Workload: seeded N(0, 1) fp32 rows of the 8B-shaped vocabulary (128256) and of a
small ragged vocabulary (100), B = 1 .. 16, with planted ties, NaNs, infinities
and signed zeros."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def reference(rows):
    out = []
    for r in rows:
        ok = ~np.isnan(r)
        if not ok.any():
            out.append(-1)
            continue
        m = r[ok].max()
        out.append(int(np.flatnonzero(ok & (r == m))[0]))  # -0 == +0 in the comparison
    return np.array(out, np.int32)


def gpu_argmax(kd, rows):
    B, V = rows.shape
    lg = torch.from_numpy(np.ascontiguousarray(rows, np.float32)).cuda()
    out = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(kd.KD_ARGMAX_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    kd.kd_argmax(lg, B, V, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("B,V", [(1, 128256), (8, 128256), (16, 128256), (5, 100), (3, 4)])
def test_argmax_random_rows(kdlib, B, V):
    rows = synth.f32_normal(0, f"argmax-{B}-{V}", (B, V))
    assert np.array_equal(gpu_argmax(kdlib, rows), reference(rows))


def test_argmax_planted_cases(kdlib):
    V = 128256
    rows = synth.f32_normal(1, "argmax-planted", (9, V)) - 10.0
    rows[0, [7, 70000, 128255]] = 5.0            # three-way tie: the lowest index wins
    rows[1, :] = np.nan                          # nothing but NaN
    rows[2, :] = np.nan
    rows[2, 90000] = -np.inf                     # -inf beats NaN
    rows[3, 1234] = np.inf
    rows[3, 50] = np.nan                         # +inf wins, NaN ignored
    rows[4, :] = -1.0
    rows[4, 3000] = -0.0
    rows[4, 2000] = 0.0                          # +0 and -0 tie: the lower index
    rows[5, :] = -np.inf
    rows[5, 128255] = -3.0e38                    # the one finite value wins
    rows[6, 128255] = 1.0e30                     # the last element
    rows[7, 0] = 1.0e30                          # the first element
    rows[8, :] = 0.0                             # all equal: index 0
    got = gpu_argmax(kdlib, rows)
    want = np.array([7, -1, 90000, 1234, 2000, 128255, 128255, 0, 0], np.int32)
    assert np.array_equal(want, reference(rows))
    assert np.array_equal(got, want)
    # the workspace is left ready: a second call on the same rows gives the same picks
    assert np.array_equal(gpu_argmax(kdlib, rows), want)
