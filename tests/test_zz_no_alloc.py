"""kd_attn_append_decode_noalloc: the KV append + split-K attention call for
callers that cannot allocate device memory where they decode (a pool or arena
that owns the GPU, or a hot path that must not take the implicit device sync of
cudaMalloc/cudaFree).  It keeps its scratch in one fixed device array inside the
library instead of a caller workspace.

Checked through the C ABI against kd_attn_append_decode (same inputs, same
caches) on two calls in a row, the second appending the next row on top of the
first.  This file is collected last; it passes alone in a fresh process (the
first call sets the array up) and after the other tests."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

NH, NKV, HD, CAP, NSLOTS = 32, 8, 128, 512, 5


def close_fp16(a16, b16):
    a = a16.astype(np.float64)
    b = b16.astype(np.float64)
    return np.all(np.abs(a - b) <= 2.0 ** -10 * np.abs(b) + 1e-4)


def test_noalloc_matches_workspace_entry_point_twice(kdlib):
    kd = kdlib
    rng = np.random.default_rng(21)
    slots = np.array([3, 0, 4], np.int32)
    pos = np.array([100, 7, 511 - 2], np.int32)
    B = len(slots)
    base_k = rng.standard_normal((NSLOTS, NKV, CAP, HD), dtype=np.float32).astype(np.float16)
    base_v = rng.standard_normal((NSLOTS, NKV, CAP, HD), dtype=np.float32).astype(np.float16)
    caches = {}
    for name in ("ref", "noalloc"):
        caches[name] = (torch.from_numpy(base_k.view(np.int16)).cuda(), torch.from_numpy(base_v.view(np.int16)).cuda())
    ws = torch.empty(kd.kd_attn_workspace_bytes(B, NH, HD, CAP), dtype=torch.uint8, device="cuda")
    for call in range(2):  # two calls in a row; the second appends the next row
        q = torch.from_numpy(synth.f32_normal(call, "nq", (B, NH, HD))).cuda()
        kn = torch.from_numpy(synth.f32_normal(call, "nk", (B, NKV, HD))).cuda()
        vn = torch.from_numpy(synth.f32_normal(call, "nv", (B, NKV, HD))).cuda()
        p = pos + call
        out_ref = torch.empty(B, NH * HD, dtype=torch.int16, device="cuda")
        out_na = torch.full((B, NH * HD), -1, dtype=torch.int16, device="cuda")
        kd.kd_attn_append_decode(q, kn, vn, *caches["ref"], slots, p, NH, NKV, HD, NSLOTS, CAP, out_ref, ws)
        kd.kd_attn_append_decode_noalloc(q, kn, vn, *caches["noalloc"], slots, p, NH, NKV, HD, NSLOTS, CAP, out_na)
        torch.cuda.synchronize()
        a = out_na.cpu().numpy().view(np.float16)
        r = out_ref.cpu().numpy().view(np.float16)
        assert np.all(np.isfinite(a))
        assert close_fp16(a, r), call
        for i in (0, 1):  # the appended rows are the same in both caches
            assert torch.equal(caches["ref"][i], caches["noalloc"][i]), (call, i)


def test_noalloc_refuses_requests_beyond_its_scratch(kdlib):
    kd = kdlib
    B, cap = 16, 32768  # 16 * 32 * 512 * 132 * 4 + 256 bytes > 16 MiB
    dummy = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(kd.KdError) as e:
        kd.kd_attn_append_decode_noalloc(dummy, dummy, dummy, dummy, dummy, np.arange(B, dtype=np.int32),
                                         np.zeros(B, np.int32), NH, NKV, HD, B, cap, dummy)
    assert e.value.name == "KD_ERR_UNSUPPORTED"
    assert "exceeds the fixed scratch" in str(e.value)
