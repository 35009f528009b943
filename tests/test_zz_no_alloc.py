"""kd_attn_append_decode_noalloc: the KV append + split-K attention call for
callers that cannot allocate device memory where they decode (a pool or arena
that owns the GPU, or a hot path that must not take the implicit device sync of
cudaMalloc/cudaFree).  It keeps its scratch in one fixed device array inside the
library instead of a caller workspace.

Checked through the C ABI against kd_attn_append_decode (same inputs, same
caches, same kernels): outputs and appended rows bit for bit, on two calls in a
row (the second appending the next row on top of the first), then on a third
call with a smaller capacity, whose partial-result layout differs from what the
shared array still holds; the first call is also compared with the oracle.  This
file is collected last; it passes alone in a fresh process (the first call sets
the array up) and after the other tests."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

NH, NKV, HD, CAP, NSLOTS = 32, 8, 128, 512, 5


def fp16_close(a16, b64):
    """Within one fp16 ulp of the exact result plus 1e-4 (the attention tests' bound)."""
    a = a16.astype(np.float64)
    return np.all(np.abs(a - b64) <= 2.0 ** -10 * np.abs(b64) + 1e-4)


def caches_for(base_k, base_v):
    return (torch.from_numpy(base_k.view(np.int16)).cuda(), torch.from_numpy(base_v.view(np.int16)).cuda())


def both_calls(kd, q, kn, vn, ref_caches, na_caches, slots, p, cap, nslots, ws):
    B = len(slots)
    out_ref = torch.empty(B, NH * HD, dtype=torch.int16, device="cuda")
    out_na = torch.full((B, NH * HD), -1, dtype=torch.int16, device="cuda")
    kd.kd_attn_append_decode(q, kn, vn, *ref_caches, slots, p, NH, NKV, HD, nslots, cap, out_ref, ws)
    kd.kd_attn_append_decode_noalloc(q, kn, vn, *na_caches, slots, p, NH, NKV, HD, nslots, cap, out_na)
    torch.cuda.synchronize()
    return out_ref, out_na


def test_noalloc_matches_workspace_entry_point_twice(kdlib):
    kd = kdlib
    rng = np.random.default_rng(21)
    slots = np.array([3, 0, 4], np.int32)
    pos = np.array([100, 7, 511 - 2], np.int32)
    B = len(slots)
    base_k = rng.standard_normal((NSLOTS, NKV, CAP, HD), dtype=np.float32).astype(np.float16)
    base_v = rng.standard_normal((NSLOTS, NKV, CAP, HD), dtype=np.float32).astype(np.float16)
    ref_c, na_c = caches_for(base_k, base_v), caches_for(base_k, base_v)
    ws = torch.empty(kd.kd_attn_workspace_bytes(B, NH, HD, CAP), dtype=torch.uint8, device="cuda")
    for call in range(2):  # two calls in a row; the second appends the next row
        q = torch.from_numpy(synth.f32_normal(call, "nq", (B, NH, HD))).cuda()
        kn = torch.from_numpy(synth.f32_normal(call, "nk", (B, NKV, HD))).cuda()
        vn = torch.from_numpy(synth.f32_normal(call, "nv", (B, NKV, HD))).cuda()
        p = pos + call
        out_ref, out_na = both_calls(kd, q, kn, vn, ref_c, na_c, slots, p, CAP, NSLOTS, ws)
        assert torch.equal(out_na, out_ref), call  # same kernels, same inputs: the same bits
        for i in (0, 1):  # the appended rows are the same in both caches
            assert torch.equal(ref_c[i], na_c[i]), (call, i)
        if call == 0:  # and both agree with the oracle on the first call
            got = out_na.cpu().numpy().view(np.float16).reshape(B, NH, HD)
            kc = ref_c[0].cpu().numpy().view(np.uint16)
            vc = ref_c[1].cpu().numpy().view(np.uint16)
            qh = q.cpu().numpy().astype(np.float64)
            for b in range(B):
                for h in range(NH):
                    g = h // (NH // NKV)
                    want = oracle.attention_head(qh[b, h], kc[slots[b], g, :p[b] + 1], vc[slots[b], g, :p[b] + 1])
                    assert fp16_close(got[b, h], want), (b, h)
    assert kd.kd_attn_device_status(None) == 0  # the allocation-free call's fault word
    assert kd.kd_attn_device_status(ws) == 0


def test_noalloc_smaller_capacity_after_larger(kdlib):
    """A call whose capacity (and so its split-record stride in the shared array)
    is smaller than the previous call's: what the array still holds is ignored."""
    kd = kdlib
    rng = np.random.default_rng(22)
    cap, nslots = 128, 2
    slots = np.array([1, 0], np.int32)
    pos = np.array([127, 64], np.int32)
    B = len(slots)
    base_k = rng.standard_normal((nslots, NKV, cap, HD), dtype=np.float32).astype(np.float16)
    base_v = rng.standard_normal((nslots, NKV, cap, HD), dtype=np.float32).astype(np.float16)
    ref_c, na_c = caches_for(base_k, base_v), caches_for(base_k, base_v)
    ws = torch.empty(kd.kd_attn_workspace_bytes(B, NH, HD, cap), dtype=torch.uint8, device="cuda")
    q = torch.from_numpy(synth.f32_normal(5, "nq", (B, NH, HD))).cuda()
    kn = torch.from_numpy(synth.f32_normal(5, "nk", (B, NKV, HD))).cuda()
    vn = torch.from_numpy(synth.f32_normal(5, "nv", (B, NKV, HD))).cuda()
    out_ref, out_na = both_calls(kd, q, kn, vn, ref_c, na_c, slots, pos, cap, nslots, ws)
    assert torch.equal(out_na, out_ref)
    for i in (0, 1):
        assert torch.equal(ref_c[i], na_c[i]), i


def test_noalloc_refuses_requests_beyond_its_scratch(kdlib):
    kd = kdlib
    B, cap = 16, 32768  # 16 * 32 * 512 * 132 * 4 + 256 bytes > 16 MiB
    dummy = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(kd.KdError) as e:
        kd.kd_attn_append_decode_noalloc(dummy, dummy, dummy, dummy, dummy, np.arange(B, dtype=np.int32),
                                         np.zeros(B, np.int32), NH, NKV, HD, B, cap, dummy)
    assert e.value.name == "KD_ERR_UNSUPPORTED"
    assert "exceeds the fixed scratch" in str(e.value)
