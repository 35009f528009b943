"""KV append + ragged GQA split-K flash-decode on the GPU against the CPU oracle.

Workload: the isolated attention configuration -- 32 query heads / 8 KV heads of
128, fp16 KV ~N(0,1), B = 8 sessions whose attended lengths are drawn uniform in
[1, 32768], each appending one new row at its own position first -- plus small
ragged cases (t_kv = 1, a split boundary, just past it) and the tiny model's
64-wide heads."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

# The output is fp16: allow one fp16 ulp of the result plus fp32 noise.
def assert_close_fp16(got16, ref):
    got = got16.astype(np.float64)
    tol = 2.0 ** -10 * np.abs(ref) + 1e-4
    err = np.abs(got - ref)
    assert np.all(err <= tol), float((err / tol).max())


def make_case(seed, B, nh, nkv, hd, lens, n_slots, cap):
    rng = np.random.default_rng(seed)
    slots = rng.permutation(n_slots)[:B].astype(np.int32)
    kc = np.full((n_slots, nkv, cap, hd), np.float16(np.nan), dtype=np.float16)
    vc = np.full_like(kc, np.float16(np.nan))
    for b in range(B):
        n = lens[b] - 1  # history rows; the step appends row n
        sub = synth.substream(seed, "attn-kv", b)
        kc[slots[b], :, :n] = sub.standard_normal((nkv, n, hd), dtype=np.float32).astype(np.float16)
        vc[slots[b], :, :n] = sub.standard_normal((nkv, n, hd), dtype=np.float32).astype(np.float16)
    q = synth.f32_normal(seed, "attn-q", (B, nh, hd))
    kn = synth.f32_normal(seed, "attn-k", (B, nkv, hd))
    vn = synth.f32_normal(seed, "attn-v", (B, nkv, hd))
    return slots, kc, vc, q, kn, vn


def run_gpu(kd, slots, kc, vc, q, kn, vn, pos, nh, nkv, hd, cap, dev_caches=None):
    B = len(slots)
    if dev_caches is None:
        dk = torch.from_numpy(kc.view(np.int16)).cuda()
        dv = torch.from_numpy(vc.view(np.int16)).cuda()
    else:
        dk, dv = dev_caches
    out = torch.empty(B, nh * hd, dtype=torch.int16, device="cuda")
    ws = torch.empty(kd.kd_attn_workspace_bytes(B, nh, hd, cap), dtype=torch.uint8, device="cuda")
    kd.kd_attn_append_decode(torch.from_numpy(q).cuda(), torch.from_numpy(kn).cuda(),
                             torch.from_numpy(vn).cuda(), dk, dv, slots, pos, nh, nkv, hd, kc.shape[0], cap,
                             out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.float16), dk, dv


def oracle_attn(slots, kc, vc, q, kn, vn, pos, nh, nkv):
    B, _, hd = q.shape
    group = nh // nkv
    ref = np.empty((B, nh, hd))
    for b in range(B):
        p = pos[b]
        K = kc[slots[b], :, : p + 1].copy()
        V = vc[slots[b], :, : p + 1].copy()
        K[:, p] = kn[b].astype(np.float16)
        V[:, p] = vn[b].astype(np.float16)
        for h in range(nh):
            ref[b, h] = oracle.attention_head(q[b, h].astype(np.float64), K[h // group].view(np.uint16),
                                              V[h // group].view(np.uint16))
    return ref.reshape(B, nh * hd)


@pytest.mark.parametrize("nh,nkv,hd,lens", [
    (32, 8, 128, [1, 2, 127, 128, 129, 256, 300, 1000]),
    (4, 2, 64, [17, 40]),
    (8, 8, 64, [1, 5, 130]),
    (16, 2, 128, [255, 257, 513]),
])
def test_attention_small_ragged(kdlib, nh, nkv, hd, lens):
    kd = kdlib
    B, cap, n_slots = len(lens), 1024, len(lens) + 3
    slots, kc, vc, q, kn, vn = make_case(5, B, nh, nkv, hd, lens, n_slots, cap)
    pos = np.array(lens, np.int32) - 1
    got, dk, dv = run_gpu(kd, slots, kc, vc, q, kn, vn, pos, nh, nkv, hd, cap)
    ref = oracle_attn(slots, kc, vc, q, kn, vn, pos, nh, nkv)
    assert_close_fp16(got, ref)
    # the appended rows are exactly fp16(k_new), fp16(v_new)
    dk = dk.cpu().numpy().view(np.float16)
    for b in range(B):
        assert np.array_equal(dk[slots[b], :, pos[b]].view(np.uint16), kn[b].astype(np.float16).view(np.uint16))


def test_attention_ragged_long_context_batch_invariant(kdlib):
    kd = kdlib
    nh, nkv, hd, cap, B = 32, 8, 128, 32768, 8
    lens = synth.ragged_lengths(0, "attn-config", B, 1, cap)
    slots, kc, vc, q, kn, vn = make_case(0, B, nh, nkv, hd, lens, B, cap)
    pos = lens - 1
    got, dk, dv = run_gpu(kd, slots, kc, vc, q, kn, vn, pos, nh, nkv, hd, cap)
    ref = oracle_attn(slots, kc, vc, q, kn, vn, pos, nh, nkv)
    assert_close_fp16(got, ref)
    # each session alone (B = 1) gives the same bits as in the batch
    for b in (0, 3, 7):
        one, _, _ = run_gpu(kd, slots[b:b + 1], kc, vc, q[b:b + 1], kn[b:b + 1], vn[b:b + 1], pos[b:b + 1],
                            nh, nkv, hd, cap, dev_caches=(dk, dv))
        assert np.array_equal(one[0].view(np.uint16), got[b].view(np.uint16)), b


def test_attention_single_key_is_value(kdlib):
    # t_kv = 1: the output is the appended value, rounded to fp16
    kd = kdlib
    nh, nkv, hd, cap = 32, 8, 128, 16
    slots, kc, vc, q, kn, vn = make_case(9, 3, nh, nkv, hd, [1, 1, 1], 4, cap)
    pos = np.zeros(3, np.int32)
    got, _, _ = run_gpu(kd, slots, kc, vc, q * 30, kn, vn, pos, nh, nkv, hd, cap)
    want = np.repeat(vn.astype(np.float16), nh // nkv, axis=1).reshape(3, nh * hd)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
