"""GPU parity of kv_attn_decode_step (the append of the new token and the decode attention in
one launch) against the CPU oracle (cache_append then decode) and against the two separate
entry points, on ragged lengths with NaN canaries past the valid prefix and in the new slot."""
import zlib

import numpy as np
import pytest

import oracle as O
import workloads as WL
from helpers import assert_bf16_close, assert_bf16_store, assert_fp32_close, bf16_bits, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from kv_cache_gqa_gb300 import build
    build.build_library(verbose=False)
    import kv_cache_gqa_gb300 as K
    return K


def _torch():
    import torch
    return torch


STEP_CASES = [
    # rope kind, sections, norm ("before"/"after"/None), input dtype, G, q_out dtype, shared weights
    ("1d", (), "before", "bf16", 2, "bf16", False),
    ("1d", (), "before", "f32", 4, "f32", True),
    ("sections", (16, 16, 16, 16), "after", "f32", 2, "bf16", False),
    ("2d", (), None, "f32", 1, None, False),
    ("none", (), "before", "bf16", 4, None, False),
    ("1d", (), None, "bf16", 1, "bf16", False),
    ("interleaved", (), "before", "f32", 2, "bf16", False),
    ("interleaved", (), "after", "bf16", 4, "f32", True),
]


@pytest.mark.parametrize("kind,secs,norm,in_dt,G,qo_dt,shared", STEP_CASES)
def test_decode_step_parity(K, kind, secs, norm, in_dt, G, qo_dt, shared):
    torch = _torch()
    rng = np.random.default_rng(zlib.crc32(repr((kind, norm, in_dt, G, qo_dt, shared)).encode()))
    Hkv, D = 2, 128
    Hq = Hkv * G
    lengths = np.array([1, 2, 17, 64, 65, 300, 1000, 4097, 777], np.int32)
    B, W = lengths.size, 4200
    n_axes = {"none": 1, "1d": 1, "sections": 4, "2d": 2, "interleaved": 1}[kind]
    base = 1.11588e7 if kind == "sections" else 1e6
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}[in_dt]
    q = O.store(rng.standard_normal((B, Hq, D)) * 3, in_dt)
    k = O.store(rng.standard_normal((B, Hkv, D)) * 3, in_dt)
    v = O.store(rng.standard_normal((B, Hkv, D)), in_dt)
    pos = rng.integers(0, 40000, size=(B, n_axes)).astype(np.int32)
    wrows = 1 if shared else B
    qw = (1 + 0.1 * rng.standard_normal((wrows, D))).astype(np.float32)
    kw = (1 + 0.1 * rng.standard_normal((wrows, D))).astype(np.float32)
    kc0 = O.store(rng.standard_normal((B, Hkv, W, D)), "bf16")
    vc0 = O.store(rng.standard_normal((B, Hkv, W, D)), "bf16")

    kd = dev(kc0, torch.bfloat16); vd = dev(vc0, torch.bfloat16)
    for b, L in enumerate(lengths):          # canaries past the prefix and in the new token's slot
        kd[b, :, L:] = float("nan"); vd[b, :, L:] = float("inf")
        kd[b, :, L - 1] = float("nan"); vd[b, :, L - 1] = float("nan")
    before_k, before_v = bf16_bits(kd), bf16_bits(vd)
    rope = K.Rope(kind, base, secs)
    norm_kw = dict(q_norm_w=dev(qw) if norm else None, k_norm_w=dev(kw) if norm else None, eps=1e-6,
                   norm_after_rope=(norm == "after"), norm_inst_stride=0 if shared else D)
    ws = torch.zeros(K.decode_workspace_bytes(B, Hkv, Hq, W, D), dtype=torch.uint8, device="cuda")
    q_out = None if qo_dt is None else torch.empty((B, Hq, D), device="cuda",
                                                     dtype={"f32": torch.float32, "bf16": torch.bfloat16}[qo_dt])
    cache = K.KVCache(kd, vd)
    outs = []
    for rep in range(2):                     # the second call rewrites the same slot and reuses the workspace
        out = torch.full((B, Hq, D), float("nan"), device="cuda")
        K.kv_attn_decode_step(dev(q, tdt), dev(k, tdt), dev(v, tdt), dev(pos), cache, dev(lengths), lengths,
                              out, ws, rope, q_out=q_out, **norm_kw)
        torch.cuda.synchronize()
        outs.append(host(out))
        zero = K.lib().kva_decode_workspace_zero_bytes(B, Hkv)
        assert int(ws[:zero].sum()) == 0
    np.testing.assert_array_equal(outs[0], outs[1])
    got = outs[0]
    assert np.all(np.isfinite(got))

    orope = O.Rope(kind, base, secs if secs else None)
    kb, vb = bf16_bits(kd), bf16_bits(vd)
    for b, L in enumerate(lengths):
        L = int(L)
        ck = kc0[b].copy(); cv = vc0[b].copy()
        wq = qw[0 if shared else b] if norm else None
        wk = kw[0 if shared else b] if norm else None
        qr = O.cache_append(q[b][None], k[b][None], v[b][None], pos[b][None], np.array([L - 1]), wq, wk, 1e-6,
                            orope, norm == "after", ck, cv, "bf16")[0]
        kr = O.qk_transform(k[b][None], pos[b][None], wk, 1e-6, orope, norm == "after")[0]
        # the new row: K within one bf16 ulp of the exact transform, V stored exactly
        assert_bf16_store(kb[b][:, L - 1], kr, f"k slot b={b}")
        np.testing.assert_array_equal(vb[b][:, L - 1], WL.f32_to_bf16_bits(O.store(v[b], "bf16").astype(np.float32)))
        # every other slot untouched (canaries included)
        other = np.ones(W, bool); other[L - 1] = False
        np.testing.assert_array_equal(kb[b][:, other], before_k[b][:, other])
        np.testing.assert_array_equal(vb[b][:, other], before_v[b][:, other])
        # attention over the prefix with the new row, q stored in bf16 as the pipeline feeds it
        ck[:, L - 1] = O.store(kr, "bf16")
        ref = O.decode(O.store(qr, "bf16"), ck, cv, L)
        assert_bf16_close(got[b], ref, f"step b={b} L={L}")
        if q_out is not None:
            if qo_dt == "f32":
                assert_fp32_close(host(q_out[b]), qr, "q_out")
            else:
                assert_bf16_store(bf16_bits(q_out[b]), qr, "q_out")


def test_decode_step_matches_append_then_decode(K):
    """The fused step and the two calls it replaces agree on the output and on the cache."""
    torch = _torch()
    rng = np.random.default_rng(4242)
    Hkv, G, D, W = 8, 2, 128, 2048
    Hq = Hkv * G
    lengths = np.array([5, 533, 1024, 2048], np.int32)
    B = lengths.size
    q = torch.from_numpy(rng.standard_normal((B, Hq, D)).astype(np.float32)).cuda().to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((B, Hkv, D)).astype(np.float32)).cuda().to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((B, Hkv, D)).astype(np.float32)).cuda().to(torch.bfloat16)
    pos = dev((lengths - 1).reshape(B, 1).astype(np.int32))
    qw = dev((1 + 0.1 * rng.standard_normal(D)).astype(np.float32))
    kw = dev((1 + 0.1 * rng.standard_normal(D)).astype(np.float32))
    kc = torch.randn((B, Hkv, W, D), device="cuda").to(torch.bfloat16)
    vc = torch.randn((B, Hkv, W, D), device="cuda").to(torch.bfloat16)
    kc2, vc2 = kc.clone(), vc.clone()
    rope = K.Rope("1d", 1e6)
    ws = torch.zeros(K.decode_workspace_bytes(B, Hkv, Hq, W, D), dtype=torch.uint8, device="cuda")
    dl = dev(lengths)

    out_f = torch.empty((B, Hq, D), device="cuda")
    K.kv_attn_decode_step(q, k, v, pos, K.KVCache(kc, vc), dl, lengths, out_f, ws, rope, q_norm_w=qw, k_norm_w=kw)

    slot = (lengths - 1).reshape(B, 1).astype(np.int32)
    q_out = torch.empty((B, 1, Hq, D), device="cuda", dtype=torch.bfloat16)
    K.kv_cache_append_rope_qknorm(q.view(B, 1, Hq, D), k.view(B, 1, Hkv, D), v.view(B, 1, Hkv, D), pos.view(B, 1, 1),
                                  dev(slot), slot, K.KVCache(kc2, vc2), q_out, rope, q_norm_w=qw, k_norm_w=kw)
    out_s = torch.empty((B, Hq, D), device="cuda")
    K.kv_attn_decode(q_out.view(B, Hq, D), K.KVCache(kc2, vc2), dl, lengths, out_s, ws)
    torch.cuda.synchronize()
    assert torch.equal(vc, vc2)
    kd = (kc.float() - kc2.float()).abs().max().item()
    assert kd <= 2 * 2.0 ** -8 * kc2.float().abs().max().item()    # at most an ulp apart
    assert_bf16_close(host(out_f), host(out_s), "fused vs two calls")


SIMT_STEP_CASES = [
    # cache dtype, Dk, Dv, Hkv, G, rope kind, sections, rot_offset, rot_dim, norm, input dtype, q_out dtype
    ("f32", 128, 128, 2, 2, "1d", (), 0, 0, "before", "f32", "f32"),        # the tiny fp32 layer's step
    ("f32", 128, 128, 2, 4, "sections", (16, 16, 16, 16), 0, 0, "after", "bf16", None),
    ("f32", 128, 128, 3, 1, "2d", (), 0, 0, None, "f32", "bf16"),
    ("bf16", 128, 128, 2, 2, "interleaved", (), 64, 64, "before", "f32", "bf16"),   # rotary sub-range
    ("bf16", 192, 128, 4, 1, "interleaved", (), 128, 64, None, "bf16", "bf16"),     # the MLA-expanded cache
    ("f32", 192, 128, 2, 2, "1d", (), 128, 64, "after", "f32", "f32"),
    ("bf16", 192, 128, 2, 4, "1d", (), 0, 0, "before", "f32", None),
]


@pytest.mark.parametrize("c_dt,Dk,Dv,Hkv,G,kind,secs,ro,rw,norm,in_dt,qo_dt", SIMT_STEP_CASES)
def test_decode_step_cuda_core_form(K, c_dt, Dk, Dv, Hkv, G, kind, secs, ro, rw, norm, in_dt, qo_dt):
    """The fused step on the CUDA-core kernel (fp32 caches, the K 192 / V 128 cache, RoPE over a
    sub-range of the head) against the oracle's append followed by its decode, with NaN canaries
    past the valid prefix and in the new token's slot."""
    torch = _torch()
    rng = np.random.default_rng(zlib.crc32(repr((c_dt, Dk, Hkv, G, kind, ro, norm, in_dt)).encode()))
    Hq = Hkv * G
    lengths = np.array([1, 2, 33, 64, 65, 300, 1000, 1500], np.int32)
    B, W = lengths.size, 1536
    n_axes = {"none": 1, "1d": 1, "sections": 4, "2d": 2, "interleaved": 1}[kind]
    base = 1.11588e7 if kind == "sections" else 1e6
    cdt = {"f32": torch.float32, "bf16": torch.bfloat16}[c_dt]
    idt = {"f32": torch.float32, "bf16": torch.bfloat16}[in_dt]
    q = O.store(rng.standard_normal((B, Hq, Dk)) * 3, in_dt)
    k = O.store(rng.standard_normal((B, Hkv, Dk)) * 3, in_dt)
    v = O.store(rng.standard_normal((B, Hkv, Dv)), in_dt)
    pos = rng.integers(0, 40000, size=(B, n_axes)).astype(np.int32)
    qw = (1 + 0.1 * rng.standard_normal((B, Dk))).astype(np.float32)
    kw = (1 + 0.1 * rng.standard_normal((B, Dk))).astype(np.float32)
    kc0 = O.store(rng.standard_normal((B, Hkv, W, Dk)), c_dt)
    vc0 = O.store(rng.standard_normal((B, Hkv, W, Dv)), c_dt)
    kd = dev(kc0, cdt); vd = dev(vc0, cdt)
    for b, L in enumerate(lengths):
        kd[b, :, L:] = float("nan"); vd[b, :, L:] = float("inf")
        kd[b, :, L - 1] = float("nan"); vd[b, :, L - 1] = float("nan")
    rope = K.Rope(kind, base, secs, rot_offset=ro, rot_dim=rw)
    ws = torch.zeros(K.decode_workspace_bytes(B, Hkv, Hq, W, Dv), dtype=torch.uint8, device="cuda")
    q_out = None if qo_dt is None else torch.empty((B, Hq, Dk), device="cuda",
                                                     dtype={"f32": torch.float32, "bf16": torch.bfloat16}[qo_dt])
    cache = K.KVCache(kd, vd)
    outs = []
    for rep in range(2):                     # the second call rewrites the same slot and reuses the workspace
        out = torch.full((B, Hq, Dv), float("nan"), device="cuda")
        K.kv_attn_decode_step(dev(q, idt), dev(k, idt), dev(v, idt), dev(pos), cache, dev(lengths), lengths, out, ws,
                              rope, q_norm_w=dev(qw) if norm else None, k_norm_w=dev(kw) if norm else None, eps=1e-6,
                              norm_after_rope=(norm == "after"), norm_inst_stride=Dk, q_out=q_out)
        torch.cuda.synchronize()
        outs.append(host(out))
    np.testing.assert_array_equal(outs[0], outs[1])
    got = outs[0]
    assert np.all(np.isfinite(got))
    orope = O.Rope(kind, base, secs if secs else None, rot_offset=ro, rot_dim=rw if rw else None)
    kh, vh = host(kd), host(vd)
    for b, L in enumerate(lengths):
        L = int(L)
        ck = kc0[b].copy(); cv = vc0[b].copy()
        wq = qw[b] if norm else None
        wk = kw[b] if norm else None
        qr = O.cache_append(q[b][None], k[b][None], v[b][None], pos[b][None], np.array([L - 1]), wq, wk, 1e-6,
                            orope, norm == "after", ck, cv, c_dt)[0]
        kr = O.qk_transform(k[b][None], pos[b][None], wk, 1e-6, orope, norm == "after")[0]
        if c_dt == "bf16":
            assert_bf16_store(bf16_bits(kd[b])[:, L - 1], kr, f"k slot b={b}")
        else:
            assert_fp32_close(kh[b][:, L - 1], kr, f"k slot b={b}")
        np.testing.assert_array_equal(vh[b][:, L - 1], cv[:, L - 1])          # v stored exactly
        other = np.ones(W, bool); other[L - 1] = False
        assert not np.any(np.isfinite(kh[b][:, L:])) and not np.any(np.isfinite(vh[b][:, L:]))   # canaries kept
        # attention over the prefix with the row the kernel wrote; the query is the exact transform
        ck[:, L - 1] = kh[b][:, L - 1]
        ref = O.decode(qr, ck, cv, L)
        if c_dt == "f32":
            assert_fp32_close(got[b], ref, f"step b={b} L={L}")
        else:
            assert_bf16_close(got[b], ref, f"step b={b} L={L}")
        if q_out is not None:
            if qo_dt == "f32":
                assert_fp32_close(host(q_out[b]), qr, "q_out")
            else:
                assert_bf16_store(bf16_bits(q_out[b]), qr, "q_out")


def test_prepared_call_matches_direct_call_and_follows_updated_lengths(K):
    """A PreparedCall marshals the arguments once; calling it again after the lengths (device
    array and host mirror) are updated in place runs the next step, as a direct call would."""
    torch = _torch()
    rng = np.random.default_rng(77)
    B, Hkv, G, D, W = 3, 2, 2, 128, 600
    Hq = Hkv * G
    kc = torch.randn((B, Hkv, W, D), device="cuda").to(torch.bfloat16); vc = torch.randn_like(kc)
    kc2, vc2 = kc.clone(), vc.clone()
    q = dev(rng.standard_normal((B, Hq, D)).astype(np.float32))
    k = dev(rng.standard_normal((B, Hkv, D)).astype(np.float32))
    v = dev(rng.standard_normal((B, Hkv, D)).astype(np.float32))
    pos = dev(np.array([[100], [200], [300]], np.int32))
    rope = K.Rope("1d", 1e6)
    ws = torch.zeros(K.decode_workspace_bytes(B, Hkv, Hq, W, D), dtype=torch.uint8, device="cuda")
    ws2 = torch.zeros_like(ws)
    lh = np.array([10, 300, 555], np.int32)
    ld = dev(lh)
    out_p = torch.empty((B, Hq, D), device="cuda")
    call = K.prepare_decode_step(q, k, v, pos, K.KVCache(kc, vc), ld, lh, out_p, ws, rope)
    for step in range(2):
        call()
        out_d = torch.empty((B, Hq, D), device="cuda")
        K.kv_attn_decode_step(q, k, v, pos, K.KVCache(kc2, vc2), ld, lh, out_d, ws2, rope)
        torch.cuda.synchronize()
        assert torch.equal(out_p, out_d) and torch.equal(kc, kc2) and torch.equal(vc, vc2), step
        lh += 1                                    # the next step: both mirrors advance in place
        ld += 1
