"""GPU parity of each C-ABI entry point against the CPU oracle on seeded inputs: small and
ragged shapes that still span several tiles, every mask / RoPE / dtype variant, and the edge
cases (empty, single key, untouched slots, NaN canaries past the valid prefix, repeated calls
sharing a workspace)."""
import zlib

import numpy as np
import pytest

import oracle as O
import workloads as WL
from helpers import (ARGMAX_MARGIN, assert_bf16_close, assert_bf16_store, assert_fp32_close, bf16_bits,
                     dev, host, row_rel_err)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from kv_cache_gqa_gb300 import build
    build.build_library(verbose=False)
    import kv_cache_gqa_gb300 as K
    return K


def T():
    import torch
    return torch


def _tdt(name):
    return {"f32": T().float32, "bf16": T().bfloat16}[name]


def _widen(x, dt):
    """Values the kernel sees after the input is stored in dtype dt."""
    return O.store(x, dt)


# ----------------------------------------------------------------------------
# (a) append
# ----------------------------------------------------------------------------
APPEND_CASES = [
    # D, rope kind, sections, norm ("before"/"after"/None), in, q_out, cache
    (128, "1d", (), "before", "f32", "f32", "f32"),
    (128, "1d", (), "before", "f32", "bf16", "bf16"),
    (128, "sections", (16, 16, 16, 16), "after", "f32", "bf16", "bf16"),
    (128, "sections", (16, 16, 16, 16), "after", "f32", "f32", "f32"),
    (128, "none", (), "before", "bf16", "f32", "bf16"),
    (72, "2d", (), None, "f32", "f32", "f32"),
    (72, "2d", (), None, "f32", "bf16", "bf16"),
    (64, "1d", (), "after", "bf16", "bf16", "f32"),
    (72, "1d", (), "before", "f32", "f32", "f32"),
    (128, "interleaved", (), "before", "f32", "bf16", "bf16"),
    (128, "interleaved", (), "after", "bf16", "f32", "f32"),
    (64, "interleaved", (), None, "f32", "f32", "bf16"),
]


@pytest.mark.parametrize("D,kind,secs,norm,in_dt,qo_dt,c_dt", APPEND_CASES)
def test_append_parity(K, D, kind, secs, norm, in_dt, qo_dt, c_dt):
    torch = T()
    rng = np.random.default_rng(zlib.crc32(repr((D, kind, norm, in_dt, qo_dt, c_dt)).encode()))
    N, Tt, Hkv, G, W = 3, 5, 4, 2, 16
    Hq = Hkv * G
    q = rng.standard_normal((N, Tt, Hq, D)).astype(np.float32) * 3
    k = rng.standard_normal((N, Tt, Hkv, D)).astype(np.float32) * 3
    v = rng.standard_normal((N, Tt, Hkv, D)).astype(np.float32)
    n_axes = {"none": 1, "1d": 1, "sections": 4, "2d": 2, "interleaved": 1}[kind]
    pos = rng.integers(0, 40000, size=(N, Tt, n_axes)).astype(np.int32)
    slot = np.stack([rng.permutation(W)[:Tt] for _ in range(N)]).astype(np.int32)
    qw = (1 + 0.1 * rng.standard_normal((N, D))).astype(np.float32)
    kw = (1 + 0.1 * rng.standard_normal((N, D))).astype(np.float32)
    base = 1.11588e7 if kind == "sections" else 1e6

    qd, kd, vd = dev(q, _tdt(in_dt)), dev(k, _tdt(in_dt)), dev(v, _tdt(in_dt))
    kc = torch.full((N, Hkv, W, D), 7.0, device="cuda", dtype=_tdt(c_dt))
    vc = torch.full_like(kc, 7.0)
    q_out = torch.empty((N, Tt, Hq, D), device="cuda", dtype=_tdt(qo_dt))
    cache = K.KVCache(kc, vc)
    K.kv_cache_append_rope_qknorm(
        qd, kd, vd, dev(pos), dev(slot), slot, cache, q_out, K.Rope(kind, base, secs),
        q_norm_w=dev(qw) if norm else None, k_norm_w=dev(kw) if norm else None, eps=1e-6,
        norm_after_rope=(norm == "after"), norm_inst_stride=D)
    torch.cuda.synchronize()

    rope = O.Rope(kind, base, secs if secs else None)
    kc_h, vc_h = host(kc), host(vc)
    for n in range(N):
        qx, kx, vx = (_widen(a[n], in_dt) for a in (q, k, v))
        ck = np.full((Hkv, W, D), 7.0); cv = np.full((Hkv, W, D), 7.0)
        qr = O.cache_append(qx, kx, vx, pos[n], slot[n], qw[n] if norm else None,
                            kw[n] if norm else None, 1e-6, rope, norm == "after", ck, cv, c_dt)
        kr = O.qk_transform(kx, pos[n], kw[n] if norm else None, 1e-6, rope, norm == "after")
        if qo_dt == "f32":
            assert_fp32_close(host(q_out[n]), qr, "q_out")
        else:
            assert_bf16_store(bf16_bits(q_out[n]), qr, "q_out")
        written = np.zeros(W, bool); written[slot[n]] = True
        if c_dt == "f32":
            assert_fp32_close(kc_h[n][:, written], ck[:, written], "k cache")
        else:
            assert_bf16_store(bf16_bits(kc[n])[:, slot[n]], kr.transpose(1, 0, 2), "k cache")
        np.testing.assert_array_equal(vc_h[n][:, written], cv[:, written])      # v stored exactly
        assert np.all(kc_h[n][:, ~written] == 7.0) and np.all(vc_h[n][:, ~written] == 7.0)


STREAM_CASES = [
    # D, rope kind, sections, norm, in, q_out, cache: long appends (>= 2 work items per SM) with a
    # ragged last token block take the streaming (bulk-copy ring) form of the append kernel
    (128, "1d", (), "before", "f32", "bf16", "bf16"),
    (128, "sections", (16, 16, 16, 16), "after", "f32", "f32", "f32"),
    (128, "2d", (), None, "bf16", "bf16", "bf16"),
    (64, "1d", (), "before", "f32", "bf16", "f32"),
    (256, "1d", (), "after", "f32", "bf16", "bf16"),
    (128, "interleaved", (), "before", "f32", "bf16", "bf16"),
    (64, "interleaved", (), "after", "f32", "f32", "f32"),
]


@pytest.mark.parametrize("D,kind,secs,norm,in_dt,qo_dt,c_dt", STREAM_CASES)
def test_append_stream_parity(K, D, kind, secs, norm, in_dt, qo_dt, c_dt):
    torch = T()
    rng = np.random.default_rng(zlib.crc32(repr(("stream", D, kind, norm, in_dt)).encode()))
    N, Tt, Hkv, G = 40, 77, 4, 2
    Hq, W = Hkv * G, 96
    q = rng.standard_normal((N, Tt, Hq, D)).astype(np.float32) * 3
    k = rng.standard_normal((N, Tt, Hkv, D)).astype(np.float32) * 3
    v = rng.standard_normal((N, Tt, Hkv, D)).astype(np.float32)
    n_axes = {"none": 1, "1d": 1, "sections": 4, "2d": 2, "interleaved": 1}[kind]
    pos = rng.integers(0, 40000, size=(N, Tt, n_axes)).astype(np.int32)
    slot = np.stack([rng.permutation(W)[:Tt] for _ in range(N)]).astype(np.int32)
    qw = (1 + 0.1 * rng.standard_normal((N, D))).astype(np.float32)
    kw = (1 + 0.1 * rng.standard_normal((N, D))).astype(np.float32)
    base = 1.11588e7 if kind == "sections" else 1e6
    kc = torch.full((N, Hkv, W, D), 7.0, device="cuda", dtype=_tdt(c_dt))
    vc = torch.full_like(kc, 7.0)
    q_out = torch.empty((N, Tt, Hq, D), device="cuda", dtype=_tdt(qo_dt))
    K.kv_cache_append_rope_qknorm(
        dev(q, _tdt(in_dt)), dev(k, _tdt(in_dt)), dev(v, _tdt(in_dt)), dev(pos), dev(slot), slot, K.KVCache(kc, vc),
        q_out, K.Rope(kind, base, secs), q_norm_w=dev(qw) if norm else None, k_norm_w=dev(kw) if norm else None,
        eps=1e-6, norm_after_rope=(norm == "after"), norm_inst_stride=D)
    torch.cuda.synchronize()
    rope = O.Rope(kind, base, secs if secs else None)
    kc_h, vc_h = host(kc), host(vc)
    kb = bf16_bits(kc) if c_dt == "bf16" else None
    for n in range(0, N, 3):
        qx, kx, vx = (_widen(a[n], in_dt) for a in (q, k, v))
        ck = np.full((Hkv, W, D), 7.0); cv = np.full((Hkv, W, D), 7.0)
        qr = O.cache_append(qx, kx, vx, pos[n], slot[n], qw[n] if norm else None, kw[n] if norm else None, 1e-6,
                            rope, norm == "after", ck, cv, c_dt)
        kr = O.qk_transform(kx, pos[n], kw[n] if norm else None, 1e-6, rope, norm == "after")
        if qo_dt == "f32":
            assert_fp32_close(host(q_out[n]), qr, f"q_out n={n}")
        else:
            assert_bf16_store(bf16_bits(q_out[n]), qr, f"q_out n={n}")
        written = np.zeros(W, bool); written[slot[n]] = True
        if c_dt == "f32":
            assert_fp32_close(kc_h[n][:, written], ck[:, written], f"k cache n={n}")
        else:
            assert_bf16_store(kb[n][:, slot[n]], kr.transpose(1, 0, 2), f"k cache n={n}")
        np.testing.assert_array_equal(vc_h[n][:, written], cv[:, written])
        assert np.all(kc_h[n][:, ~written] == 7.0) and np.all(vc_h[n][:, ~written] == 7.0)


def test_append_shared_positions_and_weights(K):
    """Instance strides of 0 share positions/slots/weights across instances (layers)."""
    torch = T()
    rng = np.random.default_rng(5)
    N, Tt, Hkv, Hq, D, W = 4, 3, 8, 16, 128, 8
    q = rng.standard_normal((N, Tt, Hq, D)).astype(np.float32)
    k = rng.standard_normal((N, Tt, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((N, Tt, Hkv, D)).astype(np.float32)
    pos = np.array([[[3], [9], [4000]]], np.int32)
    slot = np.array([[5, 0, 7]], np.int32)
    qw = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    kw = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    kc = torch.zeros((N, Hkv, W, D), device="cuda"); vc = torch.zeros_like(kc)
    q_out = torch.empty((N, Tt, Hq, D), device="cuda")
    K.kv_cache_append_rope_qknorm(dev(q), dev(k), dev(v), dev(pos), dev(slot), slot, K.KVCache(kc, vc), q_out,
                                  K.Rope("1d", 1e6), q_norm_w=dev(qw), k_norm_w=dev(kw))
    torch.cuda.synchronize()
    for n in range(N):
        ck = np.zeros((Hkv, W, D)); cv = np.zeros((Hkv, W, D))
        qr = O.cache_append(q[n], k[n], v[n], pos[0], slot[0], qw, kw, 1e-6, O.Rope("1d", 1e6), False,
                            ck, cv, "f32")
        assert_fp32_close(host(q_out[n]), qr, "q_out")
        assert_fp32_close(host(kc[n])[:, slot[0]], ck[:, slot[0]], "k")


# ----------------------------------------------------------------------------
# (b) prefill
# ----------------------------------------------------------------------------
def _prefill_case(K, D, S, mask, dt, G, seed, N=2, Hkv=2, W=None, perm=False):
    torch = T()
    rng = np.random.default_rng(seed)
    W = W or S + 3
    Hq = Hkv * G
    q = rng.standard_normal((N, S, Hq, D))
    kc = rng.standard_normal((N, Hkv, W, D))
    vc = rng.standard_normal((N, Hkv, W, D))
    q, kc, vc = (O.store(a, dt) for a in (q, kc, vc))   # what the kernel reads
    seg = None
    if mask == "segment":
        cuts = np.sort(rng.choice(np.arange(1, S), size=min(S - 1, 4), replace=False)) if S > 1 else []
        seg = np.zeros(S, np.int32)
        for c in cuts:
            seg[c:] += 1
    row_of_slot = rng.permutation(S).astype(np.int32) if perm else None
    tdt = _tdt(dt)
    out = torch.full((N, S, Hq, D), float("nan"), device="cuda")
    K.kv_attn_prefill(dev(q, tdt), K.KVCache(dev(kc, tdt), dev(vc, tdt)), out, mask=mask,
                      segment=dev(seg) if seg is not None else None, segment_host=seg,
                      row_of_slot=dev(row_of_slot) if perm else None)
    torch.cuda.synchronize()
    got = host(out)
    for n in range(N):
        q_slots = q[n][row_of_slot] if perm else q[n]
        ref = O.prefill(q_slots, kc[n], vc[n], S, mask, seg)
        g = got[n][row_of_slot] if perm else got[n]
        if dt == "f32":
            assert_fp32_close(g, ref, f"prefill D={D} S={S} {mask}")
        else:
            assert_bf16_close(g, ref, f"prefill D={D} S={S} {mask}")


@pytest.mark.parametrize("S", [1, 2, 3, 63, 64, 65, 127, 129, 200])
@pytest.mark.parametrize("mask", ["causal", "full", "segment"])
def test_prefill_f32_ragged(K, S, mask):
    _prefill_case(K, 128, S, mask, "f32", 2, seed=S * 7 + len(mask))


@pytest.mark.parametrize("mask", ["causal", "segment"])
def test_prefill_f32_wide_grid(K, mask):
    """Enough (instance, head, row tile) work that the fp32 kernel keeps 64-row CTAs (the small
    cases above run 48-row CTAs, which spread a one-wave grid more evenly): 16 instances x 16
    heads x 256 tokens."""
    _prefill_case(K, 128, 256, mask, "f32", 2, seed=256 + len(mask), N=16, Hkv=8)


@pytest.mark.parametrize("S", [1, 5, 64, 127, 128, 129, 255, 300])
@pytest.mark.parametrize("mask", ["causal", "full", "segment"])
def test_prefill_bf16_ragged(K, S, mask):
    _prefill_case(K, 128, S, mask, "bf16", 2, seed=S * 11 + len(mask))


@pytest.mark.parametrize("mask", ["causal", "full", "segment"])
@pytest.mark.parametrize("G", [1, 2])
def test_prefill_bf16_many_instances(K, mask, G):
    """Enough instances that the tensor-core prefill pairs two query tiles per work unit (the
    small cases above give one tile per unit): the heads of a GQA pair, or row tiles t and
    n-1-t of one head."""
    _prefill_case(K, 128, 300, mask, "bf16", G, seed=500 + G + len(mask), N=48, Hkv=2)


@pytest.mark.parametrize("G", [1, 2])
def test_prefill_bf16_two_rounds_last_quarter_full(K, G):
    """Full-mask paired work units in two rounds over the SMs, the second filling about a
    quarter of them (N chosen from the GPU's SM count); 3 row tiles, so for G = 1 (row tiles
    t and n-1-t of one head) one unit per head holds a single tile."""
    mask = "full"
    torch = T()
    P = torch.cuda.get_device_properties(0).multi_processor_count
    nq, pairs = 3, 2                               # S = 300: 3 row tiles; 2 heads or 2 head pairs
    per_inst = pairs * (nq if G == 2 else (nq + 1) // 2)
    N = (P + P // 4) // per_inst + 1
    units = per_inst * N
    assert units > P and 2 * (units - P) <= P
    _prefill_case(K, 128, 300, mask, "bf16", G, seed=700 + G + len(mask), N=N, Hkv=2)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("mask", ["full", "segment"])
def test_prefill_d72_mha_permuted(K, dt, mask):
    _prefill_case(K, 72, 150, mask, dt, 1, seed=99, Hkv=3, perm=True)


@pytest.mark.parametrize("dt,N", [("bf16", 2), ("f32", 2), ("bf16", 48)])
@pytest.mark.parametrize("layout", ["image", "spans"])
def test_prefill_causal_segment(K, dt, N, layout):
    """Causal mask with image spans fully visible to their own rows (N = 48: paired tiles)."""
    torch = T()
    rng = np.random.default_rng(zlib.crc32(repr(("cseg", dt, layout)).encode()))
    if layout == "image":
        seg = WL.image_span_segments(20, 16, 16, 218)          # the 512-row image-span prompt
    else:                                                     # several spans, ragged tail
        seg = np.arange(300, dtype=np.int32)
        for s0, s1 in ((5, 40), (120, 130), (131, 256), (290, 300)):
            seg[s0:s1] = s0
    S, Hkv, Hq, D = seg.size, 2, 4, 128
    q = O.store(rng.standard_normal((N, S, Hq, D)), dt)
    kc = O.store(rng.standard_normal((N, Hkv, S + 8, D)), dt)
    vc = O.store(rng.standard_normal((N, Hkv, S + 8, D)), dt)
    out = T().empty((N, S, Hq, D), device="cuda")
    tdt = _tdt(dt)
    K.kv_attn_prefill(dev(q, tdt), K.KVCache(dev(kc, tdt), dev(vc, tdt)), out, mask="causal_segment",
                      segment=dev(seg), segment_host=seg)
    torch.cuda.synchronize()
    got = host(out)
    for n in range(N):
        ref = O.prefill(q[n], kc[n], vc[n], S, "causal_segment", seg)
        if dt == "f32":
            assert_fp32_close(got[n], ref, f"causal_segment n={n}")
        else:
            assert_bf16_close(got[n].reshape(-1, D), ref.reshape(-1, D), f"causal_segment n={n}")


@pytest.mark.parametrize("G", [1, 4])
def test_prefill_group_sizes(K, G):
    _prefill_case(K, 128, 130, "causal", "bf16", G, seed=G)
    _prefill_case(K, 64, 70, "causal", "f32", G, seed=G + 10)


# ----------------------------------------------------------------------------
# (c) decode
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("dt,G", [("bf16", 2), ("f32", 2), ("bf16", 1), ("bf16", 4), ("f32", 4)])
def test_decode_parity_ragged_with_canaries(K, dt, G):
    torch = T()
    rng = np.random.default_rng(31 + G)
    Hkv, D = 4, 128
    Hq = Hkv * G
    lengths = np.array([1, 2, 63, 64, 65, 300, 1000, 4097, 777], np.int32)
    B, W = lengths.size, 4200
    q = O.store(rng.standard_normal((B, Hq, D)), dt)
    kc = O.store(rng.standard_normal((B, Hkv, W, D)), dt)
    vc = O.store(rng.standard_normal((B, Hkv, W, D)), dt)
    tdt = _tdt(dt)
    kd, vd = dev(kc, tdt), dev(vc, tdt)
    for b, L in enumerate(lengths):          # canaries past the valid prefix
        kd[b, :, L:] = float("nan"); vd[b, :, L:] = float("inf")
    ws = torch.zeros(K.decode_workspace_bytes(B, Hkv, Hq, W, D), dtype=torch.uint8, device="cuda")
    for rep in range(2):                     # second call reuses the self-clearing workspace
        out = torch.full((B, Hq, D), float("nan"), device="cuda")
        K.kv_attn_decode(dev(q, tdt), K.KVCache(kd, vd), dev(lengths), lengths, out, ws)
        torch.cuda.synchronize()
        got = host(out)
        assert np.all(np.isfinite(got))
        for b in range(B):
            ref = O.decode(q[b], kc[b], vc[b], int(lengths[b]))
            if dt == "f32":
                assert_fp32_close(got[b], ref, f"decode b={b} L={lengths[b]}")
            else:
                assert_bf16_close(got[b], ref, f"decode b={b} L={lengths[b]}")
        zero = K.lib().kva_decode_workspace_zero_bytes(B, Hkv)
        assert int(ws[:zero].sum()) == 0     # counters left at zero


def test_decode_single_key_returns_value(K):
    torch = T()
    B, Hkv, D, W = 3, 8, 128, 4
    kc = torch.randn((B, Hkv, W, D), device="cuda").to(torch.bfloat16)
    vc = torch.randn((B, Hkv, W, D), device="cuda").to(torch.bfloat16)
    q = torch.randn((B, 16, D), device="cuda")
    ws = torch.zeros(K.decode_workspace_bytes(B, Hkv, 16, W, D), dtype=torch.uint8, device="cuda")
    out = torch.empty((B, 16, D), device="cuda")
    lengths = np.ones(B, np.int32)
    K.kv_attn_decode(q, K.KVCache(kc, vc), dev(lengths), lengths, out, ws)
    torch.cuda.synchronize()
    expect = vc[:, :, 0].float().repeat_interleave(2, dim=1)
    assert torch.equal(out, expect)


def test_decode_equals_prefill_last_row_fp32(K):
    """Decode at step t equals prefill row t over the same cache (the pages report 3.0e-7)."""
    torch = T()
    rng = np.random.default_rng(77)
    S, Hkv, Hq, D = 80, 8, 16, 128
    q = rng.standard_normal((1, S, Hq, D)).astype(np.float32)
    kc = rng.standard_normal((1, Hkv, S, D)).astype(np.float32)
    vc = rng.standard_normal((1, Hkv, S, D)).astype(np.float32)
    cache = K.KVCache(dev(kc), dev(vc))
    pre = torch.empty((1, S, Hq, D), device="cuda")
    K.kv_attn_prefill(dev(q), cache, pre, mask="causal")
    ws = torch.zeros(K.decode_workspace_bytes(1, Hkv, Hq, S, D), dtype=torch.uint8, device="cuda")
    for t in (0, 1, 40, 63, 64, 79):
        out = torch.empty((1, Hq, D), device="cuda")
        L = np.array([t + 1], np.int32)
        K.kv_attn_decode(dev(q[:, t]), cache, dev(L), L, out, ws)
        torch.cuda.synchronize()
        assert row_rel_err(host(out[0]), host(pre[0, t])) <= 1e-5


# ----------------------------------------------------------------------------
# (d) lm_head + argmax
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("B,H,V,Vrows,wdt", [(1, 1024, 1000, 1000, "bf16"), (3, 1024, 1001, 1013, "bf16"),
                                             (9, 64, 37, 37, "f32"), (64, 1024, 5000, 5000, "bf16"),
                                             (1, 8, 300, 300, "f32"), (1, 1024, 151936, 151936, "bf16"),
                                             (17, 2048, 3001, 3001, "bf16"), (128, 1024, 1290, 1290, "bf16"),
                                             (2, 1032, 700, 700, "bf16"), (1, 2560, 999, 1000, "bf16")])
def test_lmhead_parity(K, B, H, V, Vrows, wdt):
    torch = T()
    rng = np.random.default_rng(B * 1000 + V)
    Wf = (0.02 * rng.standard_normal((Vrows, H))).astype(np.float32)
    W = WL.f32_to_bf16_bits(Wf) if wdt == "bf16" else Wf
    h = rng.standard_normal((B, H)).astype(np.float32)
    Wd = dev(W)
    ws = torch.zeros(K.lmhead_workspace_bytes(B, H), dtype=torch.uint8, device="cuda")
    zero = K.lib().kva_lmhead_workspace_zero_bytes(B)
    for rep in range(2):
        ids = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        mx = torch.empty((B,), device="cuda")
        logits = torch.empty((B, V), device="cuda")
        K.lmhead_argmax(dev(h), Wd, ids, ws, V=V, out_max=mx, logits=logits)
        torch.cuda.synchronize()
        ref_ids, ref_max, margin = O.lmhead_argmax(h, W, V)
        z = np.stack([O.lm_logits(h[b], W, V) for b in range(B)])
        assert np.max(np.abs(host(logits) - z)) <= 1e-5 * max(1.0, float(np.max(np.abs(z))))
        got = ids.cpu().numpy()
        for b in range(B):
            if margin[b] > ARGMAX_MARGIN:
                assert got[b] == ref_ids[b]
            else:                            # near-tie: any id within the margin is a valid pick
                assert z[b, got[b]] >= ref_max[b] - ARGMAX_MARGIN
            assert abs(float(mx[b]) - ref_max[b]) <= 1e-5 * max(1.0, abs(ref_max[b]))
        assert int(ws[:zero].sum()) == 0                 # counter and keys left at zero


def test_lmhead_ties_lowest_id_last_row_and_clamp(K):
    torch = T()
    H, Vrows = 64, 4099
    W = np.zeros((Vrows, H), np.float32)
    h = np.ones((4, H), np.float32)
    W[17] = 0.5; W[4000] = 0.5            # exact tie between 17 and 4000 (batch 0)
    h[1] = -1.0                            # batch 1: every row ties at 0 except the negatives
    W[4098] = 1.0                          # last row: wins for batch 2 / 3 unless clamped
    Wd = dev(W)
    ws = torch.zeros(K.lmhead_workspace_bytes(4, H), dtype=torch.uint8, device="cuda")
    ids = torch.empty((4,), dtype=torch.int32, device="cuda")
    K.lmhead_argmax(dev(h), Wd, ids, ws, V=Vrows)
    torch.cuda.synchronize()
    got = ids.cpu().numpy()
    assert got[0] == 4098 and got[1] == 0 and got[2] == 4098
    K.lmhead_argmax(dev(h), Wd, ids, ws, V=4098)          # clamp: row 4098 is not a candidate
    torch.cuda.synchronize()
    got = ids.cpu().numpy()
    assert got[0] == 17 and got[1] == 0 and got[2] == 17
    # a +0 / -0 tie: with h = 2^-100 a row of -2^-100 weights gives products that round to
    # -0, so its logit is -0.0; a row of zeros gives +0.0; every other row is negative.
    # The two zeros are equal logits, so the lower id wins whichever sign it carries.
    tiny = 2.0 ** -100
    for lo_row, hi_row, lo_val, hi_val in ((5, 4000, -tiny, 0.0), (5, 4000, 0.0, -tiny)):
        W = np.full((Vrows, H), -1.0, np.float32)
        W[lo_row] = lo_val
        W[hi_row] = hi_val
        for Wd in (dev(W), dev(W).to(torch.bfloat16)):           # exact in both dtypes
            for B in (1, 4):
                hz = np.full((B, H), tiny, np.float32)
                ids = torch.empty((B,), dtype=torch.int32, device="cuda")
                K.lmhead_argmax(dev(hz), Wd, ids, ws, V=Vrows)
                torch.cuda.synchronize()
                assert np.all(ids.cpu().numpy() == lo_row), (Wd.dtype, B, lo_val, ids.cpu().numpy())


def test_lmhead_b1_pipeline_ties_across_stages_and_ctas(K):
    """The batch-1 pipelined kernel (hidden 1024, bf16 table of the full vocabulary) hands its
    16-row stages to the CTAs in turn (CTA c takes stages c, c + P, ...): exact ties between
    rows that different CTAs reduce, or that one CTA reduces in different stages, go to the
    lowest id, as do ties with the last row."""
    torch = T()
    H, V = 1024, 151936
    P = torch.cuda.get_device_properties(0).multi_processor_count
    W = torch.full((V, H), -0.01, device="cuda", dtype=torch.bfloat16)
    h = torch.ones((1, H), device="cuda")
    ws = torch.zeros(K.lmhead_workspace_bytes(1, H), dtype=torch.uint8, device="cuda")
    ids = torch.empty((1,), dtype=torch.int32, device="cuda")
    cases = [(20, 5000),                          # stages 1 and 312: different CTAs
             (20, 20 + 16 * P),                   # one CTA, stages 1 and 1 + P
             (20 + 16 * P * 3, 7),                # the higher id reduced first by its CTA
             (V - 1, V - 2), (3, V - 1)]          # the last rows
    for rows in cases:
        W[list(rows)] = 0.01
        K.lmhead_argmax(h, W, ids, ws)
        torch.cuda.synchronize()
        assert int(ids.cpu()[0]) == min(rows), (rows, int(ids.cpu()[0]))
        W[list(rows)] = -0.01


@pytest.mark.parametrize("mask", ["causal", "full"])
def test_prefill_bf16_long_prompt_sampled_rows(K, mask):
    """A 4096-token prompt (32 row tiles, 32 key tiles per row tile under the full mask), two
    instances, 16/8 heads: every head of sampled rows against the oracle."""
    torch = T()
    N, S, Hkv, G, D = 2, 4096, 8, 2, 128
    Hq = Hkv * G
    g = torch.Generator(device="cuda"); g.manual_seed(4096 + len(mask))
    kc = torch.randn((N, Hkv, S, D), device="cuda", generator=g).to(torch.bfloat16)
    vc = torch.randn_like(kc)
    q = torch.randn((N, S, Hq, D), device="cuda", generator=g).to(torch.bfloat16)
    out = torch.full((N, S, Hq, D), float("nan"), device="cuda")
    K.kv_attn_prefill(q, K.KVCache(kc, vc), out, mask=mask)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    rows = np.array([0, 1, 127, 128, 1000, 2047, 2048, 3071, 4094, 4095])
    for n in range(N):
        kh, vh = host(kc[n]), host(vc[n])
        allowed = np.zeros((rows.size, S), bool)
        for i, r in enumerate(rows):
            allowed[i, :(r + 1 if mask == "causal" else S)] = True
        ref = O.attend(host(q[n])[rows], kh, vh, allowed)
        assert_bf16_close(host(out[n])[rows], ref, f"long prompt n={n} {mask}")
