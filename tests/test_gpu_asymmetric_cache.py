"""GPU parity of the asymmetric MLA-expanded cache (K rows 192 wide, V rows 128, Hq = Hkv = 32, a
512-slot window, interleaved RoPE on the last 64 K dims: Youtu-VL-4B port, section 6 and
implementation difficulty 2) against the oracle, through every entry point that takes it: the
general-layout append (also with QK-Norm, other RoPE kinds on sub-ranges and head widths the fast
append forms do not tile), prefill with causal / full / segment masks and GQA groups, split-KV
decode with ragged lengths and NaN canaries, and the whole append -> prefill -> decode chain.

The prefill and decode kernels for this layout compute in fp32 from the stored values, so they are
held to the fp32 bound (1e-5 per-row relative) for bf16 caches too."""
import zlib

import numpy as np
import pytest

import oracle as O
from helpers import assert_bf16_close, assert_bf16_store, assert_fp32_close, bf16_bits, dev, host

pytestmark = pytest.mark.gpu

DK, DV = 192, 128
MLA_ROPE = dict(kind="interleaved", base=1e6, rot_offset=128, rot_dim=64)


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


def _orope(kind, base, rot_offset, rot_dim, sections=None):
    return O.Rope(kind, base, sections, rot_offset=rot_offset, rot_dim=rot_dim)


# ----------------------------------------------------------------------------
# append (general-layout form)
# ----------------------------------------------------------------------------
APPEND_CASES = [
    # Dk, Dv, Hkv, G, rope kind, sections, rot_offset, rot_dim, norm, in, q_out, cache
    (DK, DV, 32, 1, "interleaved", None, 128, 64, None, "bf16", "bf16", "bf16"),      # the MLA layer
    (DK, DV, 32, 1, "interleaved", None, 128, 64, None, "f32", "f32", "f32"),
    (DK, DV, 4, 2, "1d", None, 64, 128, "before", "f32", "bf16", "bf16"),
    (DK, DV, 4, 1, "2d", None, 32, 96, "after", "f32", "f32", "f32"),
    (DK, DV, 4, 4, "sections", (8, 8, 8, 8), 128, 64, "before", "bf16", "f32", "bf16"),
    (96, 96, 2, 2, "1d", None, 0, 0, "before", "f32", "f32", "f32"),                  # a width the fast forms skip
    (128, 128, 4, 2, "1d", None, 64, 64, None, "f32", "bf16", "bf16"),                # sub-range, symmetric head
    (136, 64, 2, 1, "interleaved", None, 8, 120, "after", "f32", "f32", "f32"),
]


@pytest.mark.parametrize("Dk,Dv,Hkv,G,kind,secs,ro,rw,norm,in_dt,qo_dt,c_dt", APPEND_CASES)
def test_append_general_parity(K, Dk, Dv, Hkv, G, kind, secs, ro, rw, norm, in_dt, qo_dt, c_dt):
    torch = T()
    rng = np.random.default_rng(zlib.crc32(repr(("gen", Dk, Dv, kind, ro, rw, norm, in_dt, qo_dt, c_dt)).encode()))
    N, Tt, W = 3, 37, 64
    Hq = Hkv * G
    q = rng.standard_normal((N, Tt, Hq, Dk)).astype(np.float32) * 3
    k = rng.standard_normal((N, Tt, Hkv, Dk)).astype(np.float32) * 3
    v = rng.standard_normal((N, Tt, Hkv, Dv)).astype(np.float32)
    n_axes = {"1d": 1, "sections": 4, "2d": 2, "interleaved": 1}[kind]
    pos = rng.integers(0, 40000, size=(N, Tt, n_axes)).astype(np.int32)
    slot = np.stack([rng.permutation(W)[:Tt] for _ in range(N)]).astype(np.int32)
    qw = (1 + 0.1 * rng.standard_normal((N, Dk))).astype(np.float32)
    kw = (1 + 0.1 * rng.standard_normal((N, Dk))).astype(np.float32)
    base = 1.11588e7 if kind == "sections" else 1e6
    kc = torch.full((N, Hkv, W, Dk), 7.0, device="cuda", dtype=_tdt(c_dt))
    vc = torch.full((N, Hkv, W, Dv), 7.0, device="cuda", dtype=_tdt(c_dt))
    q_out = torch.empty((N, Tt, Hq, Dk), device="cuda", dtype=_tdt(qo_dt))
    K.kv_cache_append_rope_qknorm(
        dev(q, _tdt(in_dt)), dev(k, _tdt(in_dt)), dev(v, _tdt(in_dt)), dev(pos), dev(slot), slot, K.KVCache(kc, vc),
        q_out, K.Rope(kind, base, secs or (), rot_offset=ro, rot_dim=rw),
        q_norm_w=dev(qw) if norm else None, k_norm_w=dev(kw) if norm else None, eps=1e-6,
        norm_after_rope=(norm == "after"), norm_inst_stride=Dk)
    torch.cuda.synchronize()
    rope = _orope(kind, base, ro, rw or None, secs)
    kc_h, vc_h = host(kc), host(vc)
    kb = bf16_bits(kc) if c_dt == "bf16" else None
    for n in range(N):
        qx, kx, vx = (O.store(a[n], in_dt) for a in (q, k, v))
        ck, cv = np.full((Hkv, W, Dk), 7.0), np.full((Hkv, W, Dv), 7.0)
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
        np.testing.assert_array_equal(vc_h[n][:, written], cv[:, written])          # V stored unchanged
        assert np.all(kc_h[n][:, ~written] == 7.0) and np.all(vc_h[n][:, ~written] == 7.0)


def test_append_general_non_rotated_dims_pass_through_bit_exact(K):
    """Without a norm the 128 dims outside the rotary range are copied: bit-exact to the input."""
    torch = T()
    rng = np.random.default_rng(41)
    N, Tt, H, W = 1, 9, 32, 16
    q = rng.standard_normal((N, Tt, H, DK)).astype(np.float32)
    k = rng.standard_normal((N, Tt, H, DK)).astype(np.float32)
    v = rng.standard_normal((N, Tt, H, DV)).astype(np.float32)
    pos = np.arange(Tt, dtype=np.int32).reshape(1, Tt, 1) + 100
    slot = np.arange(Tt, dtype=np.int32).reshape(1, Tt)
    kc = torch.zeros((N, H, W, DK), device="cuda")
    vc = torch.zeros((N, H, W, DV), device="cuda")
    q_out = torch.empty((N, Tt, H, DK), device="cuda")
    K.kv_cache_append_rope_qknorm(dev(q), dev(k), dev(v), dev(pos), dev(slot), slot, K.KVCache(kc, vc), q_out,
                                  K.Rope(**MLA_ROPE))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(q_out)[..., :128], q[..., :128])
    np.testing.assert_array_equal(host(kc)[0, :, :Tt, :128], k[0].transpose(1, 0, 2)[..., :128])


# ----------------------------------------------------------------------------
# prefill
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("S,mask,G", [(1, "causal", 1), (63, "causal", 1), (300, "causal", 1), (512, "causal", 1),
                                      (130, "full", 2), (200, "segment", 1), (129, "causal", 4)])
def test_prefill_asymmetric(K, dt, S, mask, G):
    torch = T()
    rng = np.random.default_rng(zlib.crc32(repr(("asym-pf", dt, S, mask, G)).encode()))
    N, Hkv, W = 2, 2, 512
    Hq = Hkv * G
    q = O.store(rng.standard_normal((N, S, Hq, DK)), dt)
    kc = O.store(rng.standard_normal((N, Hkv, W, DK)), dt)
    vc = O.store(rng.standard_normal((N, Hkv, W, DV)), dt)
    seg = None
    if mask == "segment":
        seg = np.repeat(np.arange((S + 63) // 64), 64)[:S].astype(np.int32)
        seg[100:] += 7                                    # a window boundary inside a tile
    tdt = _tdt(dt)
    kd, vd = dev(kc, tdt), dev(vc, tdt)
    kd[:, :, S:] = float("nan"); vd[:, :, S:] = float("inf")     # slots past S are never read
    out = torch.full((N, S, Hq, DV), float("nan"), device="cuda")
    K.kv_attn_prefill(dev(q, tdt), K.KVCache(kd, vd), out, mask=mask,
                      segment=dev(seg) if seg is not None else None, segment_host=seg)
    torch.cuda.synchronize()
    got = host(out)
    for n in range(N):
        ref = O.prefill(q[n], kc[n], vc[n], S, mask, seg)
        if dt == "f32":
            assert_fp32_close(got[n], ref, f"asym prefill n={n} S={S} {mask}")
        else:                      # tensor-core path: P enters P V as bf16 (bf16-cache tolerance)
            assert_bf16_close(got[n], ref, f"asym prefill n={n} S={S} {mask}")


# ----------------------------------------------------------------------------
# decode
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("dt,G", [("bf16", 1), ("f32", 1), ("bf16", 2), ("bf16", 4), ("f32", 4)])
def test_decode_asymmetric_ragged_with_canaries(K, dt, G):
    torch = T()
    rng = np.random.default_rng(zlib.crc32(repr(("asym-dec", dt, G)).encode()))
    Hkv = 4
    Hq = Hkv * G
    lengths = np.array([1, 2, 63, 64, 65, 511, 512, 3000], np.int32)
    B, W = lengths.size, 3072
    q = O.store(rng.standard_normal((B, Hq, DK)), dt)
    kc = O.store(rng.standard_normal((B, Hkv, W, DK)), dt)
    vc = O.store(rng.standard_normal((B, Hkv, W, DV)), dt)
    tdt = _tdt(dt)
    kd, vd = dev(kc, tdt), dev(vc, tdt)
    for b, L in enumerate(lengths):
        kd[b, :, L:] = float("nan"); vd[b, :, L:] = float("inf")
    ws = torch.zeros(K.decode_workspace_bytes(B, Hkv, Hq, W, DV), dtype=torch.uint8, device="cuda")
    for rep in range(2):                                 # the second call reuses the self-clearing workspace
        out = torch.full((B, Hq, DV), float("nan"), device="cuda")
        K.kv_attn_decode(dev(q, tdt), K.KVCache(kd, vd), dev(lengths), lengths, out, ws)
        torch.cuda.synchronize()
        got = host(out)
        assert np.all(np.isfinite(got))
        zero = K.lib().kva_decode_workspace_zero_bytes(B, Hkv)
        assert int(ws[:zero].sum()) == 0
    for b in range(B):
        ref = O.decode(q[b], kc[b], vc[b], int(lengths[b]))
        assert_fp32_close(got[b], ref, f"asym decode b={b} L={lengths[b]}")


# ----------------------------------------------------------------------------
# the whole layer step over the 512-slot window
# ----------------------------------------------------------------------------
def test_mla_append_prefill_decode_chain(K):
    """Append a 300-token prompt (interleaved RoPE on dims 128..191), prefill it, then three decode
    steps (append one token, attend to the prefix): every output against the oracle's chain."""
    torch = T()
    rng = np.random.default_rng(77)
    H, W, S, steps = 32, 512, 300, 3
    rope_o = _orope("interleaved", 1e6, 128, 64)
    rope_k = K.Rope(**MLA_ROPE)
    kc = torch.zeros((1, H, W, DK), device="cuda", dtype=torch.bfloat16)
    vc = torch.zeros((1, H, W, DV), device="cuda", dtype=torch.bfloat16)
    cache = K.KVCache(kc, vc)
    ck, cv = np.zeros((H, W, DK)), np.zeros((H, W, DV))
    q = O.store(rng.standard_normal((1, S, H, DK)), "bf16")
    k = O.store(rng.standard_normal((1, S, H, DK)), "bf16")
    v = O.store(rng.standard_normal((1, S, H, DV)), "bf16")
    pos = np.arange(S, dtype=np.int32).reshape(1, S, 1)
    slot = np.arange(S, dtype=np.int32).reshape(1, S)
    q_out = torch.empty((1, S, H, DK), device="cuda", dtype=torch.bfloat16)
    K.kv_cache_append_rope_qknorm(dev(q, torch.bfloat16), dev(k, torch.bfloat16), dev(v, torch.bfloat16), dev(pos),
                                  dev(slot), slot, cache, q_out, rope_k)
    out = torch.empty((1, S, H, DV), device="cuda")
    K.kv_attn_prefill(q_out, cache, out, mask="causal")
    torch.cuda.synchronize()
    qr = O.cache_append(q[0], k[0], v[0], pos[0], slot[0], None, None, 1e-6, rope_o, False, ck, cv, "bf16")
    k_exact = [O.qk_transform(k[0], pos[0], None, 1e-6, rope_o, False)]
    # each stage against the oracle on that stage's own inputs: the stored queries and cache rows
    # (which the append check bounds against the oracle's to one bf16 rounding)
    assert_bf16_store(bf16_bits(q_out)[0], qr, "prompt q_out")
    # the bf16 prompt prefill runs on the tensor cores (P enters P V as bf16): bf16-cache tolerance
    assert_bf16_close(host(out)[0], O.prefill(host(q_out)[0], host(kc)[0], host(vc)[0], S, "causal"),
                      "prompt prefill")
    ws = torch.zeros(K.decode_workspace_bytes(1, H, H, W, DV), dtype=torch.uint8, device="cuda")
    for s in range(steps):
        L = S + s + 1
        qn = O.store(rng.standard_normal((1, 1, H, DK)), "bf16")
        kn = O.store(rng.standard_normal((1, 1, H, DK)), "bf16")
        vn = O.store(rng.standard_normal((1, 1, H, DV)), "bf16")
        p = np.array([[[L - 1]]], np.int32)
        sl = np.array([[L - 1]], np.int32)
        qo = torch.empty((1, 1, H, DK), device="cuda", dtype=torch.bfloat16)
        K.kv_cache_append_rope_qknorm(dev(qn, torch.bfloat16), dev(kn, torch.bfloat16), dev(vn, torch.bfloat16),
                                      dev(p), dev(sl), sl, cache, qo, rope_k)
        lens = np.array([L], np.int32)
        o = torch.empty((1, H, DV), device="cuda")
        K.kv_attn_decode(qo[:, 0], cache, dev(lens), lens, o, ws)
        torch.cuda.synchronize()
        qn_r = O.cache_append(qn[0], kn[0], vn[0], p[0], sl[0], None, None, 1e-6, rope_o, False, ck, cv, "bf16")
        k_exact.append(O.qk_transform(kn[0], p[0], None, 1e-6, rope_o, False))
        assert_bf16_store(bf16_bits(qo)[0], qn_r, f"decode step {s} q_out")
        assert_fp32_close(host(o)[0], O.decode(host(qo)[0, 0], host(kc)[0], host(vc)[0], L), f"decode step {s}")
    # the cache after the chain: K within one bf16 rounding of the exact rotated keys (and
    # bit-exact outside the rotary dims), V bit-exact, the rest of the window untouched
    n = S + steps
    kex = np.concatenate(k_exact, axis=0).transpose(1, 0, 2)          # [H, n, DK]
    assert_bf16_store(bf16_bits(kc)[0][:, :n], kex, "cache K after the chain")
    kh = host(kc)[0]
    np.testing.assert_array_equal(kh[:, :n, :128], ck[:, :n, :128])
    np.testing.assert_array_equal(host(vc)[0][:, :n], cv[:, :n])
    assert not np.any(kh[:, n:]) and not np.any(host(vc)[0][:, n:])


@pytest.mark.parametrize("fused", [True, False], ids=["decode_step", "append_then_decode"])
def test_mla_benchmark_shapes_full_window(K, fused):
    """The shapes the benchmark times for the MLA-expanded cache: a 512-token prompt filling the
    512-slot window (append + causal prefill), then a token written into the last slot and
    decoded over the whole window (fused: one kv_attn_decode_step launch, as the benchmark runs
    it); sampled prompt rows and the token against the oracle."""
    torch = T()
    rng = np.random.default_rng(78)
    H, W = 32, 512
    rope_o = _orope("interleaved", 1e6, 128, 64)
    rope_k = K.Rope(**MLA_ROPE)
    kc = torch.zeros((1, H, W, DK), device="cuda", dtype=torch.bfloat16)
    vc = torch.zeros((1, H, W, DV), device="cuda", dtype=torch.bfloat16)
    cache = K.KVCache(kc, vc)
    q = O.store(rng.standard_normal((1, W, H, DK)), "bf16")
    k = O.store(rng.standard_normal((1, W, H, DK)), "bf16")
    v = O.store(rng.standard_normal((1, W, H, DV)), "bf16")
    pos = np.arange(W, dtype=np.int32).reshape(1, W, 1)
    slot = np.arange(W, dtype=np.int32).reshape(1, W)
    q_out = torch.empty((1, W, H, DK), device="cuda", dtype=torch.bfloat16)
    K.kv_cache_append_rope_qknorm(dev(q, torch.bfloat16), dev(k, torch.bfloat16), dev(v, torch.bfloat16), dev(pos),
                                  dev(slot), slot, cache, q_out, rope_k)
    out = torch.empty((1, W, H, DV), device="cuda")
    K.kv_attn_prefill(q_out, cache, out, mask="causal")
    torch.cuda.synchronize()
    rows = np.array([0, 1, 127, 128, 255, 256, 383, 384, 510, 511])
    kh, vh, qh = host(kc)[0], host(vc)[0], host(q_out)[0]
    allowed = np.zeros((rows.size, W), bool)
    for i, r in enumerate(rows):
        allowed[i, :r + 1] = True
    assert_bf16_close(host(out)[0][rows], O.attend(qh[rows], kh, vh, allowed), "prompt prefill rows")
    # the token: written into slot W - 1 (position W - 1), decode over all W slots
    qn = O.store(rng.standard_normal((1, 1, H, DK)), "bf16")
    kn = O.store(rng.standard_normal((1, 1, H, DK)), "bf16")
    vn = O.store(rng.standard_normal((1, 1, H, DV)), "bf16")
    p = np.array([[[W - 1]]], np.int32)
    sl = np.array([[W - 1]], np.int32)
    qo = torch.empty((1, 1, H, DK), device="cuda", dtype=torch.bfloat16)
    lens = np.array([W], np.int32)
    ws = torch.zeros(K.decode_workspace_bytes(1, H, H, W, DV), dtype=torch.uint8, device="cuda")
    o = torch.empty((1, H, DV), device="cuda")
    if fused:
        K.kv_attn_decode_step(dev(qn[0], torch.bfloat16), dev(kn[0], torch.bfloat16), dev(vn[0], torch.bfloat16),
                              dev(p[0]), cache, dev(lens), lens, o, ws, rope_k, q_out=qo[:, 0])
    else:
        K.kv_cache_append_rope_qknorm(dev(qn, torch.bfloat16), dev(kn, torch.bfloat16), dev(vn, torch.bfloat16),
                                      dev(p), dev(sl), sl, cache, qo, rope_k)
        K.kv_attn_decode(qo[:, 0], cache, dev(lens), lens, o, ws)
    torch.cuda.synchronize()
    kex = O.qk_transform(kn[0], p[0], None, 1e-6, rope_o, False)            # [1, H, DK]
    assert_bf16_store(bf16_bits(kc)[0][:, W - 1:W], kex.transpose(1, 0, 2), "token K row")
    qex = O.qk_transform(qn[0], p[0], None, 1e-6, rope_o, False)[0]         # [H, DK], exact
    assert_bf16_store(bf16_bits(qo)[0, 0], qex, "token q_out")
    # the fused step attends with its fp32 query, the two calls with the stored bf16 one
    q_used = qex if fused else host(qo)[0, 0]
    assert_fp32_close(host(o)[0], O.decode(q_used, host(kc)[0], host(vc)[0], W), "token decode")
