"""Pins of the CPU oracle against things other than itself: hand-derived closed forms,
invariants the mathematics fixes, library routines, brute force on tiny inputs, and the
values the pages print (tests/golden/page_values.json).

Each pin is chosen so that a plausible slip in the oracle (a dropped term, a wrong sign
or index, a transposed operand, a swapped axis) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O
import workloads as WL

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_values.json")))


# ----------------------------------------------------------------------------
# QK-Norm
# ----------------------------------------------------------------------------
def test_rmsnorm_hand_example():
    # x = [3, 4]: mean square 12.5, so y = x / sqrt(12.5) * w (eps = 0).
    y = O.rms_norm(np.array([3.0, 4.0]), np.array([2.0, 0.5]), 0.0)
    np.testing.assert_allclose(y, [1.6970562748477140, 0.5656854249492380], rtol=1e-15)


def test_rmsnorm_eps_inside_sqrt():
    # x = [1, 1], eps = 1: 1 / sqrt(1 + 1) = 0.7071...
    y = O.rms_norm(np.array([1.0, 1.0]), np.ones(2), 1.0)
    np.testing.assert_allclose(y, [0.7071067811865476] * 2, rtol=1e-15)
    # all-zero row stays finite and zero
    assert np.all(O.rms_norm(np.zeros(8), np.ones(8), 1e-6) == 0.0)


def test_rmsnorm_unit_rms_closed_form():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 3, 128)) * 7.0
    eps = 1e-6
    y = O.rms_norm(x, np.ones(128), eps)
    ms = np.mean(x * x, axis=-1)
    rms_y = np.sqrt(np.mean(y * y, axis=-1))
    np.testing.assert_allclose(rms_y, np.sqrt(ms / (ms + eps)), rtol=1e-14)


def test_rmsnorm_scale_invariance():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((4, 128))
    w = 1 + 0.1 * rng.standard_normal(128)
    np.testing.assert_allclose(O.rms_norm(37.0 * x, w, 0.0), O.rms_norm(x, w, 0.0), rtol=1e-13)


# ----------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------
ROPE1D = O.Rope("1d", base=100.0)


def test_rope_hand_examples_1d():
    # D = 4, base 100: inv = [1, 100^(-2/4)] = [1, 0.1].
    x = np.eye(4)[:, None, :]                      # 4 "tokens" = unit vectors e0..e3
    pos = np.array([[1], [2], [1], [2]])
    y = O.rope_apply(x, pos, ROPE1D)[:, 0, :]
    # e0 at pos 1: pair (0, 2), angle 1 -> y0 = cos 1, y2 = sin 1
    np.testing.assert_allclose(y[0], [0.5403023058681398, 0, 0.8414709848078965, 0], atol=1e-16)
    # e1 at pos 2: pair (1, 3), angle 0.2 -> y1 = cos .2, y3 = sin .2
    np.testing.assert_allclose(y[1], [0, 0.9800665778412416, 0, 0.19866933079506122], atol=1e-16)
    # e2 at pos 1 (second half of pair 0): y0 = -sin 1, y2 = cos 1
    np.testing.assert_allclose(y[2], [-0.8414709848078965, 0, 0.5403023058681398, 0], atol=1e-16)
    # e3 at pos 2: y1 = -sin .2, y3 = cos .2
    np.testing.assert_allclose(y[3], [0, -0.19866933079506122, 0, 0.9800665778412416], atol=1e-16)


def test_rope_position_zero_is_identity():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 2, 128))
    for rope, n_axes in ((O.Rope("1d", 1e6), 1), (O.Rope("sections", 1.11588e7, (16,) * 4), 4),
                         (O.Rope("2d", 1e6), 2)):
        np.testing.assert_array_equal(O.rope_apply(x, np.zeros((3, n_axes), int), rope), x)


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((7, 3, 128))
    pos = rng.integers(0, 40000, size=(7, 1))
    y = O.rope_apply(x, pos, O.Rope("1d", 1e6))
    n_in = x[..., :64] ** 2 + x[..., 64:] ** 2
    n_out = y[..., :64] ** 2 + y[..., 64:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-13)


def test_rope_relative_position_property():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 1, 128))
    k = rng.standard_normal((1, 1, 128))
    rope = O.Rope("1d", 1e6)
    dots = []
    for p in (0, 5, 333, 4096):
        qr = O.rope_apply(q, [[p + 17]], rope)
        kr = O.rope_apply(k, [[p]], rope)
        dots.append(float(np.sum(qr * kr)))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-11)


def test_xdrope_sections_pick_axes():
    # D = 8, four sections of one frequency each, base 16: inv = 16^(-j/4) = 1, 1/2, 1/4, 1/8.
    # Positions (1, 2, 4, 8) on the four axes give angle 1 for every pair.
    rope = O.Rope("sections", base=16.0, sections=(1, 1, 1, 1))
    x = np.zeros((1, 1, 8)); x[..., :4] = 1.0
    y = O.rope_apply(x, [[1, 2, 4, 8]], rope)[0, 0]
    np.testing.assert_allclose(y[:4], [math.cos(1.0)] * 4, rtol=1e-15)
    np.testing.assert_allclose(y[4:], [math.sin(1.0)] * 4, rtol=1e-15)


def test_xdrope_equal_axes_is_1d():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((6, 2, 128))
    p = rng.integers(0, 600, size=(6, 1))
    a = O.rope_apply(x, np.repeat(p, 4, axis=1), O.Rope("sections", 1.11588e7, (16,) * 4))
    b = O.rope_apply(x, p, O.Rope("1d", 1.11588e7))
    np.testing.assert_allclose(a, b, rtol=0, atol=0)


def test_rope_2d_hand_example_and_axes():
    # D = 8 -> halves of 4, base 1e6: inv (width 4) = [1, 1e-3].
    rope = O.Rope("2d", 1e6)
    x = np.zeros((1, 1, 8)); x[0, 0, 4] = 1.0      # first element of the column half
    y = O.rope_apply(x, [[5, 1]], rope)[0, 0]       # row 5, col 1
    np.testing.assert_allclose(y, [0, 0, 0, 0, math.cos(1.0), 0, math.sin(1.0), 0], atol=1e-16)
    x = np.zeros((1, 1, 8)); x[0, 0, 1] = 1.0      # second frequency of the row half
    y = O.rope_apply(x, [[5, 1]], rope)[0, 0]
    np.testing.assert_allclose(y, [0, math.cos(5e-3), 0, math.sin(5e-3), 0, 0, 0, 0], atol=1e-16)


def test_rope_2d_equal_axes_is_per_half_1d():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((5, 3, 72))
    p = rng.integers(0, 92, size=(5, 1))
    a = O.rope_apply(x, np.repeat(p, 2, axis=1), O.Rope("2d", 1e6))
    one = O.Rope("1d", 1e6)
    b = np.concatenate([O.rope_apply(x[..., :36], p, one), O.rope_apply(x[..., 36:], p, one)], -1)
    np.testing.assert_allclose(a, b, rtol=0, atol=0)


def test_norm_rope_order():
    rng = np.random.default_rng(10)
    x = rng.standard_normal((4, 2, 128))
    pos = rng.integers(0, 1000, size=(4, 1))
    rope = O.Rope("1d", 1e6)
    ones = np.ones(128)
    a = O.qk_transform(x, pos, ones, 1e-6, rope, norm_after_rope=False)
    b = O.qk_transform(x, pos, ones, 1e-6, rope, norm_after_rope=True)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)   # RoPE keeps the RMS
    w = 1 + 0.1 * rng.standard_normal(128)
    a = O.qk_transform(x, pos, w, 1e-6, rope, norm_after_rope=False)
    b = O.qk_transform(x, pos, w, 1e-6, rope, norm_after_rope=True)
    assert np.max(np.abs(a - b)) > 1e-3                          # the flag matters


def test_norm_rope_order_direction_hand_worked():
    # D = 4, base 100: inv = [1, 0.1]; position 1 turns pair (0, 2) by 1 rad and pair (1, 3)
    # by 0.1 rad.  w = [2, 0.5, 1, 1], eps = 0.
    #   x = e0:  norm first:  e0 / sqrt(1/4) * w = [4, 0, 0, 0]      -> RoPE [4 cos 1, 0, 4 sin 1, 0]
    #            RoPE first:  [cos 1, 0, sin 1, 0] / (1/2) * w       -> [4 cos 1, 0, 2 sin 1, 0]
    #   x = e1:  norm first:  [0, 1, 0, 0]                            -> [0, cos .1, 0, sin .1]
    #            RoPE first:  [0, 2 cos .1, 0, 2 sin .1] * w          -> [0, cos .1, 0, 2 sin .1]
    # Qwen3 normalises, then rotates (Penguin-VL port, section 5.4: q_proj, q_norm, q_rope);
    # HunyuanOCR rotates, then normalises, before the cache write (HunyuanOCR v1.0 port,
    # section five item 2).  The flag names the second order.
    rope = O.Rope("1d", base=100.0)
    w = np.array([2.0, 0.5, 1.0, 1.0])
    x = np.zeros((2, 1, 4)); x[0, 0, 0] = 1.0; x[1, 0, 1] = 1.0
    pos = np.array([[1], [1]])
    c1, s1, c2, s2 = math.cos(1.0), math.sin(1.0), math.cos(0.1), math.sin(0.1)
    norm_then_rope = [[4 * c1, 0, 4 * s1, 0], [0, c2, 0, s2]]
    rope_then_norm = [[4 * c1, 0, 2 * s1, 0], [0, c2, 0, 2 * s2]]
    a = O.qk_transform(x, pos, w, 0.0, rope, norm_after_rope=False)[:, 0]
    b = O.qk_transform(x, pos, w, 0.0, rope, norm_after_rope=True)[:, 0]
    np.testing.assert_allclose(a, norm_then_rope, rtol=1e-15, atol=1e-16)
    np.testing.assert_allclose(b, rope_then_norm, rtol=1e-15, atol=1e-16)
    # the cache append takes the same flag for q and for k
    ck = np.zeros((1, 2, 4)); cv = np.zeros((1, 2, 4))
    qr = O.cache_append(x, x, x, pos, [0, 1], w, w, 0.0, rope, True, ck, cv, "f32")
    np.testing.assert_allclose(qr[:, 0], rope_then_norm, rtol=1e-15, atol=1e-16)
    np.testing.assert_allclose(ck[0], np.float32(rope_then_norm).astype(np.float64), rtol=0, atol=0)


# ----------------------------------------------------------------------------
# bf16 storage
# ----------------------------------------------------------------------------
def test_bf16_round_ties_to_even():
    u = 2.0 ** -8
    vals = [1 + u, 1 + 3 * u, -(1 + u), 1 + 0.9 * u, 1 + 1.1 * u, 0.0, 2.0 ** -20 * (1 + u)]
    expect = [1.0, 1 + 4 * u, -1.0, 1.0, 1 + 2 * u, 0.0, 2.0 ** -20]
    np.testing.assert_array_equal(O.bf16_round(vals), expect)


def test_bf16_round_matches_library_on_fp32_inputs():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    # add exact ties: low 16 bits 0x8000
    bits = x.view(np.uint32).copy()
    bits[::7] = (bits[::7] & 0xFFFF0000) | 0x8000
    x = bits.view(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.bf16_round(x.astype(np.float64)), ref)


# ----------------------------------------------------------------------------
# Attention
# ----------------------------------------------------------------------------
def test_attention_two_key_closed_form():
    # D = 2, scale 1/sqrt(2).  q = [sqrt(2) ln 3, 0], k0 = 0, k1 = e0  ->  logits 0, ln 3
    # -> p = [1/4, 3/4] -> o = v0/4 + 3 v1/4 = [0.25, 1.5].
    q = np.array([[[math.sqrt(2) * math.log(3.0), 0.0]]])
    K = np.array([[[0.0, 0.0], [1.0, 0.0]]])
    V = np.array([[[1.0, 0.0], [0.0, 2.0]]])
    o = O.attend(q, K, V, np.array([[True, True]]))
    np.testing.assert_allclose(o[0, 0], [0.25, 1.5], rtol=1e-15)


def test_attention_large_logits_stable():
    # logits 1000 and 1000 + ln 3 must not overflow: same p = [1/4, 3/4].
    q = np.array([[[1000.0, math.log(3.0)]]])
    K = np.array([[[1.0, 0.0], [1.0, 1.0]]])
    V = np.array([[[1.0, 0.0], [0.0, 2.0]]])
    o = O.attend(q, K, V, np.array([[True, True]]), scale=1.0)
    np.testing.assert_allclose(o[0, 0], [0.25, 1.5], rtol=1e-12)
    # logits near 1e5: exp of anything but (logit - row max) overflows float64
    q = np.array([[[1.0e5, math.log(3.0)]]])
    o = O.attend(q, K, V, np.array([[True, True]]), scale=1.0)
    np.testing.assert_allclose(o[0, 0], [0.25, 1.5], rtol=1e-12)


def _rand_case(seed, S=9, Hq=4, Hkv=2, D=8, W=12):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((S, Hq, D)), rng.standard_normal((Hkv, W, D)),
            rng.standard_normal((Hkv, W, D)))


def test_attention_brute_force_tiny():
    # Independent formulation: direct ratio sum_j e^{s_j} v_j / sum_j e^{s_j}, scalar loops,
    # no max subtraction, math.fsum.
    q, K, V = _rand_case(12)
    S, Hq, D = q.shape
    allowed = O.prefill_mask(S, "causal")
    allowed = np.concatenate([allowed, np.zeros((S, K.shape[1] - S), bool)], axis=1)
    o = O.attend(q, K, V, allowed)
    for i in range(S):
        for h in range(Hq):
            g = h // 2
            w = []
            for j in range(i + 1):
                s = math.fsum(q[i, h, d] * K[g, j, d] for d in range(D)) / math.sqrt(D)
                w.append(math.exp(s))
            den = math.fsum(w)
            for d in range(D):
                num = math.fsum(w[j] * V[g, j, d] for j in range(i + 1))
                assert abs(o[i, h, d] - num / den) <= 1e-13 * (1 + abs(num / den))


def test_softmax_rows_sum_to_one_and_mask_is_honoured():
    # V = identity rows: o[i] equals the probability row itself.
    rng = np.random.default_rng(13)
    S, D = 10, 10
    q = rng.standard_normal((S, 1, D)) * 3
    K = rng.standard_normal((1, S, D))
    V = np.eye(S)[None]
    for kind, seg in (("causal", None), ("full", None), ("segment", [0, 0, 0, 1, 1, 2, 2, 2, 2, 3])):
        p = O.prefill(q, K, V, S, kind, seg)[:, 0, :]
        np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
        assert np.all(p >= 0)
        assert np.all(p[~O.prefill_mask(S, kind, seg)] == 0.0)


def test_logit_shift_invariance():
    rng = np.random.default_rng(14)
    q = rng.standard_normal((3, 1, 6))
    K = rng.standard_normal((1, 5, 6))
    V = rng.standard_normal((1, 5, 4))
    # append a constant feature: every logit of a row shifts by the same c
    q2 = np.concatenate([q, np.full((3, 1, 1), 2.5)], axis=-1)
    K2 = np.concatenate([K, np.ones((1, 5, 1))], axis=-1)
    allowed = np.ones((3, 5), bool)
    np.testing.assert_allclose(O.attend(q2, K2, V, allowed, scale=1.0),
                               O.attend(q, K, V, allowed, scale=1.0), rtol=1e-13)


def test_causal_row0_and_uniform_v():
    q, K, V = _rand_case(15)
    o = O.prefill(q, K, V, q.shape[0], "causal")
    for h in range(q.shape[1]):
        np.testing.assert_array_equal(o[0, h], V[h // 2, 0])        # only key 0 visible
    Vc = np.full_like(V, -1.25)
    np.testing.assert_allclose(O.prefill(q, K, Vc, q.shape[0], "causal"), -1.25, rtol=1e-15)


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(16)
    K = np.repeat(rng.standard_normal((1, 1, 8)), 6, axis=1)
    V = rng.standard_normal((1, 6, 8))
    q = rng.standard_normal((1, 1, 8))
    o = O.attend(q, K, V, np.ones((1, 6), bool))
    np.testing.assert_allclose(o[0, 0], V[0].mean(axis=0), rtol=1e-14)


def test_gqa_equals_mha_on_repeated_kv():
    q, K, V = _rand_case(17, Hq=8, Hkv=2)
    S = q.shape[0]
    Krep, Vrep = np.repeat(K, 4, axis=0), np.repeat(V, 4, axis=0)   # repeat_interleave
    np.testing.assert_allclose(O.prefill(q, K, V, S, "causal"), O.prefill(q, Krep, Vrep, S, "causal"),
                               rtol=1e-15)


def test_decode_equals_prefill_row():
    q, K, V = _rand_case(18)
    S = q.shape[0]
    pre = O.prefill(q, K, V, S, "causal")
    bound = GOLDEN["decode_vs_prefill_rel_err"]["value"]
    for t in range(S):
        dec = O.decode(q[t], K, V, t + 1)
        rel = np.linalg.norm(dec - pre[t]) / np.linalg.norm(pre[t])
        assert rel <= bound * 1e-6                                   # far inside the page's 3.0e-7


def test_segment_mask_equals_separate_windows_and_is_permutation_invariant():
    rng = np.random.default_rng(19)
    seg = np.array([0, 0, 0, 1, 1, 1, 1, 2, 2])
    S = seg.size
    q = rng.standard_normal((S, 2, 8)); K = rng.standard_normal((2, S, 8)); V = rng.standard_normal((2, S, 8))
    o = O.prefill(q, K, V, S, "segment", seg)
    for w in range(3):
        idx = np.nonzero(seg == w)[0]
        ow = O.prefill(q[idx], K[:, idx], V[:, idx], idx.size, "full")
        np.testing.assert_allclose(o[idx], ow, rtol=1e-13, atol=1e-15)
    perm = np.array([2, 0, 1, 5, 3, 6, 4, 8, 7])                     # permute inside windows
    op = O.prefill(q[perm], K[:, perm], V[:, perm], S, "segment", seg[perm])
    np.testing.assert_allclose(op, o[perm], rtol=1e-13, atol=1e-15)
    # a single segment is full attention
    np.testing.assert_allclose(O.prefill(q, K, V, S, "segment", np.zeros(S, int)),
                               O.prefill(q, K, V, S, "full"), rtol=0, atol=0)


def test_cache_append_slots_and_storage():
    rng = np.random.default_rng(20)
    T, Hq, Hkv, D, W = 3, 4, 2, 8, 6
    q = rng.standard_normal((T, Hq, D)); k = rng.standard_normal((T, Hkv, D)); v = rng.standard_normal((T, Hkv, D))
    ck = np.full((Hkv, W, D), 7.0); cv = np.full((Hkv, W, D), 7.0)
    slot = np.array([4, 0, 2])
    rope = O.Rope("1d", 1e6)
    qr = O.cache_append(q, k, v, [[3], [4], [5]], slot, None, None, 1e-6, rope, False, ck, cv, "bf16")
    np.testing.assert_allclose(qr, O.rope_apply(q, [[3], [4], [5]], rope))
    for t in range(T):
        np.testing.assert_array_equal(cv[:, slot[t]], O.bf16_round(v[t]))
        np.testing.assert_array_equal(ck[:, slot[t]], O.bf16_round(O.rope_apply(k, [[3], [4], [5]], rope)[t]))
    assert np.all(ck[:, [1, 3, 5]] == 7.0) and np.all(cv[:, [1, 3, 5]] == 7.0)   # other slots untouched
    with pytest.raises(IndexError):
        O.cache_append(q[:1], k[:1], v[:1], [[0]], [W], None, None, 1e-6, rope, False, ck, cv, "f32")


# ----------------------------------------------------------------------------
# lm_head + argmax
# ----------------------------------------------------------------------------
def test_lm_logits_against_exact_sums_and_bf16_widening():
    rng = np.random.default_rng(21)
    W = WL.f32_to_bf16_bits(rng.standard_normal((50, 16)).astype(np.float32) * 0.02)
    h = rng.standard_normal(16)
    z = O.lm_logits(h, W, 50)
    Wf = WL.bf16_bits_to_f32(W).astype(np.float64)
    for v in range(50):
        assert abs(z[v] - math.fsum(Wf[v, i] * h[i] for i in range(16))) <= 1e-15
    one = np.array([[0x3F80, 0xC000]], dtype=np.uint16)              # 1.0, -2.0
    np.testing.assert_array_equal(O.lm_logits(np.array([3.0, 0.5]), one, 1), [2.0])


def test_argmax_ties_lowest_id_vocab_clamp_and_last_row():
    H = 8
    W = np.zeros((20, H), dtype=np.float32)
    h = np.ones(H)
    W[7] = 1.0; W[3] = 1.0                                             # tie: 3 and 7
    ids, mx, mg = O.lmhead_argmax(h, W, 20)
    assert ids[0] == 3 and mx[0] == 8.0 and mg[0] == 0.0
    W[19] = 2.0                                                        # last row wins...
    assert O.lmhead_argmax(h, W, 20)[0][0] == 19
    assert O.lmhead_argmax(h, W, 19)[0][0] == 3                        # ...unless clamped away


# ----------------------------------------------------------------------------
# Page-printed values: workload layouts
# ----------------------------------------------------------------------------
def test_image_span_layout_matches_pages():
    g = GOLDEN["image_span"]["value"]
    pos = WL.image_span_positions(0, g["grid_rows"], g["grid_cols"], 0)
    assert pos.shape[0] == g["rows"] == 1 + 16 * 17 + 1
    vt = GOLDEN["visual_token_count"]["value"]
    gh, gw = vt["patch_grid"]; m = vt["merge_size"]
    assert (gh // m) * (gw // m + 1) + 2 == vt["tokens"] == pos.shape[0]
    full = WL.image_span_positions(20, 16, 16, 218)
    assert full.shape == (512, 4)
    assert np.array_equal(full[:20], np.repeat(np.arange(20)[:, None], 4, 1))
    assert np.all(full[:, 0] == np.arange(512))                      # axis 0 is the sequence position
    assert tuple(full[21]) == (21, 0, 0, 0) and tuple(full[21 + 16]) == (37, 0, 16, 0)
    assert tuple(full[292]) == (292, 15, 16, 0)


def test_vision_layout_matches_pages():
    g = GOLDEN["vision_grid"]["value"]
    lay = WL.vision_window_layout()
    assert lay.pos_rc.shape[0] == g["patches"] == g["patch_rows"] * g["patch_cols"]
    assert g["merged_tokens"] == g["patches"] // 4
    assert sum(lay.window_sizes) == g["patches"]
    assert lay.window_sizes == [224] * 5 + [168]
    assert np.array_equal(np.sort(lay.slot), np.arange(1288))
    assert np.array_equal(lay.row_of_slot[lay.slot], np.arange(1288))
    assert np.all(np.diff(lay.segment) >= 0)
    # every window spans 16 patch columns (8 merged) except the ragged last one
    for w in range(6):
        toks = lay.row_of_slot[lay.segment == w]
        cols = lay.pos_rc[toks, 1]
        assert cols.min() == 16 * w and cols.max() == min(16 * w + 15, 91)


def test_qwen3_constants_match_pages():
    g = GOLDEN["qwen3_geometry"]["value"]
    assert (WL.QWEN3_N_Q_HEADS, WL.QWEN3_N_KV_HEADS, WL.QWEN3_HEAD_DIM, WL.QWEN3_HIDDEN,
            WL.QWEN3_LAYERS, WL.QWEN3_VOCAB) == (g["n_q_heads"], g["n_kv_heads"], g["head_dim"],
                                                g["hidden"], g["layers"], g["vocab"])
    assert WL.QWEN3_ROPE_THETA == g["rope_theta"] and WL.QWEN3_RMS_EPS == g["rms_eps"]
    assert GOLDEN["xdrope"]["value"]["effective_base"] == WL.XDROPE_BASE
    assert tuple(GOLDEN["xdrope"]["value"]["sections"]) == WL.XDROPE_SECTIONS


# ----------------------------------------------------------------------------
# speculative-decoding verify block (HunyuanOCR v1.5 port, section 3.8)
# ----------------------------------------------------------------------------
def test_verify_block_equals_prefill_rows_and_decode():
    """Row i of a k-token verify block is row L-k+i of a causal prefill over the same L slots;
    a 1-token block is a decode step."""
    rng = np.random.default_rng(11)
    L, k, Hq, Hkv, D = 23, 5, 4, 2, 8
    q_all = rng.standard_normal((L, Hq, D))
    ck = rng.standard_normal((Hkv, L + 3, D))
    cv = rng.standard_normal((Hkv, L + 3, D))
    pre = O.prefill(q_all, ck, cv, L, "causal")
    ver = O.verify_block(q_all[L - k:], ck, cv, L)
    np.testing.assert_allclose(ver, pre[L - k:], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(O.verify_block(q_all[L - 1:], ck, cv, L)[0], O.decode(q_all[L - 1], ck, cv, L),
                               rtol=1e-13, atol=1e-15)


def test_verify_block_brute_force_tiny():
    """L = 3, k = 2, one head, D = 2: row 0 sees keys 0..1, row 1 sees keys 0..2 (scalar sums)."""
    q = np.array([[[0.3, -1.2]], [[0.7, 0.4]]])
    K = np.array([[[1.0, 0.0], [0.5, -0.5], [-1.0, 2.0]]])
    V = np.array([[[1.0, 2.0], [3.0, -1.0], [0.0, 4.0]]])
    got = O.verify_block(q, K, V, 3)
    for i, n_keys in ((0, 2), (1, 3)):
        logits = [(q[i, 0, 0] * K[0, j, 0] + q[i, 0, 1] * K[0, j, 1]) / math.sqrt(2) for j in range(n_keys)]
        w = [math.exp(x) for x in logits]
        tot = math.fsum(w)
        for d in range(2):
            assert abs(got[i, 0, d] - math.fsum(w[j] * V[0, j, d] for j in range(n_keys)) / tot) < 1e-14


def test_verify_accept_hand_cases():
    # block = [current, c1, c2, c3]; posterior[i] is the target's id after block[i]
    assert O.verify_accept([5, 7, 9, 2], [1, 5, 7, 3], 40) == (2, 9, 39)      # c1, c2 accepted, c3 corrected
    assert O.verify_accept([5, 7, 3, 8], [1, 5, 7, 3], 40) == (3, 8, 40)      # all accepted, next token 8
    assert O.verify_accept([6, 7, 3, 8], [1, 5, 7, 3], 40) == (0, 6, 37)      # first candidate rejected
    assert O.verify_accept([4], [1], 17) == (0, 4, 17)                        # k = 1: a greedy decode step


def test_verify_accept_is_lossless_for_greedy():
    """Over many blocks with random drafts, the emitted tokens equal the target's own greedy
    sequence and the committed length counts exactly the tokens whose K/V stay cached."""
    rng = np.random.default_rng(3)
    vocab = 13
    nxt = rng.integers(0, vocab, size=vocab)          # a deterministic toy target: greedy id after t
    for _ in range(200):
        t0 = int(rng.integers(vocab))
        t, length, emitted = t0, 10, []
        for _ in range(6):
            k = int(rng.integers(1, 7))
            draft = [t]
            for _ in range(k - 1):                     # drafts: the true continuation, sometimes wrong
                draft.append(int(nxt[draft[-1]]) if rng.random() < 0.7 else int(rng.integers(vocab)))
            posterior = [int(nxt[x]) for x in draft]
            a, new_t, committed = O.verify_accept(posterior, draft, length + k)   # block appended
            emitted += draft[1:a + 1] + [new_t]
            assert committed == length + 1 + a         # current token + accepted candidates
            t, length = new_t, committed
        chain = [int(nxt[t0])]
        while len(chain) < len(emitted):
            chain.append(int(nxt[chain[-1]]))
        assert emitted == chain


# ----------------------------------------------------------------------------
# final RMSNorm + lm_head top-k
# ----------------------------------------------------------------------------
def test_topk_hand_ties_and_order():
    z = np.array([0.5, 2.0, -1.0, 2.0, 0.5, 3.0, 0.5])
    ids, vals = O.topk_lowest(z, 5)
    assert ids.tolist() == [5, 1, 3, 0, 4]             # 3.0; 2.0 twice (lower id first); 0.5 x3 -> 0, 4
    assert vals.tolist() == [3.0, 2.0, 2.0, 0.5, 0.5]
    # brute force: repeatedly take the first maximum and remove it
    rng = np.random.default_rng(2)
    for _ in range(50):
        z = rng.integers(-3, 4, size=40).astype(np.float64)   # many ties
        k = int(rng.integers(1, 12))
        rest, picked = list(range(40)), []
        for _ in range(k):
            best = max(rest, key=lambda v: (z[v], -v))
            picked.append(best); rest.remove(best)
        assert O.topk_lowest(z, k)[0].tolist() == picked


def test_lmhead_topk_top1_is_argmax_and_norm_is_scale_invariant():
    rng = np.random.default_rng(4)
    H, V = 64, 300
    W = WL.f32_to_bf16_bits((0.02 * rng.standard_normal((V, H))).astype(np.float32))
    h = rng.standard_normal((3, H))
    ids1, vals1 = O.lmhead_topk(h, W, V, 1)
    a_ids, a_max, _ = O.lmhead_argmax(h, W, V)
    assert ids1[:, 0].tolist() == a_ids.tolist() and np.allclose(vals1[:, 0], a_max, rtol=0, atol=0)
    w = 1 + 0.1 * rng.standard_normal(H)
    ids_n, vals_n = O.lmhead_topk(h, W, V, 7, norm_w=w)
    ids_s, vals_s = O.lmhead_topk(5.0 * h, W, V, 7, norm_w=w)          # RMSNorm removes the scale
    assert ids_n.tolist() == ids_s.tolist()
    np.testing.assert_allclose(vals_n, vals_s, rtol=1e-6)
    # the norm is applied: equal to logits of the explicitly normalised rows
    hn = np.stack([O.rms_norm(r, w, 1e-6) for r in h])
    ref_ids, ref_vals = O.lmhead_topk(hn, W, V, 7)
    assert ids_n.tolist() == ref_ids.tolist()
    np.testing.assert_allclose(vals_n, ref_vals, rtol=1e-13)


# ----------------------------------------------------------------------------
# image span fully visible to its own rows (MNN llm_demo walkthrough, section 3.3)
# ----------------------------------------------------------------------------
def test_causal_segment_mask_reduces_and_spans():
    S = 30
    uniq = np.arange(S)
    assert np.array_equal(O.prefill_mask(S, "causal_segment", uniq), O.prefill_mask(S, "causal"))
    assert np.array_equal(O.prefill_mask(S, "causal_segment", np.zeros(S, int)), O.prefill_mask(S, "full"))
    seg = WL.image_span_segments(3, 2, 4, 5)           # 3 text, begin, 2x5 grid rows, end, 5 text
    m = O.prefill_mask(seg.size, "causal_segment", seg)
    g0, g1 = 4, 14
    for i in range(seg.size):
        vis = np.nonzero(m[i])[0]
        end = g1 if g0 <= i < g1 else i + 1            # a grid row sees the whole grid
        assert vis.tolist() == list(range(end)), i
    # text after the span sees the span (causally) but the begin marker does not see it
    assert m[g1 + 1, g0:g1].all() and not m[g0 - 1, g0:g1].any()


def test_causal_segment_prefill_equals_bidirectional_span_by_hand():
    """Span rows attend over [0, span end): equal to attend() with that explicit key range."""
    rng = np.random.default_rng(8)
    seg = WL.image_span_segments(2, 2, 2, 3)
    S, Hq, Hkv, D = seg.size, 2, 1, 4
    q = rng.standard_normal((S, Hq, D)); ck = rng.standard_normal((Hkv, S, D)); cv = rng.standard_normal((Hkv, S, D))
    out = O.prefill(q, ck, cv, S, "causal_segment", seg)
    for i in range(S):
        end = int(np.max(np.nonzero(seg == seg[i])[0])) + 1 if np.sum(seg == seg[i]) > 1 else i + 1
        allowed = np.zeros((1, S), bool); allowed[0, :end] = True
        np.testing.assert_allclose(out[i], O.attend(q[i:i + 1], ck, cv, allowed)[0], rtol=1e-13, atol=1e-15)


# ----------------------------------------------------------------------------
# interleaved RoPE (Youtu-VL-4B port, implementation difficulty 2)
# ----------------------------------------------------------------------------
def test_rope_interleaved_hand_example():
    """D = 4, base 100: output [a c0 - b s0, c c1 - d s1, b c0 + a s0, d c1 + c s1] for input
    [a, b, c, d] (pairs (a, b) and (c, d) rotated, results de-interleaved)."""
    a, b, c, d = 0.3, -1.1, 2.0, 0.7
    p = 5
    t0, t1 = p * 1.0, p * 100.0 ** -0.5
    got = O.rope_apply(np.array([[[a, b, c, d]]]), np.array([[p]]), O.Rope("interleaved", 100.0))[0, 0]
    ref = [a * math.cos(t0) - b * math.sin(t0), c * math.cos(t1) - d * math.sin(t1),
           b * math.cos(t0) + a * math.sin(t0), d * math.cos(t1) + c * math.sin(t1)]
    np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-15)


def test_rope_interleaved_matches_the_pages_matrix_form():
    """The page rewrites the step as two constant matrices: q_rot = (q @ P) * cos + (q @ PR) * sin
    with P the de-interleave permutation and PR = P @ R (R the rotate-half +-1 matrix)."""
    rng = np.random.default_rng(6)
    D, T = 64, 9
    P = np.zeros((D, D))
    for j in range(D // 2):
        P[2 * j, j] = 1.0                     # column j of the output takes x_{2j}
        P[2 * j + 1, D // 2 + j] = 1.0        # column D/2 + j takes x_{2j+1}
    R = np.zeros((D, D))                      # y @ R = rotate_half(y) = [-y2, y1]
    for j in range(D // 2):
        R[D // 2 + j, j] = -1.0
        R[j, D // 2 + j] = 1.0
    x = rng.standard_normal((T, 1, D))
    pos = rng.integers(0, 3000, size=(T, 1))
    inv = O.inv_freq(1e6, D)
    ang = np.concatenate([pos * inv[None, :], pos * inv[None, :]], axis=1)     # [T, D]
    ref = (x[:, 0] @ P) * np.cos(ang) + (x[:, 0] @ (P @ R)) * np.sin(ang)
    np.testing.assert_allclose(O.rope_apply(x, pos, O.Rope("interleaved", 1e6))[:, 0], ref, rtol=1e-12, atol=1e-13)


def test_rope_interleaved_pairs_position_zero_and_relative_property():
    rng = np.random.default_rng(12)
    D = 32
    x = rng.standard_normal((1, 1, D))
    rope = O.Rope("interleaved", 1e6)
    y0 = O.rope_apply(x, np.array([[0]]), rope)[0, 0]
    np.testing.assert_array_equal(y0, np.concatenate([x[0, 0, 0::2], x[0, 0, 1::2]]))   # pure de-interleave
    y = O.rope_apply(x, np.array([[777]]), rope)[0, 0]
    np.testing.assert_allclose(y[:D // 2] ** 2 + y[D // 2:] ** 2, x[0, 0, 0::2] ** 2 + x[0, 0, 1::2] ** 2, rtol=1e-13)
    q, k = rng.standard_normal((1, 1, D)), rng.standard_normal((1, 1, D))
    d1 = np.dot(O.rope_apply(q, np.array([[50]]), rope)[0, 0], O.rope_apply(k, np.array([[20]]), rope)[0, 0])
    d2 = np.dot(O.rope_apply(q, np.array([[1030]]), rope)[0, 0], O.rope_apply(k, np.array([[1000]]), rope)[0, 0])
    assert abs(d1 - d2) < 1e-10


# ----------------------------------------------------------------------------
# asymmetric MLA-expanded cache: K = 192 (the last 64 dims rotated, interleaved), V = 128
# (Youtu-VL-4B port, section 6 and implementation difficulty 2)
# ----------------------------------------------------------------------------
def _mla_rope():
    return O.Rope("interleaved", 1e6, rot_offset=128, rot_dim=64)


def test_rope_subrange_leaves_the_rest_and_matches_the_block_matrix():
    """The rotation acts on dims 128..191 only, with frequencies of a 64-wide head: the whole
    192-wide step is the block matrix diag(I_128, page form on 64) with P and PR = P @ R the
    64x64 permutation and +-1 matrices."""
    rng = np.random.default_rng(21)
    T, Dk, w = 7, 192, 64
    P = np.zeros((w, w))
    R = np.zeros((w, w))
    for j in range(w // 2):
        P[2 * j, j] = 1.0
        P[2 * j + 1, w // 2 + j] = 1.0
        R[w // 2 + j, j] = -1.0
        R[j, w // 2 + j] = 1.0
    x = rng.standard_normal((T, 1, Dk))
    pos = rng.integers(0, 5000, size=(T, 1))
    got = O.rope_apply(x, pos, _mla_rope())[:, 0]
    np.testing.assert_array_equal(got[:, :128], x[:, 0, :128])
    j = np.arange(w // 2)
    inv = 1e6 ** (-2.0 * j / w)                       # a 64-wide head, not a 192-wide one
    ang = np.concatenate([pos * inv[None, :], pos * inv[None, :]], axis=1)
    xr = x[:, 0, 128:]
    ref = (xr @ P) * np.cos(ang) + (xr @ (P @ R)) * np.sin(ang)
    np.testing.assert_allclose(got[:, 128:], ref, rtol=1e-12, atol=1e-13)


def test_rope_subrange_relative_property_over_the_whole_head():
    """q.k over all 192 dims depends on the positions only through their difference, and a
    zero-width shift of both leaves the score unchanged."""
    rng = np.random.default_rng(22)
    rope = _mla_rope()
    q, k = rng.standard_normal((1, 1, 192)), rng.standard_normal((1, 1, 192))
    s = [np.dot(O.rope_apply(q, np.array([[m]]), rope)[0, 0], O.rope_apply(k, np.array([[n]]), rope)[0, 0])
         for m, n in ((70, 3), (1067, 1000), (40067, 40000))]
    assert abs(s[0] - s[1]) < 1e-10 and abs(s[0] - s[2]) < 1e-9
    nope = np.dot(q[0, 0, :128], k[0, 0, :128])
    same = np.dot(O.rope_apply(q, np.array([[9]]), rope)[0, 0], O.rope_apply(k, np.array([[9]]), rope)[0, 0])
    np.testing.assert_allclose(same, np.dot(q[0, 0], k[0, 0]), rtol=1e-12)
    assert abs(nope - np.dot(q[0, 0, :128], k[0, 0, :128])) == 0.0


def test_asymmetric_attention_two_keys_scale_follows_the_key_width():
    """Two keys whose logits differ by d: the output is sigmoid(d / sqrt(192)) V0 + (1 - ...) V1,
    with V 128 wide; the default scale uses the key width (192), not the value width."""
    rng = np.random.default_rng(23)
    q = rng.standard_normal((1, 1, 192))
    K = rng.standard_normal((1, 2, 192))
    V = rng.standard_normal((1, 2, 128))
    d = float(q[0, 0] @ (K[0, 0] - K[0, 1]))
    p0 = 1.0 / (1.0 + math.exp(-d / math.sqrt(192)))
    got = O.attend(q, K, V, np.ones((1, 2), bool))[0, 0]
    assert got.shape == (128,)
    np.testing.assert_allclose(got, p0 * V[0, 0] + (1 - p0) * V[0, 1], rtol=1e-13, atol=1e-14)


def test_asymmetric_attention_value_columns_are_independent():
    """Splitting V [.., 128] into two 64-wide halves and attending with each gives the two halves
    of the full result (the softmax weights see only K); the same for the decode and prefill forms."""
    rng = np.random.default_rng(24)
    H, W, S = 3, 40, 40
    q = rng.standard_normal((S, H, 192))
    K = rng.standard_normal((H, W, 192))
    V = rng.standard_normal((H, W, 128))
    full = O.prefill(q, K, V, S, "causal")
    a = O.prefill(q, K, V[..., :64], S, "causal")
    b = O.prefill(q, K, V[..., 64:], S, "causal")
    np.testing.assert_allclose(full, np.concatenate([a, b], axis=-1), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(O.decode(q[S - 1], K, V, S), full[S - 1], rtol=1e-12, atol=1e-14)


def test_cache_append_asymmetric_shapes():
    """An append into K [H, W, 192] / V [H, W, 128] without QK-Norm: K gets the sub-range rotation
    and bf16 rounding, V is stored unchanged, other slots stay untouched."""
    rng = np.random.default_rng(25)
    H, W, T = 4, 16, 3
    q = rng.standard_normal((T, H, 192))
    k = rng.standard_normal((T, H, 192))
    v = rng.standard_normal((T, H, 128))
    pos = np.array([[5], [6], [11]])
    slot = np.array([2, 3, 9])
    ck, cv = np.full((H, W, 192), 7.0), np.full((H, W, 128), 7.0)
    qr = O.cache_append(q, k, v, pos, slot, None, None, 1e-6, _mla_rope(), False, ck, cv, "bf16")
    np.testing.assert_array_equal(qr[..., :128], q[..., :128])
    for t in range(T):
        np.testing.assert_array_equal(ck[:, slot[t], :128], O.bf16_round(k[t, :, :128]))
        np.testing.assert_array_equal(cv[:, slot[t]], O.bf16_round(v[t]))
    rest = np.setdiff1d(np.arange(W), slot)
    assert np.all(ck[:, rest] == 7.0) and np.all(cv[:, rest] == 7.0)
