"""GPU parity of the whole hot path on the five synthetic workloads at their full sizes, against
the CPU oracle on identical seeded inputs.  The Qwen3-shaped and the batched serving workloads
run twice: once through the fused decode-step call the benchmark times, in its launch
configuration (28 layer instances or 64 sequences per launch), and once through the separate
append and decode calls.
Where the oracle cannot cover every output at full size it checks sampled outputs (every
layer / head of sampled rows and steps, sampled sequences)."""
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


def _argmax_check(got_ids, z_cols, what):
    """got_ids [B]; z_cols [V, B] oracle logits: ids must match where the margin > 1e-3."""
    for b in range(z_cols.shape[1]):
        i, top, margin = O.argmax_lowest(z_cols[:, b])
        if margin > ARGMAX_MARGIN:
            assert int(got_ids[b]) == i, f"{what}: batch {b} id {got_ids[b]} != {i} (margin {margin:.2e})"
        else:
            assert z_cols[got_ids[b], b] >= top - ARGMAX_MARGIN


# ----------------------------------------------------------------------------
# 1. tiny fp32 single layer: prefill 64, 16 decode steps
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("fused", [True, False], ids=["decode_step", "append_then_decode"])
def test_tiny_fp32_prefill_decode(K, fused):
    """fused: each decode step is one kv_attn_decode_step launch (the CUDA-core form on the fp32
    cache), as the benchmark times it; otherwise an append and a decode."""
    torch = T()
    w = WL.tiny_fp32(0)
    Hq, Hkv, D, W = 16, 8, 128, w["capacity"]
    P = w["n_prefill"]
    kc = torch.zeros((1, Hkv, W, D), device="cuda"); vc = torch.zeros_like(kc)
    cache = K.KVCache(kc, vc)
    rope = K.Rope("1d", w["base"])
    qw, kw = dev(w["q_norm_w"]), dev(w["k_norm_w"])
    q_pre = torch.empty((1, P, Hq, D), device="cuda")
    slot = np.arange(P, dtype=np.int32)[None]
    K.kv_cache_append_rope_qknorm(dev(w["q"][None, :P]), dev(w["k"][None, :P]), dev(w["v"][None, :P]),
                                  dev(w["pos"][None, :P]), dev(slot), slot, cache, q_pre, rope,
                                  q_norm_w=qw, k_norm_w=kw, eps=w["eps"])
    out_pre = torch.empty((1, P, Hq, D), device="cuda")
    K.kv_attn_prefill(q_pre, cache, out_pre, mask="causal")
    ws = torch.zeros(K.decode_workspace_bytes(1, Hkv, Hq, W, D), dtype=torch.uint8, device="cuda")
    dec = []
    for t in range(P, W):
        qd = torch.empty((1, 1, Hq, D), device="cuda")
        s = np.array([[t]], np.int32)
        o = torch.empty((1, Hq, D), device="cuda")
        L = np.array([t + 1], np.int32)
        if fused:
            K.kv_attn_decode_step(dev(w["q"][t:t + 1]), dev(w["k"][t:t + 1]), dev(w["v"][t:t + 1]),
                                  dev(w["pos"][t:t + 1]), cache, dev(L), L, o, ws, rope, q_norm_w=qw, k_norm_w=kw,
                                  eps=w["eps"])
        else:
            K.kv_cache_append_rope_qknorm(dev(w["q"][None, t:t + 1]), dev(w["k"][None, t:t + 1]),
                                          dev(w["v"][None, t:t + 1]), dev(w["pos"][None, t:t + 1]), dev(s), s,
                                          cache, qd, rope, q_norm_w=qw, k_norm_w=kw, eps=w["eps"])
            K.kv_attn_decode(qd[:, 0], cache, dev(L), L, o, ws)
        dec.append(o)
    torch.cuda.synchronize()

    ck = np.zeros((Hkv, W, D)); cv = np.zeros((Hkv, W, D))
    qr = O.cache_append(w["q"], w["k"], w["v"], w["pos"], np.arange(W), w["q_norm_w"], w["k_norm_w"],
                        w["eps"], O.Rope("1d", w["base"]), False, ck, cv, "f32")
    assert_fp32_close(host(q_pre[0]), qr[:P], "q after norm+rope")
    assert_fp32_close(host(kc[0]), ck, "k cache")
    ref_pre = O.prefill(qr[:P], ck, cv, P, "causal")
    assert_fp32_close(host(out_pre[0]), ref_pre, "prefill")
    for i, t in enumerate(range(P, W)):
        assert_fp32_close(host(dec[i][0]), O.decode(qr[t], ck, cv, t + 1), f"decode t={t}")

    # decode == prefill: a full 80-token parallel prefill over the same cache
    q_all = torch.empty((1, W, Hq, D), device="cuda")
    kc2 = torch.zeros_like(kc); vc2 = torch.zeros_like(vc)
    slot = np.arange(W, dtype=np.int32)[None]
    K.kv_cache_append_rope_qknorm(dev(w["q"][None]), dev(w["k"][None]), dev(w["v"][None]), dev(w["pos"][None]),
                                  dev(slot), slot, K.KVCache(kc2, vc2), q_all, rope, q_norm_w=qw, k_norm_w=kw,
                                  eps=w["eps"])
    out_all = torch.empty((1, W, Hq, D), device="cuda")
    K.kv_attn_prefill(q_all, K.KVCache(kc2, vc2), out_all, mask="causal")
    torch.cuda.synchronize()
    for i, t in enumerate(range(P, W)):
        assert row_rel_err(host(dec[i][0]), host(out_all[0, t])) <= 1e-5


# ----------------------------------------------------------------------------
# 2. Qwen3-0.6B-shaped: 28 layers, 512 prefill, 256 decode steps, lm_head every step
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("fused", [True, False], ids=["decode_step", "append_then_decode"])
def test_qwen3_28_layers_full(K, fused):
    """fused: each decode step is one kv_attn_decode_step launch over the 28 layer caches, with
    the benchmark's arguments (raw fp32 projections, one shared position id, per-layer norm
    weights); otherwise the append and the decode are separate calls."""
    torch = T()
    w = WL.qwen3_layers(0)
    NL, P, S_dec, W = 28, w["prompt"], w["steps"], w["capacity"]
    Hq, Hkv, D = 16, 8, 128
    kc = torch.zeros((NL, Hkv, W, D), device="cuda", dtype=torch.bfloat16); vc = torch.zeros_like(kc)
    cache = K.KVCache(kc, vc)
    rope = K.Rope("1d", w["base"])
    qw, kw = dev(w["q_norm_w"]), dev(w["k_norm_w"])
    slot = np.arange(P, dtype=np.int32)[None]
    pos = np.arange(P, dtype=np.int32)[None, :, None]
    q_pre = torch.empty((NL, P, Hq, D), device="cuda", dtype=torch.bfloat16)
    K.kv_cache_append_rope_qknorm(dev(w["q"]), dev(w["k"]), dev(w["v"]), dev(pos), dev(slot), slot, cache, q_pre,
                                  rope, q_norm_w=qw, k_norm_w=kw, eps=w["eps"], norm_inst_stride=D)
    out_pre = torch.empty((NL, P, Hq, D), device="cuda")
    K.kv_attn_prefill(q_pre, cache, out_pre, mask="causal")

    Wlm = WL.lm_head_weights(1)
    Wd = dev(Wlm)
    hs = WL.hidden_states(2, S_dec + 1)
    lm_ws = torch.zeros(K.lmhead_workspace_bytes(1, 1024), dtype=torch.uint8, device="cuda")
    dec_ws = torch.zeros(K.decode_workspace_bytes(NL, Hkv, Hq, W, D), dtype=torch.uint8, device="cuda")
    ids = torch.empty((S_dec + 1,), dtype=torch.int32, device="cuda")
    K.lmhead_argmax(dev(hs[0]), Wd, ids[0:1], lm_ws)
    sample_steps = (0, 1, 128, 255)
    dec_out = {}
    for s in range(S_dec):
        t = P + s
        qd = torch.empty((NL, 1, Hq, D), device="cuda", dtype=torch.bfloat16)
        sl = np.array([[t]], np.int32)
        o = torch.empty((NL, Hq, D), device="cuda")
        L = np.full(NL, t + 1, np.int32)
        if fused:
            K.kv_attn_decode_step(dev(w["dq"][s]), dev(w["dk"][s]), dev(w["dv"][s]), dev(sl), cache, dev(L), L, o,
                                  dec_ws, rope, q_norm_w=qw, k_norm_w=kw, eps=w["eps"], norm_inst_stride=D,
                                  q_out=qd[:, 0])
        else:
            K.kv_cache_append_rope_qknorm(dev(w["dq"][s][:, None]), dev(w["dk"][s][:, None]),
                                          dev(w["dv"][s][:, None]), dev(sl[:, :, None]), dev(sl), sl, cache, qd, rope,
                                          q_norm_w=qw, k_norm_w=kw, eps=w["eps"], norm_inst_stride=D)
            K.kv_attn_decode(qd[:, 0], cache, dev(L), L, o, dec_ws)
        if s in sample_steps:
            dec_out[s] = (o, qd)
        K.lmhead_argmax(dev(hs[s + 1]), Wd, ids[s + 1:s + 2], lm_ws)
    torch.cuda.synchronize()

    rope_o = O.Rope("1d", w["base"])
    rows = np.array([0, 1, 2, 63, 64, 127, 128, 255, 256, 383, 384, 510, 511])
    kc_bits = bf16_bits(kc)
    for n in range(NL):
        ck = np.zeros((Hkv, W, D), np.float32); cv = np.zeros((Hkv, W, D), np.float32)
        qr = O.cache_append(w["q"][n], w["k"][n], w["v"][n], np.arange(P)[:, None], np.arange(P),
                            w["q_norm_w"][n], w["k_norm_w"][n], w["eps"], rope_o, False, ck, cv, "bf16")
        assert_bf16_store(bf16_bits(q_pre[n]), qr, f"q layer {n}")
        qdec = []
        for s in range(S_dec):
            qdec.append(O.cache_append(w["dq"][s][n][None], w["dk"][s][n][None], w["dv"][s][n][None], [[P + s]],
                                       [P + s], w["q_norm_w"][n], w["k_norm_w"][n], w["eps"], rope_o, False,
                                       ck, cv, "bf16")[0])
        k_all = np.concatenate([w["k"][n], w["dk"][:, n]], axis=0)
        kr = O.qk_transform(k_all, np.arange(P + S_dec)[:, None], w["k_norm_w"][n], w["eps"], rope_o, False)
        assert_bf16_store(kc_bits[n][:, :P + S_dec], kr.transpose(1, 0, 2), f"k cache layer {n}")
        allowed = np.zeros((rows.size, W), bool)
        for a_i, r in enumerate(rows):
            allowed[a_i, :r + 1] = True
        ref = O.attend(qr[rows], ck, cv, allowed)
        assert_bf16_close(host(out_pre[n])[rows], ref, f"prefill layer {n}")
        for s, (o, qd) in dec_out.items():
            assert_bf16_close(host(o[n]), O.decode(qdec[s], ck, cv, P + s + 1), f"decode layer {n} step {s}")
            assert_bf16_store(bf16_bits(qd[n]), qdec[s][None], f"decode q layer {n} step {s}")
        # the V rows every step wrote (bit-exact: v is stored as given)
        np.testing.assert_array_equal(host(vc[n])[:, :P + S_dec], cv[:, :P + S_dec].astype(np.float64))

    got = ids.cpu().numpy()
    chk = [0, 1, 100, 256]
    z = O.lm_logits(hs[chk][:, 0, :].T, Wlm, WL.QWEN3_VOCAB)          # [V, len(chk)]
    _argmax_check(got[chk], z, "lm_head")


# ----------------------------------------------------------------------------
# 3. VLM image span: xdRoPE sections, norm after RoPE, causal, then 64 decode steps
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("fused", [True, False], ids=["decode_step", "append_then_decode"])
def test_image_span_xdrope(K, fused):
    """fused: the 64 decode steps through kv_attn_decode_step, as the benchmark times them."""
    torch = T()
    w = WL.image_span_prefill(0)
    S, W, steps = w["pos"].shape[0], w["capacity"], w["dq"].shape[0]
    Hq, Hkv, D = 16, 8, 128
    kc = torch.zeros((1, Hkv, W, D), device="cuda", dtype=torch.bfloat16); vc = torch.zeros_like(kc)
    cache = K.KVCache(kc, vc)
    rope = K.Rope("sections", w["base"], w["sections"])
    qw, kw = dev(w["q_norm_w"]), dev(w["k_norm_w"])
    slot = np.arange(S, dtype=np.int32)[None]
    q_pre = torch.empty((1, S, Hq, D), device="cuda", dtype=torch.bfloat16)
    K.kv_cache_append_rope_qknorm(dev(w["q"][None]), dev(w["k"][None]), dev(w["v"][None]), dev(w["pos"][None]),
                                  dev(slot), slot, cache, q_pre, rope, q_norm_w=qw, k_norm_w=kw, eps=w["eps"],
                                  norm_after_rope=True)
    out_pre = torch.empty((1, S, Hq, D), device="cuda")
    K.kv_attn_prefill(q_pre, cache, out_pre, mask="causal")
    ws = torch.zeros(K.decode_workspace_bytes(1, Hkv, Hq, W, D), dtype=torch.uint8, device="cuda")
    dec = []
    for s in range(steps):
        t = S + s
        qd = torch.empty((1, 1, Hq, D), device="cuda", dtype=torch.bfloat16)
        sl = np.array([[t]], np.int32)
        o = torch.empty((1, Hq, D), device="cuda")
        L = np.array([t + 1], np.int32)
        if fused:
            K.kv_attn_decode_step(dev(w["dq"][s:s + 1]), dev(w["dk"][s:s + 1]), dev(w["dv"][s:s + 1]),
                                  dev(w["dpos"][s:s + 1]), cache, dev(L), L, o, ws, rope, q_norm_w=qw, k_norm_w=kw,
                                  eps=w["eps"], norm_after_rope=True)
        else:
            K.kv_cache_append_rope_qknorm(dev(w["dq"][None, s:s + 1]), dev(w["dk"][None, s:s + 1]),
                                          dev(w["dv"][None, s:s + 1]), dev(w["dpos"][None, s:s + 1]), dev(sl), sl,
                                          cache, qd, rope, q_norm_w=qw, k_norm_w=kw, eps=w["eps"],
                                          norm_after_rope=True)
            K.kv_attn_decode(qd[:, 0], cache, dev(L), L, o, ws)
        dec.append(o)
    torch.cuda.synchronize()

    rope_o = O.Rope("sections", w["base"], w["sections"])
    ck = np.zeros((Hkv, W, D)); cv = np.zeros((Hkv, W, D))
    qr = O.cache_append(w["q"], w["k"], w["v"], w["pos"], np.arange(S), w["q_norm_w"], w["k_norm_w"], w["eps"],
                        rope_o, True, ck, cv, "bf16")
    qdr = O.cache_append(w["dq"], w["dk"], w["dv"], w["dpos"], np.arange(S, S + steps), w["q_norm_w"],
                         w["k_norm_w"], w["eps"], rope_o, True, ck, cv, "bf16")
    kr = O.qk_transform(np.concatenate([w["k"], w["dk"]]), np.concatenate([w["pos"], w["dpos"]]), w["k_norm_w"],
                        w["eps"], rope_o, True)
    assert_bf16_store(bf16_bits(kc[0])[:, :S + steps], kr.transpose(1, 0, 2), "k cache")
    assert_bf16_close(host(out_pre[0]), O.prefill(qr, ck, cv, S, "causal"), "image-span prefill")
    for s in range(steps):
        assert_bf16_close(host(dec[s][0]), O.decode(qdr[s], ck, cv, S + s + 1), f"decode step {s}")


# ----------------------------------------------------------------------------
# 4. vision windowed attention: 14x92 grid, D=72, 2D RoPE, window segments + full pass
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_vision_windowed(K, dt):
    torch = T()
    w = WL.vision_windowed(0)
    lay = w["layout"]
    S, H, D = lay.pos_rc.shape[0], 16, 72
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    kc = torch.zeros((1, H, S, D), device="cuda", dtype=tdt); vc = torch.zeros_like(kc)
    cache = K.KVCache(kc, vc)
    q_out = torch.empty((1, S, H, D), device="cuda", dtype=tdt)
    slot = lay.slot[None]
    K.kv_cache_append_rope_qknorm(dev(w["q"][None]), dev(w["k"][None]), dev(w["v"][None]), dev(lay.pos_rc[None]),
                                  dev(slot), slot, cache, q_out, K.Rope("2d", w["base"]))
    outs = {}
    for mask in ("segment", "full"):
        o = torch.empty((1, S, H, D), device="cuda")
        K.kv_attn_prefill(q_out, cache, o, mask=mask, segment=dev(lay.segment) if mask == "segment" else None,
                          segment_host=lay.segment if mask == "segment" else None, row_of_slot=dev(lay.row_of_slot))
        outs[mask] = o
    torch.cuda.synchronize()

    ck = np.zeros((H, S, D)); cv = np.zeros((H, S, D))
    qr = O.cache_append(w["q"], w["k"], w["v"], lay.pos_rc, lay.slot, None, None, 0.0, O.Rope("2d", w["base"]),
                        False, ck, cv, dt)
    q_slots = O.store(qr, dt)[lay.row_of_slot]          # the kernel reads q stored in the cache dtype
    for mask in ("segment", "full"):
        ref_slots = O.prefill(q_slots, ck, cv, S, mask, lay.segment)
        ref = np.empty_like(ref_slots); ref[lay.row_of_slot] = ref_slots
        got = host(outs[mask][0])
        if dt == "f32":
            assert_fp32_close(got, ref, f"vision {mask}")
        else:
            assert_bf16_close(got, ref, f"vision {mask}")


# ----------------------------------------------------------------------------
# 5. batched serving decode: B=64, contexts uniform in [1024, 32768], 128 steps
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("fused", [True, False], ids=["decode_step", "append_then_decode"])
def test_batched_serving_decode(K, fused):
    """fused: each step is one kv_attn_decode_step launch (the benchmark's serving step) with a
    position id per sequence; otherwise the append and the decode are separate calls."""
    torch = T()
    seed, B, steps = 0, 64, 128
    Hq, Hkv, D = 16, 8, 128
    ctx = WL.serving_contexts(seed, B)
    W = int(ctx.max()) + steps
    kc = torch.empty((B, Hkv, W, D), device="cuda", dtype=torch.bfloat16); vc = torch.empty_like(kc)
    g = torch.Generator(device="cuda"); g.manual_seed(1234)
    for b in range(B):
        kc[b, :, :ctx[b]] = torch.randn((Hkv, int(ctx[b]), D), device="cuda", generator=g).to(torch.bfloat16)
        vc[b, :, :ctx[b]] = torch.randn((Hkv, int(ctx[b]), D), device="cuda", generator=g).to(torch.bfloat16)
    sampled = sorted({0, 1, int(np.argmin(ctx)), int(np.argmax(ctx))})
    prefix = {}
    for b in sampled:
        kb, vb = WL.serving_prefix(seed, b, int(ctx[b]))
        prefix[b] = (kb, vb)
        kc[b, :, :ctx[b]] = dev(kb); vc[b, :, :ctx[b]] = dev(vb)
    cache = K.KVCache(kc, vc)
    qw_np, kw_np = WL.serving_norm_weights(seed)
    qw, kw = dev(qw_np), dev(kw_np)
    rope = K.Rope("1d", WL.QWEN3_ROPE_THETA)
    Wlm = WL.lm_head_weights(1)
    Wd = dev(Wlm)
    dec_ws = torch.zeros(K.decode_workspace_bytes(B, Hkv, Hq, W, D), dtype=torch.uint8, device="cuda")
    lm_ws = torch.zeros(K.lmhead_workspace_bytes(B, 1024), dtype=torch.uint8, device="cuda")
    sample_steps = (0, 1, 63, 127)
    lm_steps = (0, 127)
    outs, lm_ids, inputs = {}, {}, []
    for s in range(steps):
        x = WL.serving_step_inputs(seed, s, B)
        inputs.append(x)
        t = (ctx + s).astype(np.int32)
        qd = torch.empty((B, 1, Hq, D), device="cuda", dtype=torch.bfloat16)
        o = torch.empty((B, Hq, D), device="cuda")
        L = t + 1
        if fused:
            K.kv_attn_decode_step(dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(t[:, None]), cache, dev(L), L, o,
                                  dec_ws, rope, q_norm_w=qw, k_norm_w=kw, eps=WL.QWEN3_RMS_EPS)
        else:
            K.kv_cache_append_rope_qknorm(dev(x["q"][:, None]), dev(x["k"][:, None]), dev(x["v"][:, None]),
                                          dev(t[:, None, None]), dev(t[:, None]), t[:, None], cache, qd, rope,
                                          q_norm_w=qw, k_norm_w=kw, eps=WL.QWEN3_RMS_EPS)
            K.kv_attn_decode(qd[:, 0], cache, dev(L), L, o, dec_ws)
        ids = torch.empty((B,), dtype=torch.int32, device="cuda")
        K.lmhead_argmax(dev(x["h"]), Wd, ids, lm_ws)
        if s in sample_steps:
            outs[s] = o
        if s in lm_steps:
            lm_ids[s] = ids
    torch.cuda.synchronize()

    rope_o = O.Rope("1d", WL.QWEN3_ROPE_THETA)
    for b in sampled:
        ck = np.zeros((Hkv, W, D), np.float32); cv = np.zeros((Hkv, W, D), np.float32)
        ck[:, :ctx[b]] = WL.bf16_bits_to_f32(prefix[b][0]); cv[:, :ctx[b]] = WL.bf16_bits_to_f32(prefix[b][1])
        qs = []
        for s in range(steps):
            x = inputs[s]
            qs.append(O.cache_append(x["q"][b][None], x["k"][b][None], x["v"][b][None], [[ctx[b] + s]], [ctx[b] + s],
                                     qw_np, kw_np, WL.QWEN3_RMS_EPS, rope_o, False, ck, cv, "bf16")[0])
        kb_new = np.stack([inputs[s]["k"][b] for s in range(steps)])
        kr = O.qk_transform(kb_new, (ctx[b] + np.arange(steps))[:, None], kw_np, WL.QWEN3_RMS_EPS, rope_o, False)
        assert_bf16_store(bf16_bits(kc[b])[:, ctx[b]:ctx[b] + steps], kr.transpose(1, 0, 2), f"k cache b={b}")
        for s in sample_steps:
            ref = O.decode(qs[s], ck, cv, int(ctx[b]) + s + 1)
            assert_bf16_close(host(outs[s][b]), ref, f"serving b={b} step {s}")
    for s in lm_steps:
        z = O.lm_logits(inputs[s]["h"].T, Wlm, WL.QWEN3_VOCAB)          # [V, B]
        _argmax_check(lm_ids[s].cpu().numpy(), z, f"lm_head step {s}")
    # every sequence's output is finite (the unsampled ones included)
    for s, o in outs.items():
        assert torch.isfinite(o).all()
