"""kv_attn_decode_static: decode attention for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: a host framework that owns every device
allocation, or a hot loop that must never reach an allocator.  kv_attn_decode_static runs
the same split-KV decode with its scratch in a fixed array inside the library's device
image.  These tests call it through the C ABI and check that
  * two calls in a row agree with kv_attn_decode (which takes a caller workspace) on the same
    inputs, including batches whose planned chunks do not fit the fixed scratch (the call then
    widens its chunks) and an fp32 cache;
  * its output matches the CPU oracle on sampled (instance, KV head) pairs of long contexts;
  * a warm call leaves the device's free memory and torch's allocator statistics unchanged.

This file is named so that pytest collects it last.
"""
import ctypes as C

import numpy as np
import pytest

import oracle as O
from helpers import FP32_ROW_REL, assert_bf16_close, host, row_rel_err


@pytest.fixture(scope="module")
def K():
    from kv_cache_gqa_gb300 import build
    build.build_library(verbose=False)
    import kv_cache_gqa_gb300 as K
    return K


def _call_static(K, q, cache, lengths_d, lengths_h, out):
    import torch
    lh = np.ascontiguousarray(lengths_h, np.int32)
    return K.lib().kv_attn_decode_static(
        q.data_ptr(), 1 if q.dtype == torch.bfloat16 else 0, cache.struct, lengths_d.data_ptr(), lh.ctypes.data,
        q.shape[0], q.shape[1], C.c_float(0.0), out.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _lengths(B, lens):
    if isinstance(lens, tuple):                          # (lo, hi): seeded uniform integers
        return np.random.default_rng(B).integers(lens[0], lens[1] + 1, size=B).astype(np.int32)
    return np.asarray(lens if lens is not None else 513 + np.arange(B), np.int32)


@pytest.mark.gpu
@pytest.mark.parametrize("B,W,lens,dt", [
    (28, 1024, None, "bf16"),                           # 28 layer instances, lengths 513..540
    (5, 33000, [1, 700, 4097, 20000, 32896], "bf16"),    # long contexts: several chunks each
    (64, 8192, (1024, 8192), "bf16"),                   # the planned 10 chunks exceed the 7 that fit
    (64, 4096, (1024, 4096), "f32"),                    # fp32 cache; 11 planned chunks, 7 fit
])
def test_static_decode_matches_workspace_decode_twice(K, B, W, lens, dt):
    import torch
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    g = torch.Generator(device="cuda"); g.manual_seed(B)
    Hkv, Hq, D = 8, 16, 128
    kc = torch.randn((B, Hkv, W, D), device="cuda", generator=g).to(tdt)
    vc = torch.randn((B, Hkv, W, D), device="cuda", generator=g).to(tdt)
    cache = K.KVCache(kc, vc)
    lengths = _lengths(B, lens)
    lengths_d = torch.from_numpy(lengths).cuda()
    ws = torch.zeros(K.decode_workspace_bytes(B, Hkv, Hq, W, D), dtype=torch.uint8, device="cuda")
    for call in range(2):                                # two calls in a row, different queries
        q = torch.randn((B, Hq, D), device="cuda", generator=g).to(tdt)
        ref = torch.empty((B, Hq, D), device="cuda")
        K.kv_attn_decode(q, cache, lengths_d, lengths, ref, ws)
        out = torch.full((B, Hq, D), float("nan"), device="cuda")
        st = _call_static(K, q, cache, lengths_d, lengths, out)
        assert st == 0, K.lib().kva_last_error()
        torch.cuda.synchronize()
        if dt == "f32":
            err = row_rel_err(host(out), host(ref))
            assert err <= FP32_ROW_REL, f"call {call}: static decode differs from workspace decode ({err:.3e})"
        else:
            # a widened plan cuts the keys into other chunks, so the bf16 probabilities the
            # tensor-core kernel rounds differ: the bf16-cache tolerance applies
            assert_bf16_close(host(out), host(ref), f"call {call}: static vs workspace decode")


@pytest.mark.gpu
def test_static_decode_matches_the_oracle_on_long_contexts(K):
    """Sampled (instance, KV head) pairs of a 5-instance batch with contexts up to 32896 keys,
    compared with the oracle's decode (softmax over the first L keys) at the bf16 tolerances."""
    import torch
    B, Hkv, Hq, D, W = 5, 8, 16, 128, 33000
    G = Hq // Hkv
    g = torch.Generator(device="cuda"); g.manual_seed(17)
    kc = torch.randn((B, Hkv, W, D), device="cuda", generator=g).to(torch.bfloat16)
    vc = torch.randn((B, Hkv, W, D), device="cuda", generator=g).to(torch.bfloat16)
    lengths = np.array([1, 700, 4097, 20000, 32896], np.int32)
    lengths_d = torch.from_numpy(lengths).cuda()
    cache = K.KVCache(kc, vc)
    for call in range(2):
        q = torch.randn((B, Hq, D), device="cuda", generator=g).to(torch.bfloat16)
        out = torch.full((B, Hq, D), float("nan"), device="cuda")
        assert _call_static(K, q, cache, lengths_d, lengths, out) == 0, K.lib().kva_last_error()
        torch.cuda.synchronize()
        got, qh = host(out), host(q)
        for b, kv in ((0, 0), (1, 7), (2, 3), (3, 5), (4, 0), (4, 6)):
            L = int(lengths[b])
            ck = host(kc[b, kv:kv + 1, :L])
            cv = host(vc[b, kv:kv + 1, :L])
            ref = O.decode(qh[b, kv * G:(kv + 1) * G], ck, cv, L)
            assert_bf16_close(got[b, kv * G:(kv + 1) * G], ref, f"call {call} instance {b} kv head {kv}")


@pytest.mark.gpu
def test_static_decode_warm_call_allocates_nothing(K):
    """After a first call on the device, a call changes neither the device's free memory
    (cudaMemGetInfo) nor torch's allocator statistics."""
    import torch
    B, Hkv, Hq, D, W = 28, 8, 16, 128, 1024
    g = torch.Generator(device="cuda"); g.manual_seed(3)
    kc = torch.randn((B, Hkv, W, D), device="cuda", generator=g).to(torch.bfloat16)
    vc = torch.randn((B, Hkv, W, D), device="cuda", generator=g).to(torch.bfloat16)
    q = torch.randn((B, Hq, D), device="cuda", generator=g).to(torch.bfloat16)
    lengths = (513 + np.arange(B)).astype(np.int32)
    lengths_d = torch.from_numpy(lengths).cuda()
    out = torch.empty((B, Hq, D), device="cuda")
    cache = K.KVCache(kc, vc)
    assert _call_static(K, q, cache, lengths_d, lengths, out) == 0, K.lib().kva_last_error()   # warm-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0, reserved0 = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    for _ in range(3):
        assert _call_static(K, q, cache, lengths_d, lengths, out) == 0, K.lib().kva_last_error()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes across warm calls"
    assert torch.cuda.memory_allocated() == alloc0 and torch.cuda.memory_reserved() == reserved0


def test_static_decode_rejects_batches_beyond_its_scratch(K):
    """B * Hq partials that cannot fit the fixed scratch are refused before any launch."""
    B, Hq = 600, 16                                      # 600*16*(128+2)*4 bytes > 4 MiB
    fake = 1 << 20
    cache = K.kv_attn._Cache(fake, fake, 1, 8, 128, 64, 8 * 64 * 128)
    lh = np.ones(B, np.int32)
    st = K.lib().kv_attn_decode_static(fake, 1, cache, fake, lh.ctypes.data, B, Hq, C.c_float(0.0), fake, None)
    assert st == K.kv_attn.KVA_EWORKSPACE
    assert b"4 MiB" in K.lib().kva_last_error()
