"""kv_attn_decode_static: decode attention for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: a host framework that owns every device
allocation, or a hot loop that must never reach an allocator.  kv_attn_decode_static runs
the same split-KV decode with its scratch in a fixed array inside the library's device
image.  These tests call it through the C ABI and check that two calls in a row agree with
kv_attn_decode (which takes a caller workspace) on the same inputs.

This file is named so that pytest collects it last.
"""
import ctypes as C

import numpy as np
import pytest

from helpers import FP32_ROW_REL, host, row_rel_err


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


@pytest.mark.gpu
@pytest.mark.parametrize("B,W,lens", [
    (28, 1024, None),                                   # 28 layer instances, lengths 513..540
    (5, 33000, [1, 700, 4097, 20000, 32896]),            # long contexts: several chunks each
])
def test_static_decode_matches_workspace_decode_twice(K, B, W, lens):
    import torch
    g = torch.Generator(device="cuda"); g.manual_seed(B)
    Hkv, Hq, D = 8, 16, 128
    kc = torch.randn((B, Hkv, W, D), device="cuda", generator=g).to(torch.bfloat16)
    vc = torch.randn((B, Hkv, W, D), device="cuda", generator=g).to(torch.bfloat16)
    cache = K.KVCache(kc, vc)
    lengths = np.asarray(lens if lens is not None else 513 + np.arange(B), np.int32)
    lengths_d = torch.from_numpy(lengths).cuda()
    ws = torch.zeros(K.decode_workspace_bytes(B, Hkv, Hq, W, D), dtype=torch.uint8, device="cuda")
    for call in range(2):                                # two calls in a row, different queries
        q = torch.randn((B, Hq, D), device="cuda", generator=g).to(torch.bfloat16)
        ref = torch.empty((B, Hq, D), device="cuda")
        K.kv_attn_decode(q, cache, lengths_d, lengths, ref, ws)
        out = torch.full((B, Hq, D), float("nan"), device="cuda")
        st = _call_static(K, q, cache, lengths_d, lengths, out)
        assert st == 0, K.lib().kva_last_error()
        torch.cuda.synchronize()
        err = row_rel_err(host(out), host(ref))
        assert err <= FP32_ROW_REL, f"call {call}: static decode differs from workspace decode ({err:.3e})"


def test_static_decode_rejects_batches_beyond_its_scratch(K):
    """B * Hq partials that cannot fit the fixed scratch are refused before any launch."""
    B, Hq = 600, 16                                      # 600*16*(128+2)*4 bytes > 4 MiB
    fake = 1 << 20
    cache = K.kv_attn._Cache(fake, fake, 1, 8, 128, 64, 8 * 64 * 128)
    lh = np.ones(B, np.int32)
    st = K.lib().kv_attn_decode_static(fake, 1, cache, fake, lh.ctypes.data, B, Hq, C.c_float(0.0), fake, None)
    assert st == K.kv_attn.KVA_EWORKSPACE
    assert b"4 MiB" in K.lib().kva_last_error()
