"""GPU parity of the speculative-decoding verify block (kv_attn_verify) and its commit
(kv_verify_commit) against the CPU oracle (verify_block, verify_accept): ragged lengths with NaN
canaries past the valid prefix, block sizes 1..33 over one to five 16-row tiles, group sizes
1/2/4, long contexts split into chunks, and a block of one token against kv_attn_decode."""
import zlib

import numpy as np
import pytest

import oracle as O
from helpers import assert_bf16_close, dev, host

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


@pytest.mark.parametrize("k,G,q_dt", [(1, 2, "bf16"), (2, 2, "bf16"), (5, 2, "f32"), (8, 2, "bf16"),
                                      (16, 2, "bf16"), (17, 2, "f32"), (3, 1, "bf16"), (16, 1, "bf16"),
                                      (4, 4, "bf16"), (7, 4, "f32"), (32, 2, "bf16"), (33, 2, "f32")])
def test_verify_parity(K, k, G, q_dt):
    torch = _torch()
    rng = np.random.default_rng(zlib.crc32(repr(("verify", k, G, q_dt)).encode()))
    Hkv, D = 2, 128
    Hq = Hkv * G
    lengths = np.array([k, k + 1, 40, 129, 700, 4111], np.int32)
    B, W = lengths.size, 4200
    q = O.store(rng.standard_normal((B, k, Hq, D)), q_dt)
    kc = O.store(rng.standard_normal((B, Hkv, W, D)), "bf16")
    vc = O.store(rng.standard_normal((B, Hkv, W, D)), "bf16")
    kd, vd = dev(kc, torch.bfloat16), dev(vc, torch.bfloat16)
    for b, L in enumerate(lengths):                    # canaries past the valid prefix
        kd[b, :, L:] = float("nan"); vd[b, :, L:] = float("inf")
    tdt = torch.float32 if q_dt == "f32" else torch.bfloat16
    ws = torch.zeros(K.verify_workspace_bytes(B, Hkv, Hq, k, W, D), dtype=torch.uint8, device="cuda")
    for rep in range(2):                               # the second call reuses the self-clearing workspace
        out = torch.full((B, k, Hq, D), float("nan"), device="cuda")
        K.kv_attn_verify(dev(q, tdt), K.KVCache(kd, vd), dev(lengths), lengths, out, ws)
        torch.cuda.synchronize()
        got = host(out)
        assert np.all(np.isfinite(got))
        zero = K.lib().kva_decode_workspace_zero_bytes(B, Hkv * ((G * k + 15) // 16))
        assert int(ws[:zero].sum()) == 0
    for b, L in enumerate(lengths):
        ref = O.verify_block(O.store(q[b], "bf16"), kc[b], vc[b], int(L))
        assert_bf16_close(got[b].reshape(-1, D), ref.reshape(-1, D), f"verify b={b} L={L} k={k}")


def test_verify_benchmark_configuration(K):
    """The launch the benchmark times: 64 sequences x 2048 valid slots, 16-token blocks, 16/8 heads,
    bf16 queries (the tcgen05 form); sampled sequences against the oracle's verify block."""
    torch = _torch()
    B, Hkv, Hq, D, L, k = 64, 8, 16, 128, 2048, 16
    g = torch.Generator(device="cuda"); g.manual_seed(7)
    kc = torch.randn((B, Hkv, L, D), device="cuda", generator=g).to(torch.bfloat16)
    vc = torch.randn((B, Hkv, L, D), device="cuda", generator=g).to(torch.bfloat16)
    q = torch.randn((B, k, Hq, D), device="cuda", generator=g).to(torch.bfloat16)
    lengths = np.full(B, L, np.int32)
    ws = torch.zeros(K.verify_workspace_bytes(B, Hkv, Hq, k, L, D), dtype=torch.uint8, device="cuda")
    out = torch.full((B, k, Hq, D), float("nan"), device="cuda")
    K.kv_attn_verify(q, K.KVCache(kc, vc), dev(lengths), lengths, out, ws)
    torch.cuda.synchronize()
    got = host(out)
    assert np.all(np.isfinite(got))
    for b in (0, 1, 31, 63):
        ref = O.verify_block(host(q[b]), host(kc[b]), host(vc[b]), L)
        assert_bf16_close(got[b].reshape(-1, D), ref.reshape(-1, D), f"verify b={b}")


def test_verify_single_token_equals_decode(K):
    torch = _torch()
    rng = np.random.default_rng(5)
    B, Hkv, Hq, D, W = 4, 8, 16, 128, 1024
    lengths = np.array([1, 333, 1000, 517], np.int32)
    q = torch.from_numpy(rng.standard_normal((B, 1, Hq, D)).astype(np.float32)).cuda().to(torch.bfloat16)
    kc = torch.randn((B, Hkv, W, D), device="cuda").to(torch.bfloat16)
    vc = torch.randn((B, Hkv, W, D), device="cuda").to(torch.bfloat16)
    ws = torch.zeros(max(K.verify_workspace_bytes(B, Hkv, Hq, 1, W, D), K.decode_workspace_bytes(B, Hkv, Hq, W, D)),
                     dtype=torch.uint8, device="cuda")
    a = torch.empty((B, 1, Hq, D), device="cuda")
    d = torch.empty((B, Hq, D), device="cuda")
    K.kv_attn_verify(q, K.KVCache(kc, vc), dev(lengths), lengths, a, ws)
    K.kv_attn_decode(q[:, 0], K.KVCache(kc, vc), dev(lengths), lengths, d, ws)
    torch.cuda.synchronize()
    assert_bf16_close(host(a[:, 0]).reshape(-1, D), host(d).reshape(-1, D), "verify k=1 vs decode")


def test_verify_commit_matches_oracle(K):
    torch = _torch()
    rng = np.random.default_rng(9)
    B, k = 37, 9
    block = rng.integers(0, 50, size=(B, k)).astype(np.int32)
    post = rng.integers(0, 50, size=(B, k)).astype(np.int32)
    for b in range(B):                                 # plant matching prefixes of every length
        a = b % k
        post[b, :a] = block[b, 1:a + 1]
    lengths = rng.integers(k, 3000, size=B).astype(np.int32)
    ld = dev(lengths)
    acc = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    K.kv_verify_commit(dev(post), dev(block), ld, acc, nxt)
    torch.cuda.synchronize()
    for b in range(B):
        a, t, new_len = O.verify_accept(post[b], block[b], int(lengths[b]))
        assert int(acc[b]) == a and int(nxt[b]) == t and int(ld[b]) == new_len
