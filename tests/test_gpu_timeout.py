"""Failure detection without a GPU fault: a kernel wait that nothing satisfies gives up after its
limit, the give-up is counted where the host can read it (kva_wait_timeouts), and the device
stays usable afterwards.  The normal kernels of a test session never give up."""
import numpy as np
import pytest

import oracle as O
from helpers import assert_bf16_close, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from kv_cache_gqa_gb300 import build
    build.build_library(verbose=False)
    import kv_cache_gqa_gb300 as K
    return K


def _small_decode(K, torch, seed):
    g = torch.Generator(device="cuda"); g.manual_seed(seed)
    B, Hkv, Hq, D, W = 3, 2, 4, 128, 300
    kc = torch.randn((B, Hkv, W, D), device="cuda", generator=g).to(torch.bfloat16)
    vc = torch.randn_like(kc)
    q = torch.randn((B, Hq, D), device="cuda", generator=g).to(torch.bfloat16)
    lengths = np.array([1, 150, 300], np.int32)
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    ws = torch.zeros(K.decode_workspace_bytes(B, Hkv, Hq, W, D), dtype=torch.uint8, device="cuda")
    K.kv_attn_decode(q, K.KVCache(kc, vc), torch.from_numpy(lengths).cuda(), lengths, out, ws)
    torch.cuda.synchronize()
    for b in range(B):
        ref = O.decode(host(q[b]), host(kc[b]), host(vc[b]), int(lengths[b]))
        assert_bf16_close(host(out[b]), ref, f"decode instance {b}")


def test_wait_timeout_is_counted_and_the_device_stays_usable(K):
    import torch
    torch.cuda.synchronize()
    assert K.wait_timeouts() == 0, "a kernel earlier in this process gave up a wait"
    _small_decode(K, torch, 1)
    assert K.wait_timeouts() == 0
    st = K.lib().kva_selftest_wait_timeout(torch.cuda.current_stream().cuda_stream)
    assert st == 0, K.lib().kva_last_error()
    torch.cuda.synchronize()                       # the wait gives up after about 2 s
    assert K.wait_timeouts() >= 1
    assert K.wait_timeouts(reset=True) >= 1
    assert K.wait_timeouts() == 0
    _small_decode(K, torch, 2)                     # kernels still run and match the oracle
    assert K.wait_timeouts() == 0
