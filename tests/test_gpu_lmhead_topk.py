"""GPU parity of lmhead_topk (final RMSNorm fused into the lm_head, k best ids) against the oracle
(lmhead_topk) on every lm_head path: batch 1 pipelined (H 1024/2048), batch 1 grid-stride (H 2560),
batched tensor-core (B 2..128) and the generic fp32-table kernel; top_k 1 (fused argmax) and
k > 1 (logits + row ranking); planted duplicate rows check the lower-id-first tie rule."""
import zlib

import numpy as np
import pytest

import oracle as O
import workloads as WL
from helpers import ARGMAX_MARGIN, dev

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


CASES = [
    # B, H, V, wdt, top_k, norm
    (1, 1024, 151936, "bf16", 1, True),
    (1, 1024, 151936, "bf16", 5, True),
    (1, 1024, 151936, "bf16", 8, True),     # the benchmark's final-norm top-8
    (1, 1024, 151936, "bf16", 32, False),
    (1, 2048, 40000, "bf16", 8, True),
    (1, 2560, 9001, "bf16", 1, True),
    (17, 2048, 3001, "bf16", 8, True),
    (64, 1024, 12000, "bf16", 4, True),
    (3, 1024, 2000, "f32", 3, True),
]


@pytest.mark.parametrize("B,H,V,wdt,k,norm", CASES)
def test_lmhead_topk_parity(K, B, H, V, wdt, k, norm):
    torch = _torch()
    rng = np.random.default_rng(zlib.crc32(repr(("topk", B, H, V, wdt, k, norm)).encode()))
    Wf = (0.02 * rng.standard_normal((V, H))).astype(np.float32)
    # planted ties: a few rows duplicated at higher ids, and the hidden vector biased toward them so
    # the duplicates land in the top ranks
    dup_src = rng.choice(V // 2, size=3, replace=False)
    dup_dst = V // 2 + rng.choice(V // 2, size=3, replace=False)
    Wf[dup_dst] = Wf[dup_src]
    h = rng.standard_normal((B, H)).astype(np.float32) * 2.0
    h += 3.0 * Wf[dup_src[0]] / np.linalg.norm(Wf[dup_src[0]]) * np.sqrt(H)
    w = (1 + 0.1 * rng.standard_normal(H)).astype(np.float32) if norm else None
    if wdt == "bf16":
        Wbits = WL.f32_to_bf16_bits(Wf)
        Wd = dev(Wbits)
        Wref = Wbits
    else:
        Wd = dev(Wf)
        Wref = Wf
    ids = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
    vals = torch.full((B, k), float("nan"), device="cuda")
    ws = torch.zeros(K.lmhead_topk_workspace_bytes(B, H, V, k), dtype=torch.uint8, device="cuda")
    for _ in range(2):                              # the second call checks the workspace was left clean
        K.lmhead_topk(dev(h), Wd, ids, ws, norm_w=dev(w) if norm else None, eps=1e-6, out_vals=vals)
        torch.cuda.synchronize()
    got_ids, got_vals = ids.cpu().numpy(), vals.cpu().numpy()
    ref_ids, ref_vals = O.lmhead_topk(h, Wref, V, k, norm_w=w, eps=1e-6)
    full_ids, full_vals = O.lmhead_topk(h, Wref, V, min(V, k + 1), norm_w=w, eps=1e-6)
    for b in range(B):
        np.testing.assert_allclose(got_vals[b], ref_vals[b], rtol=2e-5, atol=2e-5 * np.abs(ref_vals[b]).max())
        zs = full_vals[b]
        for r in range(k):
            gap_prev = zs[r - 1] - zs[r] if r > 0 else np.inf
            gap_next = zs[r] - zs[r + 1] if r + 1 < len(zs) else np.inf
            if min(gap_prev, gap_next) > ARGMAX_MARGIN:
                assert got_ids[b, r] == ref_ids[b, r], (b, r, got_ids[b], ref_ids[b])
        # exact ties (duplicated rows) rank the lower id first
        pos = {int(v): r for r, v in enumerate(got_ids[b])}
        for s_, d_ in zip(dup_src, dup_dst):
            if int(s_) in pos and int(d_) in pos:
                assert pos[int(s_)] < pos[int(d_)]
                assert got_vals[b, pos[int(s_)]] == got_vals[b, pos[int(d_)]]
        assert len(set(got_ids[b].tolist())) == k and got_ids[b].min() >= 0 and got_ids[b].max() < V
