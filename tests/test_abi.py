"""The C-ABI library loads, exports every function include/kv_attn.h declares, and its host-side
validation rejects bad arguments with the documented status before launching anything (these
calls never reach the GPU, so they run without one)."""
import ctypes as C
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def K():
    try:
        import torch
        if torch.cuda.is_available():
            # the calls below pass dummy device addresses; a validation gap must never reach a GPU
            pytest.skip("ABI validation tests run on hosts without a GPU")
    except ImportError:
        pass
    from kv_cache_gqa_gb300 import build
    build.build_library(verbose=False)
    import kv_cache_gqa_gb300.kv_attn as K
    K.lib()
    return K


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kv_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", src)) - {"sizeof"})


def test_exports_every_declared_symbol(K):
    names = declared_functions()
    assert {"kv_cache_append_rope_qknorm", "kv_attn_prefill", "kv_attn_decode", "lmhead_argmax"} <= set(names)
    for n in names:
        assert hasattr(K.lib(), n), f"libkv_attn.so does not export {n}"


def test_workspace_size_dispatcher_matches_the_per_call_sizers(K):
    L = K.lib()
    for B, Hkv, Hq, Lmax, D in ((1, 8, 16, 80, 128), (28, 8, 16, 768, 128), (64, 8, 16, 32896, 128),
                                (16, 32, 32, 512, 128), (3, 2, 8, 5000, 128)):
        want = L.kva_decode_workspace_size(B, Hkv, Hq, Lmax, D)
        assert want > 0 and K.workspace_bytes("decode", B=B, n_kv_heads=Hkv, n_q_heads=Hq, max_len=Lmax,
                                              head_dim=D) == want
        for k in (1, 4, 17):
            assert K.workspace_bytes("verify", B=B, n_kv_heads=Hkv, n_q_heads=Hq, max_len=Lmax, head_dim=D,
                                     block=k) == L.kva_verify_workspace_size(B, Hkv, Hq, k, Lmax, D) > 0
    for B, H, V in ((1, 1024, 151936), (64, 1024, 151936), (5, 512, 4099)):
        assert K.workspace_bytes("lmhead", B=B, hidden=H) == L.kva_lmhead_workspace_size(B, H) > 0
        for k in (1, 8):
            assert K.workspace_bytes("lmhead_topk", B=B, hidden=H, vocab=V, block=k) == \
                L.kva_lmhead_topk_workspace_size(B, H, V, k) > 0
    # an unknown kind, a NULL descriptor or a dimension that is not positive: 0
    assert L.kva_workspace_size(7, C.byref(K._WorkspaceDims(1, 8, 16, 80, 128, 1024, 100, 1))) == 0
    assert L.kva_workspace_size(0, None) == 0
    assert K.workspace_bytes("decode", B=0, n_kv_heads=8, n_q_heads=16, max_len=80, head_dim=128) == 0
    assert K.workspace_bytes("lmhead", B=2, hidden=0) == 0


def test_strerror_and_version(K):
    L = K.lib()
    for s in range(7):
        assert L.kva_strerror(s)
    assert L.kva_strerror(0) == b"ok"
    assert L.kva_version() >= 100
    assert L.kva_launch_count() >= 0


def _cache(ptr=16, dtype=1, hkv=8, d=128, cap=1024, stride=None, dv=0, stride_v=0):
    import kv_cache_gqa_gb300.kv_attn as K
    return K._Cache(ptr, ptr, dtype, hkv, d, cap, stride if stride is not None else hkv * cap * d, dv, stride_v)


def _rope(kind=1, base=1e6, secs=(0, 0, 0, 0), n_axes=1, rot_offset=0, rot_dim=0):
    import kv_cache_gqa_gb300.kv_attn as K
    return K._Rope(kind, n_axes, (C.c_int32 * 4)(*secs), base, rot_offset, rot_dim)


def _norm(q=0, k=0, eps=1e-6):
    import kv_cache_gqa_gb300.kv_attn as K
    return K._Norm(q or None, k or None, 0, eps, 0)


FAKE = 1 << 20   # a 16-byte aligned dummy address: never dereferenced, validation fails first


def append(K, *, N=1, T=1, Hq=16, slot_host=None, cache=None, rope=None, norm=None, q=FAKE, in_dtype=0):
    sh = np.zeros(max(1, N * T), np.int32) if slot_host is None else np.asarray(slot_host, np.int32)
    return K.lib().kv_cache_append_rope_qknorm(
        q, FAKE, FAKE, in_dtype, N, T, Hq, FAKE, 0, FAKE, T, sh.ctypes.data,
        norm or _norm(), rope or _rope(), FAKE, 1, cache or _cache(FAKE), None)


def test_append_validation(K):
    assert append(K, N=0) == K.KVA_OK and append(K, T=0) == K.KVA_OK        # empty: no-op
    assert append(K, N=-1) == K.KVA_EINVAL
    assert append(K, Hq=12) == K.KVA_EINVAL                                 # not a multiple of Hkv
    assert append(K, slot_host=[1024]) == K.KVA_ECAPACITY                   # beyond the window
    assert append(K, slot_host=[-1]) == K.KVA_ECAPACITY
    assert append(K, q=FAKE + 4) == K.KVA_EALIGN
    assert append(K, cache=_cache(FAKE, d=100)) == K.KVA_EALIGN              # D % 8
    assert append(K, cache=_cache(FAKE, d=264)) == K.KVA_EUNSUPPORTED        # D above 256
    assert append(K, rope=_rope(kind=2, secs=(16, 16, 16, 8), n_axes=4)) == K.KVA_EINVAL  # sum != D/2
    assert append(K, rope=_rope(kind=3, n_axes=1)) == K.KVA_EINVAL
    assert append(K, rope=_rope(kind=5)) == K.KVA_EINVAL
    assert append(K, rope=_rope(base=-1.0)) == K.KVA_EINVAL
    assert append(K, norm=_norm(q=FAKE)) == K.KVA_EINVAL                     # q weight without k weight
    assert append(K, cache=_cache(FAKE, stride=5), N=2, slot_host=[0, 0]) == K.KVA_EINVAL
    assert b"stride" in K.lib().kva_last_error()


def test_asymmetric_cache_and_rotary_range_validation(K):
    """K rows 192 wide, V rows 128 (MLA-expanded cache) and RoPE over a sub-range of the head."""
    asym = dict(hkv=32, d=192, dv=128, cap=512)
    assert append(K, rope=_rope(kind=4, rot_offset=128, rot_dim=63), Hq=32, cache=_cache(FAKE, **asym)) == K.KVA_EINVAL
    assert append(K, rope=_rope(kind=4, rot_offset=160, rot_dim=64), Hq=32, cache=_cache(FAKE, **asym)) == K.KVA_EINVAL
    assert append(K, rope=_rope(kind=1, rot_offset=8), cache=_cache(FAKE)) == K.KVA_EINVAL   # offset without width
    assert append(K, rope=_rope(kind=3, n_axes=2, rot_offset=0, rot_dim=62)) == K.KVA_EINVAL  # 2D needs W % 4
    assert append(K, rope=_rope(kind=2, secs=(16, 8, 0, 0), n_axes=2, rot_dim=64)) == K.KVA_EINVAL  # sum != W/2
    assert append(K, Hq=32, cache=_cache(FAKE, hkv=32, d=192, dv=264, cap=512)) == K.KVA_EUNSUPPORTED
    assert append(K, Hq=32, cache=_cache(FAKE, **asym, stride_v=-16)) == K.KVA_EINVAL
    two = dict(N=2, slot_host=[0, 0], Hq=32)
    assert append(K, cache=_cache(FAKE, hkv=32, d=192, dv=128, cap=512, stride_v=32 * 512 * 128 - 8), **two) == K.KVA_EINVAL
    assert b"inst_stride_v" in K.lib().kva_last_error()
    assert append(K, cache=_cache(FAKE, stride_v=8 * 1024 * 128 + 64), N=2, slot_host=[0, 0]) == K.KVA_EINVAL  # symmetric
    assert append(K, Hq=32, cache=_cache(FAKE, hkv=32, d=192, dv=100, cap=512)) == K.KVA_EALIGN
    L = K.lib()
    lh = np.array([3], np.int32)
    ac = _cache(FAKE, hkv=32, d=192, dv=64, cap=64)
    assert L.kv_attn_decode(FAKE, 1, ac, FAKE, lh.ctypes.data, 1, 32, 0.0, FAKE, FAKE, 1 << 30, None) == K.KVA_EUNSUPPORTED
    # the fused step takes the 192/128 cache and rotary sub-ranges (the CUDA-core form): validation
    # passes, and without a GPU the launch itself is what fails
    ac = _cache(FAKE, hkv=32, d=192, dv=128, cap=64)
    assert L.kv_attn_decode_step(FAKE, FAKE, FAKE, 0, FAKE, 0, _norm(), _rope(), ac, FAKE, lh.ctypes.data, 1, 32,
                                 0.0, None, 0, FAKE, FAKE, 1 << 30, None) in (K.KVA_OK, K.KVA_ECUDA)
    bad = _cache(FAKE, hkv=32, d=192, dv=64, cap=64)                      # value width not built
    assert L.kv_attn_decode_step(FAKE, FAKE, FAKE, 0, FAKE, 0, _norm(), _rope(), bad, FAKE, lh.ctypes.data, 1, 32,
                                 0.0, None, 0, FAKE, FAKE, 1 << 30, None) == K.KVA_EUNSUPPORTED
    sc = _cache(FAKE, cap=64)
    assert L.kv_attn_decode_step(FAKE, FAKE, FAKE, 0, FAKE, 0, _norm(), _rope(rot_offset=64, rot_dim=64), sc, FAKE,
                                 lh.ctypes.data, 1, 16, 0.0, None, 0, FAKE, FAKE, 1 << 30, None) in (K.KVA_OK, K.KVA_ECUDA)
    assert L.kv_attn_decode_step(FAKE, FAKE, FAKE, 0, FAKE, 0, _norm(), _rope(rot_offset=64, rot_dim=96), sc, FAKE,
                                 lh.ctypes.data, 1, 16, 0.0, None, 0, FAKE, FAKE, 1 << 30, None) == K.KVA_EINVAL
    assert L.kv_attn_verify(FAKE, 1, ac, FAKE, lh.ctypes.data, 1, 2, 32, 0.0, FAKE, FAKE, 1 << 30, None) == K.KVA_EUNSUPPORTED
    assert L.kv_attn_decode_static(FAKE, 1, ac, FAKE, lh.ctypes.data, 1, 32, 0.0, FAKE, None) == K.KVA_EUNSUPPORTED
    pc = _cache(FAKE, hkv=32, d=160, dv=128, cap=64)
    assert L.kv_attn_prefill(FAKE, 1, pc, 1, 3, 32, 0, None, None, None, 0.0, FAKE, None) == K.KVA_EUNSUPPORTED


def test_prefill_validation(K):
    L = K.lib()
    seg_bad = np.array([0, 1, 0], np.int32)
    def pf(S=3, mask=0, seg=None, segh=None, qd=1, cache=None):
        return L.kv_attn_prefill(FAKE, qd, cache or _cache(FAKE, cap=4), 1, S, 16, mask, seg, segh,
                                 None, 0.0, FAKE, None)
    assert pf(S=0) == K.KVA_OK
    assert pf(S=5) == K.KVA_ECAPACITY
    assert pf(qd=0) == K.KVA_EINVAL                                         # q dtype != cache dtype
    assert pf(mask=2) == K.KVA_EINVAL                                       # segment mask without ids
    assert pf(mask=2, seg=FAKE, segh=seg_bad.ctypes.data) == K.KVA_EINVAL   # not non-decreasing
    assert pf(mask=7) == K.KVA_EINVAL
    assert pf(mask=3) == K.KVA_EINVAL                                       # causal-segment without ids
    assert pf(mask=3, seg=FAKE, segh=seg_bad.ctypes.data) == K.KVA_EINVAL


def test_decode_validation(K):
    L = K.lib()
    def dec(lens, ws=FAKE, ws_bytes=1 << 30, cache=None, Hq=16):
        lh = np.asarray(lens, np.int32)
        return L.kv_attn_decode(FAKE, 1, cache or _cache(FAKE, cap=64), FAKE, lh.ctypes.data, len(lens), Hq,
                                0.0, FAKE, ws, ws_bytes, None)
    assert L.kv_attn_decode(FAKE, 1, _cache(FAKE), FAKE, None, 0, 16, 0.0, FAKE, FAKE, 0, None) == K.KVA_OK
    assert dec([0]) == K.KVA_ECAPACITY                                       # empty prefix
    assert dec([65]) == K.KVA_ECAPACITY                                      # beyond the window
    assert dec([3], ws=None) == K.KVA_EWORKSPACE
    assert dec([3], cache=_cache(FAKE, d=64, cap=64)) == K.KVA_EUNSUPPORTED   # decode built for D=128
    assert dec([3], Hq=64) == K.KVA_EUNSUPPORTED                             # group size 8
    assert L.kva_decode_workspace_size(4, 8, 16, 1000, 128) > L.kva_decode_workspace_zero_bytes(4, 8) > 0


def test_decode_step_validation(K):
    L = K.lib()
    def step(lens, ws=FAKE, ws_bytes=1 << 30, cache=None, Hq=16, k=FAKE, rope=None, pos=FAKE, norm=None):
        lh = np.asarray(lens, np.int32)
        return L.kv_attn_decode_step(FAKE, k, FAKE, 0, pos, 0, norm or _norm(), rope or _rope(),
                                     cache or _cache(FAKE, cap=64), FAKE, lh.ctypes.data, len(lens), Hq, 0.0,
                                     None, 0, FAKE, ws, ws_bytes, None)
    assert step([]) == K.KVA_OK
    assert step([0]) == K.KVA_ECAPACITY                                      # no slot for the new token
    assert step([65]) == K.KVA_ECAPACITY
    assert step([3], k=None) == K.KVA_EINVAL
    assert step([3], pos=None) == K.KVA_EINVAL                               # RoPE without positions
    assert step([3], norm=_norm(k=FAKE)) == K.KVA_EINVAL
    assert step([3], ws=None) == K.KVA_EWORKSPACE
    assert step([3], ws_bytes=16) == K.KVA_EWORKSPACE
    assert step([3], cache=_cache(FAKE, dtype=0, cap=64)) in (K.KVA_OK, K.KVA_ECUDA)   # f32 cache: CUDA-core form
    assert step([3], cache=_cache(FAKE, d=64, cap=64)) == K.KVA_EUNSUPPORTED
    assert step([3], Hq=64) == K.KVA_EUNSUPPORTED                            # group size 8
    assert step([3], rope=_rope(kind=2, secs=(16, 16, 16, 8), n_axes=4)) == K.KVA_EINVAL


def test_verify_validation(K):
    L = K.lib()
    def ver(lens, k=2, ws=FAKE, ws_bytes=1 << 30, cache=None, Hq=16):
        lh = np.asarray(lens, np.int32)
        return L.kv_attn_verify(FAKE, 1, cache or _cache(FAKE, cap=64), FAKE, lh.ctypes.data, len(lens), k, Hq,
                                0.0, FAKE, ws, ws_bytes, None)
    assert ver([]) == K.KVA_OK
    assert ver([3], k=0) == K.KVA_EINVAL
    assert ver([3], k=65) == K.KVA_EINVAL                                    # beyond the largest block
    assert ver([1], k=2) == K.KVA_ECAPACITY                                  # fewer slots than block tokens
    assert ver([65]) == K.KVA_ECAPACITY
    assert ver([3], ws=None) == K.KVA_EWORKSPACE
    assert ver([3], ws_bytes=16) == K.KVA_EWORKSPACE
    assert ver([3], cache=_cache(FAKE, dtype=0, cap=64)) == K.KVA_EUNSUPPORTED
    assert ver([3], Hq=12) == K.KVA_EINVAL
    assert L.kva_verify_workspace_size(4, 8, 16, 16, 1000, 128) > L.kva_verify_workspace_size(4, 8, 16, 1, 1000, 128)
    assert L.kv_verify_commit(FAKE, FAKE, 0, 4, FAKE, FAKE, FAKE, None) == K.KVA_OK
    assert L.kv_verify_commit(None, FAKE, 2, 4, FAKE, FAKE, FAKE, None) == K.KVA_EINVAL
    assert L.kv_verify_commit(FAKE, FAKE, 2, 0, FAKE, FAKE, FAKE, None) == K.KVA_EINVAL


def test_lmhead_validation(K):
    L = K.lib()
    def lm(B=1, H=1024, V=100, Vr=100, ws=FAKE, wsb=1 << 20, h=FAKE):
        return L.lmhead_argmax(h, FAKE, 1, B, H, V, Vr, FAKE, None, None, ws, wsb, None)
    assert lm(B=0) == K.KVA_OK
    assert lm(V=101) == K.KVA_EINVAL                                         # vocab beyond the table rows
    assert lm(H=1020) == K.KVA_EALIGN
    assert lm(ws=None) == K.KVA_EWORKSPACE
    assert lm(wsb=8) == K.KVA_EWORKSPACE
    assert lm(B=64, wsb=L.kva_lmhead_workspace_size(64, 1024) - 1) == K.KVA_EWORKSPACE
    assert L.kva_lmhead_workspace_size(64, 1024) > L.kva_lmhead_workspace_zero_bytes(64) > 0
    assert lm(h=FAKE + 8) == K.KVA_EALIGN
    assert lm(H=8192) == K.KVA_EUNSUPPORTED


def test_lmhead_topk_validation(K):
    L = K.lib()
    def tk(B=1, H=1024, V=100, Vr=100, k=4, ws=FAKE, wsb=1 << 24, norm=None, eps=1e-6):
        return L.lmhead_topk(FAKE, norm, eps, FAKE, 1, B, H, V, Vr, k, FAKE, None, ws, wsb, None)
    assert tk(B=0) == K.KVA_OK
    assert tk(k=0) == K.KVA_EINVAL
    assert tk(k=33) == K.KVA_EINVAL
    assert tk(V=10, Vr=10, k=11) == K.KVA_EINVAL                            # more ranks than vocab
    assert tk(V=101) == K.KVA_EINVAL
    assert tk(norm=FAKE, eps=-1.0) == K.KVA_EINVAL
    assert tk(norm=FAKE + 4) == K.KVA_EALIGN
    assert tk(wsb=16) == K.KVA_EWORKSPACE
    assert L.kva_lmhead_topk_workspace_size(2, 1024, 5000, 8) > L.kva_lmhead_topk_workspace_size(2, 1024, 5000, 1)


def test_binding_refuses_cpu_tensors(K):
    torch = pytest.importorskip("torch")
    with pytest.raises(K.KvaError):
        K._ptr(torch.zeros(4))
