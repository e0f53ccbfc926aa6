"""Thin ctypes binding of the C ABI in include/kv_attn.h.

Argument marshalling only: every step of the attention path runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (PyTorch supplies device memory and streams);
their data pointers, sizes and the current CUDA stream go straight to the C entry points
of the same names.  There is no fallback: if libkv_attn.so is missing or a call fails, a
KvaError is raised.
"""
from __future__ import annotations

import ctypes as C
import dataclasses
import os
from typing import Optional, Sequence

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkv_attn.so")

# enums (include/kv_attn.h)
KVA_OK, KVA_EINVAL, KVA_ECAPACITY, KVA_EUNSUPPORTED, KVA_ECUDA, KVA_EALIGN, KVA_EWORKSPACE = range(7)
KVA_F32, KVA_BF16 = 0, 1
MASKS = {"causal": 0, "full": 1, "segment": 2, "causal_segment": 3}
ROPE_KINDS = {"none": 0, "1d": 1, "sections": 2, "2d": 3, "interleaved": 4}


class KvaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"[{status}] {msg}")
        self.status = status


class _Cache(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("dtype", C.c_int),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("capacity", C.c_int32),
                ("inst_stride", C.c_int64), ("head_dim_v", C.c_int32), ("inst_stride_v", C.c_int64)]


class _Rope(C.Structure):
    _fields_ = [("kind", C.c_int), ("n_axes", C.c_int32), ("sections", C.c_int32 * 4),
                ("base", C.c_double), ("rot_offset", C.c_int32), ("rot_dim", C.c_int32)]


class _Norm(C.Structure):
    _fields_ = [("q_w", C.c_void_p), ("k_w", C.c_void_p), ("inst_stride", C.c_int64),
                ("eps", C.c_float), ("after_rope", C.c_int32)]


class _WorkspaceDims(C.Structure):
    _fields_ = [("B", C.c_int32), ("n_kv_heads", C.c_int32), ("n_q_heads", C.c_int32), ("max_len", C.c_int32),
                ("head_dim", C.c_int32), ("hidden", C.c_int32), ("vocab", C.c_int32), ("block", C.c_int32)]


WORKSPACE_KINDS = {"decode": 0, "verify": 1, "lmhead": 2, "lmhead_topk": 3}

_lib = None


def lib() -> C.CDLL:
    """Load libkv_attn.so (built by kv_cache_gqa_gb300/build.py); raises if it is absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise KvaError(KVA_EUNSUPPORTED, f"{_LIB_PATH} is missing: run kv_cache_gqa_gb300/build.py "
                           "(there is no CPU fallback)")
        L = C.CDLL(_LIB_PATH)
        vp, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
        L.kv_cache_append_rope_qknorm.argtypes = [vp, vp, vp, C.c_int, i32, i32, i32, vp, i64, vp, i64,
                                                  vp, _Norm, _Rope, vp, C.c_int, _Cache, vp]
        L.kv_attn_prefill.argtypes = [vp, C.c_int, _Cache, i32, i32, i32, C.c_int, vp, vp, vp,
                                      C.c_float, vp, vp]
        L.kv_attn_decode.argtypes = [vp, C.c_int, _Cache, vp, vp, i32, i32, C.c_float, vp, vp, sz, vp]
        L.kv_attn_decode_step.argtypes = [vp, vp, vp, C.c_int, vp, i64, _Norm, _Rope, _Cache, vp, vp, i32, i32,
                                          C.c_float, vp, C.c_int, vp, vp, sz, vp]
        L.kv_attn_decode_step.restype = C.c_int
        L.kv_attn_verify.argtypes = [vp, C.c_int, _Cache, vp, vp, i32, i32, i32, C.c_float, vp, vp, sz, vp]
        L.kv_attn_verify.restype = C.c_int
        L.kva_verify_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        L.kva_verify_workspace_size.restype = sz
        L.kv_verify_commit.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp]
        L.kv_verify_commit.restype = C.c_int
        L.lmhead_topk.argtypes = [vp, vp, C.c_float, vp, C.c_int, i32, i32, i32, i32, i32, vp, vp, vp, sz, vp]
        L.lmhead_topk.restype = C.c_int
        L.kva_lmhead_topk_workspace_size.argtypes = [i32, i32, i32, i32]
        L.kva_lmhead_topk_workspace_size.restype = sz
        L.kv_attn_decode_static.argtypes = [vp, C.c_int, _Cache, vp, vp, i32, i32, C.c_float, vp, vp]
        L.kv_attn_decode_static.restype = C.c_int
        L.lmhead_argmax.argtypes = [vp, vp, C.c_int, i32, i32, i32, i32, vp, vp, vp, vp, sz, vp]
        L.kva_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        L.kva_decode_workspace_size.restype = sz
        L.kva_decode_workspace_zero_bytes.argtypes = [i32, i32]
        L.kva_decode_workspace_zero_bytes.restype = sz
        L.kva_lmhead_workspace_size.argtypes = [i32, i32]
        L.kva_lmhead_workspace_size.restype = sz
        L.kva_lmhead_workspace_zero_bytes.argtypes = [i32]
        L.kva_lmhead_workspace_zero_bytes.restype = sz
        L.kva_workspace_size.argtypes = [i32, C.POINTER(_WorkspaceDims)]
        L.kva_workspace_size.restype = sz
        L.kva_strerror.argtypes = [C.c_int]
        L.kva_strerror.restype = C.c_char_p
        L.kva_last_error.restype = C.c_char_p
        L.kva_launch_count.restype = C.c_uint64
        L.kva_version.restype = C.c_int32
        L.kva_wait_timeouts.argtypes = [i32]
        L.kva_wait_timeouts.restype = i64
        L.kva_selftest_wait_timeout.argtypes = [vp]
        L.kva_selftest_wait_timeout.restype = C.c_int
        for f in ("kv_cache_append_rope_qknorm", "kv_attn_prefill", "kv_attn_decode", "lmhead_argmax"):
            getattr(L, f).restype = C.c_int
        _lib = L
    return _lib


def _check(status: int):
    if status != KVA_OK:
        raise KvaError(status, lib().kva_last_error().decode())


_torch = None


def _t():
    global _torch
    if _torch is None:
        import torch
        _torch = torch
    return _torch


def _dtype_code(t) -> int:
    torch = _t()
    if t.dtype == torch.float32:
        return KVA_F32
    if t.dtype == torch.bfloat16:
        return KVA_BF16
    raise KvaError(KVA_EINVAL, f"unsupported dtype {t.dtype}")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    if not t.is_cuda:
        raise KvaError(KVA_EINVAL, "expected a CUDA tensor")
    return t.data_ptr()


def _host_i32(a) -> np.ndarray:
    """Host mirror (int32, C-contiguous) of an index array given as numpy or a CPU tensor."""
    if type(a) is np.ndarray and a.dtype == np.int32 and a.flags.c_contiguous:
        return a
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _stream(stream) -> Optional[int]:
    s = stream if stream is not None else _t().cuda.current_stream()
    return s.cuda_stream


@dataclasses.dataclass
class KVCache:
    """N cache instances: k [N, Hkv, capacity, Dk] and v [N, Hkv, capacity, Dv] torch CUDA
    tensors (f32 or bf16); Dv differs from Dk for an asymmetric (MLA-expanded) cache."""
    k: object
    v: object

    def __setattr__(self, name, value):
        object.__setattr__(self, name, value)
        object.__setattr__(self, "_struct", None)        # rebuilt on the next call

    @property
    def struct(self) -> _Cache:
        st = getattr(self, "_struct", None)
        if st is None:
            st = self._build_struct()
            object.__setattr__(self, "_struct", st)
        return st

    def _build_struct(self) -> _Cache:
        k, v = self.k, self.v
        if k.dim() != 4 or v.dim() != 4 or v.shape[:3] != k.shape[:3] or v.dtype != k.dtype:
            raise KvaError(KVA_EINVAL, "cache k/v must be [N, Hkv, W, Dk] / [N, Hkv, W, Dv] tensors of one dtype")
        if not (k.is_contiguous() and v.is_contiguous()):
            raise KvaError(KVA_EINVAL, "cache tensors must be contiguous")
        N, Hkv, W, D = k.shape
        Dv = v.shape[3]
        return _Cache(k.data_ptr(), v.data_ptr(), _dtype_code(k), Hkv, D, W, Hkv * W * D, Dv, Hkv * W * Dv)

    @property
    def n_kv_heads(self):
        return self.k.shape[1]

    @property
    def head_dim(self):
        return self.k.shape[3]

    @property
    def head_dim_v(self):
        return self.v.shape[3]

    @property
    def capacity(self):
        return self.k.shape[2]


@dataclasses.dataclass
class Rope:
    """kind: 'none' | '1d' | 'sections' | '2d' | 'interleaved'; sections for 'sections' (sum W/2).
    rot_offset / rot_dim: rotate head dims [rot_offset, rot_offset + rot_dim) only (W = rot_dim);
    rot_dim 0 = the whole head."""
    kind: str = "1d"
    base: float = 1e6
    sections: Sequence[int] = ()
    rot_offset: int = 0
    rot_dim: int = 0

    @property
    def n_axes(self) -> int:
        return {"none": 0, "1d": 1, "2d": 2, "interleaved": 1}.get(self.kind, len(self.sections))

    def __setattr__(self, name, value):
        object.__setattr__(self, name, value)
        object.__setattr__(self, "_struct", None)        # rebuilt on the next call

    @property
    def struct(self) -> _Rope:
        st = getattr(self, "_struct", None)
        if st is None:
            secs = (C.c_int32 * 4)(*(list(self.sections) + [0] * (4 - len(self.sections))))
            st = _Rope(ROPE_KINDS[self.kind], self.n_axes, secs, float(self.base), int(self.rot_offset),
                       int(self.rot_dim))
            object.__setattr__(self, "_struct", st)
        return st


def kv_cache_append_rope_qknorm(q, k, v, pos, slot, slot_host, cache: KVCache, q_out, rope: Rope,
                                q_norm_w=None, k_norm_w=None, eps: float = 1e-6,
                                norm_after_rope: bool = False, norm_inst_stride: int = 0,
                                pos_inst_stride: Optional[int] = None,
                                slot_inst_stride: Optional[int] = None, stream=None):
    """q [N,T,Hq,D], k/v [N,T,Hkv,D] (CUDA, f32|bf16); pos [N|1,T,n_axes] int32 CUDA;
    slot [N|1,T] int32 CUDA with host mirror slot_host; q_out [N,T,Hq,D] CUDA f32|bf16.
    Instance strides of pos/slot default to T*n_axes / T when the leading dim is N, else 0."""
    N, T, Hq, _ = q.shape
    if pos_inst_stride is None:
        pos_inst_stride = 0 if (pos is None or pos.dim() < 3 or pos.shape[0] == 1) else pos.shape[1] * pos.shape[2]
    if slot_inst_stride is None:
        slot_inst_stride = 0 if (slot.dim() < 2 or slot.shape[0] == 1) else slot.shape[1]
    sh = _host_i32(slot_host)
    norm = _Norm(_ptr(q_norm_w), _ptr(k_norm_w), norm_inst_stride, eps, 1 if norm_after_rope else 0)
    _check(lib().kv_cache_append_rope_qknorm(
        _ptr(q), _ptr(k), _ptr(v), _dtype_code(q), N, T, Hq,
        _ptr(pos), pos_inst_stride, _ptr(slot), slot_inst_stride, sh.ctypes.data,
        norm, rope.struct, _ptr(q_out), _dtype_code(q_out), cache.struct, _stream(stream)))


def kv_attn_prefill(q, cache: KVCache, out, mask: str = "causal", segment=None, segment_host=None,
                    row_of_slot=None, scale: float = 0.0, stream=None):
    """q [N,S,Hq,D] (CUDA, dtype of the cache); out [N,S,Hq,D] float32 CUDA."""
    N, S, Hq, _ = q.shape
    segh = _host_i32(segment_host) if segment_host is not None else None
    _check(lib().kv_attn_prefill(
        _ptr(q), _dtype_code(q), cache.struct, N, S, Hq, MASKS[mask],
        _ptr(segment), segh.ctypes.data if segh is not None else None, _ptr(row_of_slot),
        float(scale), _ptr(out), _stream(stream)))


def decode_workspace_bytes(B: int, n_kv_heads: int, n_q_heads: int, max_len: int, head_dim: int) -> int:
    return int(lib().kva_decode_workspace_size(B, n_kv_heads, n_q_heads, max_len, head_dim))


def lmhead_workspace_bytes(B: int, H: int = 1024) -> int:
    return int(lib().kva_lmhead_workspace_size(B, H))


def workspace_bytes(kind: str, B: int = 0, n_kv_heads: int = 0, n_q_heads: int = 0, max_len: int = 0,
                    head_dim: int = 0, hidden: int = 0, vocab: int = 0, block: int = 0) -> int:
    """kva_workspace_size: the workspace of the call `kind` names ('decode', 'verify', 'lmhead',
    'lmhead_topk'); 0 for dimensions that are not positive."""
    d = _WorkspaceDims(B, n_kv_heads, n_q_heads, max_len, head_dim, hidden, vocab, block)
    return int(lib().kva_workspace_size(WORKSPACE_KINDS[kind], C.byref(d)))


def kv_attn_decode(q, cache: KVCache, lengths, lengths_host, out, workspace, scale: float = 0.0,
                   stream=None):
    """q [B,Hq,D] CUDA; lengths [B] int32 CUDA + host mirror; out [B,Hq,D] float32 CUDA;
    workspace: uint8 CUDA tensor (zeroed once before first use)."""
    B, Hq, _ = q.shape
    lh = _host_i32(lengths_host)
    _check(lib().kv_attn_decode(
        _ptr(q), _dtype_code(q), cache.struct, _ptr(lengths), lh.ctypes.data, B, Hq, float(scale),
        _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


_norm_cache = {}


def _norm_struct(q_norm_w, k_norm_w, inst_stride, eps, after):
    """The QK-Norm descriptor (cached: a decode loop passes the same weights every step)."""
    key = (_ptr(q_norm_w), _ptr(k_norm_w), int(inst_stride), float(eps), int(after))
    st = _norm_cache.get(key)
    if st is None:
        if len(_norm_cache) > 64:
            _norm_cache.clear()
        st = _norm_cache[key] = _Norm(key[0], key[1], key[2], key[3], key[4])
    return st


class PreparedCall:
    """One C-ABI call whose arguments were marshalled once.  Calling it calls the entry point
    again: the library validates, plans and launches every time; only the Python-side conversion
    of tensors into pointers and descriptors is skipped.  The tensors and host arrays it was made
    from must stay alive and keep their storage (their contents may change between calls, which
    is how a decode loop advances its lengths), and the stream is the one current (or given)
    when it was made."""
    __slots__ = ("_fn", "_args", "_keep")

    def __init__(self, fn, args, keep):
        self._fn, self._args, self._keep = fn, args, keep

    def __call__(self):
        st = self._fn(*self._args)
        if st != KVA_OK:
            raise KvaError(st, lib().kva_last_error().decode())


def prepare_decode_step(q, k, v, pos, cache: KVCache, lengths, lengths_host, out, workspace, rope: Rope,
                        q_norm_w=None, k_norm_w=None, eps: float = 1e-6, norm_after_rope: bool = False,
                        norm_inst_stride: int = 0, pos_inst_stride: Optional[int] = None, q_out=None,
                        scale: float = 0.0, stream=None) -> PreparedCall:
    """kv_attn_decode_step with its arguments marshalled once (see PreparedCall)."""
    B, Hq, _ = q.shape
    if pos_inst_stride is None:
        pos_inst_stride = 0 if (pos is None or pos.dim() < 2 or pos.shape[0] == 1) else pos.shape[-1]
    lh = _host_i32(lengths_host)
    norm = _norm_struct(q_norm_w, k_norm_w, norm_inst_stride, eps, 1 if norm_after_rope else 0)
    args = (_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(pos), pos_inst_stride, norm, rope.struct,
            cache.struct, _ptr(lengths), lh.ctypes.data, B, Hq, float(scale), _ptr(q_out),
            _dtype_code(q_out) if q_out is not None else 0, _ptr(out), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream))
    return PreparedCall(lib().kv_attn_decode_step, args, (lh, cache, rope))


def kv_attn_decode_step(q, k, v, pos, cache: KVCache, lengths, lengths_host, out, workspace, rope: Rope,
                        q_norm_w=None, k_norm_w=None, eps: float = 1e-6, norm_after_rope: bool = False,
                        norm_inst_stride: int = 0, pos_inst_stride: Optional[int] = None, q_out=None,
                        scale: float = 0.0, stream=None):
    """Fused append + decode of one new token per instance.  q [B,Hq,Dk], k [B,Hkv,Dk], v [B,Hkv,Dv]
    raw projections (CUDA f32|bf16); pos [B|1, n_axes] int32 CUDA; lengths [B] int32 CUDA (valid
    slots incl. the new token, which is written to slot L-1) + host mirror; out [B,Hq,Dv] f32."""
    prepare_decode_step(q, k, v, pos, cache, lengths, lengths_host, out, workspace, rope, q_norm_w=q_norm_w,
                        k_norm_w=k_norm_w, eps=eps, norm_after_rope=norm_after_rope,
                        norm_inst_stride=norm_inst_stride, pos_inst_stride=pos_inst_stride, q_out=q_out,
                        scale=scale, stream=stream)()


def verify_workspace_bytes(B: int, n_kv_heads: int, n_q_heads: int, k: int, max_len: int, head_dim: int) -> int:
    return int(lib().kva_verify_workspace_size(B, n_kv_heads, n_q_heads, k, max_len, head_dim))


def kv_attn_verify(q, cache: KVCache, lengths, lengths_host, out, workspace, scale: float = 0.0, stream=None):
    """q [B,k,Hq,D] (CUDA, f32|bf16): the block's queries, its tokens already in the last k valid
    slots; lengths [B] int32 CUDA (slots incl. the block) + host copy; out [B,k,Hq,D] f32."""
    B, k, Hq, _ = q.shape
    lh = _host_i32(lengths_host)
    _check(lib().kv_attn_verify(_ptr(q), _dtype_code(q), cache.struct, _ptr(lengths), lh.ctypes.data, B, k, Hq,
                                float(scale), _ptr(out), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream)))


def kv_verify_commit(posterior, block_tokens, lengths, accepted, next_token, stream=None):
    """posterior, block_tokens [B,k] int32 CUDA; lengths [B] int32 CUDA (updated in place);
    accepted, next_token [B] int32 CUDA outputs."""
    B, k = block_tokens.shape
    _check(lib().kv_verify_commit(_ptr(posterior), _ptr(block_tokens), B, k, _ptr(lengths), _ptr(accepted),
                                  _ptr(next_token), _stream(stream)))


def lmhead_topk_workspace_bytes(B: int, H: int, V: int, top_k: int) -> int:
    return int(lib().kva_lmhead_topk_workspace_size(B, H, V, top_k))


def lmhead_topk(h, W, out_ids, workspace, norm_w=None, eps: float = 1e-6, V=None, out_vals=None, stream=None):
    """h [B,H] f32 CUDA; W [V_rows,H] f32|bf16 CUDA; norm_w [H] f32 CUDA or None (final RMSNorm);
    out_ids [B,k] int32 CUDA (k = top_k); out_vals [B,k] f32 CUDA or None."""
    h2 = h if h.dim() == 2 else h.view(1, -1)
    B, H = h2.shape
    k = out_ids.shape[-1] if out_ids.dim() > 1 else 1
    V_rows = W.shape[0]
    _check(lib().lmhead_topk(_ptr(h2), _ptr(norm_w), float(eps), _ptr(W), _dtype_code(W), B, H,
                             V_rows if V is None else int(V), V_rows, k, _ptr(out_ids), _ptr(out_vals),
                             _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def prepare_lmhead_argmax(h, W, out_ids, workspace, V: Optional[int] = None, out_max=None, logits=None,
                          stream=None) -> PreparedCall:
    """lmhead_argmax with its arguments marshalled once (see PreparedCall)."""
    B, H = h.shape
    V_rows = W.shape[0]
    V = V_rows if V is None else V
    args = (_ptr(h), _ptr(W), _dtype_code(W), B, H, V, V_rows, _ptr(out_ids), _ptr(out_max), _ptr(logits),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    return PreparedCall(lib().lmhead_argmax, args, ())


def lmhead_argmax(h, W, out_ids, workspace, V: Optional[int] = None, out_max=None, logits=None,
                  stream=None):
    """h [B,H] float32 CUDA; W [V_rows,H] bf16|f32 CUDA; out_ids [B] int32 CUDA."""
    prepare_lmhead_argmax(h, W, out_ids, workspace, V=V, out_max=out_max, logits=logits, stream=stream)()


def launch_count() -> int:
    return int(lib().kva_launch_count())


def version() -> int:
    return int(lib().kva_version())


def wait_timeouts(reset: bool = False) -> int:
    """kva_wait_timeouts: kernel waits that gave up on the current device since the last reset
    (synchronise first); -1 if the count could not be read."""
    return int(lib().kva_wait_timeouts(1 if reset else 0))


# Raw C entry points for callers that marshal pointers themselves (tests of the ABI).
def raw():
    return lib()
