"""Plain fp64 CPU oracle for the KV-cache GQA attention step.

TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline / reference leg import this module.  The CUDA library never calls it and
shares no code with it.

It is the plain definition of what the hot path computes, written out from the
pages in float64 with numpy (a matmul serves as the dot-product step, nothing is
blocked, fused or reordered):

  * QK-Norm: per-head RMSNorm over head_dim, eps 1e-6, one weight vector per q and
    per k shared by all heads (Penguin-VL ncnn port, section 2.1 structure
    parameters and section 4.2, norm order [input, q_norm, k_norm, post]).
  * RoPE, rotate-half form x*cos + rotate_half(x)*sin (Youtu-VL-4B ncnn port,
    implementation difficulty 2), theta 1e6 (Penguin-VL section 2.1); xdRoPE
    with sections [16,16,16,16] and effective base 1.11588e7 (HunyuanOCR v1.0
    port, section five items 1 and 3; HunyuanOCR v1.5 port, section 3.3);
    2D vision RoPE over two head-dim halves, rows then columns (Penguin-VL
    section 2.3).
  * Norm/RoPE order: norm then RoPE for Qwen3; RoPE then norm, before the cache
    write, for HunyuanOCR (HunyuanOCR v1.0 port, section five item 2).
  * Cache write of k/v into the slot of the new token, by the runtime between the
    qkv step and the attention step (Youtu-VL-4B port, implementation step 6;
    HunyuanOCR v1.0 port, section four step 4); the decoder cache may be stored
    in bf16 with fp32 accumulation (HunyuanOCR v1.5 port, section 3.7).
  * GQA head mapping: K/V heads repeat-interleaved to the query heads, so query
    head h reads KV head h // (Hq/Hkv) (Penguin-VL section 3 item 2).
  * Attention: QK^T * scale + mask, softmax unrolled as amax -> sub -> exp -> sum
    -> div, then times V (Youtu-VL-4B port, implementation difficulty 3); masked
    keys are those the additive 0/-1e9 mask hides (Youtu-VL-4B port, step 7).
  * Decode at step t is the prefill row t over the same cache (Youtu-VL-4B
    port, results table: two-stage decode replay vs parallel prefill).
  * Tied lm_head row dot products over the whole vocab and greedy argmax
    (Youtu-VL-4B port, step 6 and "decoding and sampling"; HunyuanOCR v1.5
    port, section 3.4); only rows below the logits length are valid
    (Penguin-VL section 4.1).

Readings taken where the pages are silent (each listed in the design notes):
scale = 1/sqrt(head_dim); inv_freq_j = base^(-2j/width); argmax ties go to the
lowest id; masked keys are excluded (identical to adding -1e9 in fp64 whenever a
row keeps at least one key, which every row here does).
"""
from __future__ import annotations

import math
import numpy as np

F64 = np.float64


# ----------------------------------------------------------------------------
# Storage rounding
# ----------------------------------------------------------------------------
def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (8 significant bits,
    ties to even), returned as float64.  This is the storage step of the Mixed
    precision mode (bf16 storage, fp32 accumulation: HunyuanOCR v1.5 port,
    section 3.7).  Values are finite and within bf16's normal range here."""
    x = np.asarray(x, dtype=F64)
    mant, expo = np.frexp(x)                     # x = mant * 2^expo, 0.5 <= |mant| < 1
    scale = np.ldexp(np.ones_like(x), expo - 8)  # one bf16 ulp at this binade
    out = np.round(x / scale) * scale            # np.round: half to even; x/scale exact
    return np.where(x == 0.0, x, out)


def store(x, dtype: str) -> np.ndarray:
    """Value a cache of `dtype` ('f32' or 'bf16') holds after storing float64 x."""
    x = np.asarray(x, dtype=F64)
    if dtype == "f32":
        return x.astype(np.float32).astype(F64)
    if dtype == "bf16":
        return bf16_round(x)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------
# QK-Norm
# ----------------------------------------------------------------------------
def rms_norm(x, w, eps: float) -> np.ndarray:
    """y = x / sqrt(mean_d(x^2) + eps) * w over the last axis (head_dim).
    Penguin-VL ncnn port, section 2.1 (RMSNorm eps 1e-6) and section 4.2 (q_norm,
    k_norm per layer)."""
    x = np.asarray(x, dtype=F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=F64)


# ----------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------
class Rope:
    """Rotary embedding layout.

    kind '1d':       one rotated block of width D, all frequencies use position axis 0.
    kind 'sections': one block of width D; frequency index j uses the axis whose
                     section contains j (xdRoPE sections [16,16,16,16]).
    kind '2d':       two blocks of width D/2; block b uses position axis b
                     (dims 0..D/2-1 rows, D/2..D-1 columns).
    kind 'interleaved': the 1D rotation after a de-interleave: the head is first reordered
                     to [x0, x2, ..., x_{D-2}, x1, x3, ..., x_{D-1}] (view as [D/2, 2],
                     transpose), then rotated like '1d'; the result stays in that order
                     (rope_interleave: Youtu-VL-4B port, implementation difficulty 2).
    kind 'none':     no rotation.

    rot_offset / rot_dim: the rotation acts on dims [rot_offset, rot_offset + rot_dim) only
    (its frequencies follow that width) and leaves the rest of the head as it is, the layout of
    an MLA head whose last 64 of 192 dims carry the position (Youtu-VL-4B port: K = 192 with a
    64x64 rotary permutation, implementation difficulty 2; V = 128).  rot_dim None = the head.
    """

    def __init__(self, kind: str, base: float = 1e6, sections=None, rot_offset: int = 0, rot_dim=None):
        self.kind, self.base = kind, float(base)
        self.sections = tuple(sections) if sections is not None else None
        self.rot_offset, self.rot_dim = int(rot_offset), rot_dim


def inv_freq(base: float, width: int) -> np.ndarray:
    """inv_j = base^(-2j/width), j = 0 .. width/2-1 (standard RoPE frequencies; the
    pages give theta but not the formula: reading)."""
    j = np.arange(width // 2, dtype=F64)
    return np.power(F64(base), -2.0 * j / width)


def rotate_half_apply(x, ang) -> np.ndarray:
    """Rotate-half RoPE on the last axis of x (width Db) with angles [..., Db/2]:
    y_j = x_j cos a_j - x_{j+Db/2} sin a_j,  y_{j+Db/2} = x_{j+Db/2} cos a_j + x_j sin a_j.
    Youtu-VL-4B ncnn port, implementation difficulty 2 (q*cos + rotate_half(q)*sin)."""
    x = np.asarray(x, dtype=F64)
    h = x.shape[-1] // 2
    x1, x2 = x[..., :h], x[..., h:]
    c, s = np.cos(ang), np.sin(ang)
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_apply(x, pos, rope: Rope) -> np.ndarray:
    """Apply `rope` to x [T, H, D] at integer positions pos [T, n_axes]."""
    x = np.asarray(x, dtype=F64)
    if rope.kind == "none":
        return x.copy()
    if rope.rot_dim is not None and (rope.rot_offset != 0 or rope.rot_dim != x.shape[-1]):
        o, w = rope.rot_offset, rope.rot_dim
        out = x.copy()
        out[..., o:o + w] = rope_apply(x[..., o:o + w], pos, Rope(rope.kind, rope.base, rope.sections))
        return out
    pos = np.asarray(pos, dtype=F64)
    D = x.shape[-1]
    if rope.kind in ("1d", "sections"):
        inv = inv_freq(rope.base, D)                          # [D/2]
        if rope.kind == "1d":
            axis_of_j = np.zeros(D // 2, dtype=np.int64)
        else:
            axis_of_j = np.repeat(np.arange(len(rope.sections)), rope.sections)
            assert axis_of_j.shape[0] == D // 2, "sections must cover D/2 frequencies"
        ang = pos[:, axis_of_j] * inv[None, :]                # [T, D/2]
        return rotate_half_apply(x, ang[:, None, :])
    if rope.kind == "interleaved":
        # de-interleave (x.view(D/2, 2).transpose) then the standard rotate-half
        xd = np.concatenate([x[..., 0::2], x[..., 1::2]], axis=-1)
        ang = pos[:, 0:1] * inv_freq(rope.base, D)[None, :]   # [T, D/2]
        return rotate_half_apply(xd, ang[:, None, :])
    if rope.kind == "2d":
        half = D // 2
        inv = inv_freq(rope.base, half)                       # [D/4]
        out = np.empty_like(x)
        for b in range(2):
            ang = pos[:, b:b + 1] * inv[None, :]              # [T, D/4]
            out[..., b * half:(b + 1) * half] = rotate_half_apply(
                x[..., b * half:(b + 1) * half], ang[:, None, :])
        return out
    raise ValueError(rope.kind)


def qk_transform(x, pos, w, eps, rope: Rope, norm_after_rope: bool) -> np.ndarray:
    """QK-Norm and RoPE in the order a model family uses: norm then RoPE (Qwen3,
    Penguin-VL section 5.4 intermediate order q_proj, q_norm, q_rope) or RoPE then
    norm (HunyuanOCR v1.0 port, section five item 2).  w=None skips the norm."""
    x = np.asarray(x, dtype=F64)
    if w is None:
        return rope_apply(x, pos, rope)
    if norm_after_rope:
        return rms_norm(rope_apply(x, pos, rope), w, eps)
    return rope_apply(rms_norm(x, w, eps), pos, rope)


# ----------------------------------------------------------------------------
# Cache append
# ----------------------------------------------------------------------------
def cache_append(q, k, v, pos, slot, q_norm_w, k_norm_w, eps, rope: Rope,
                 norm_after_rope: bool, cache_k, cache_v, cache_dtype: str):
    """One append of T tokens into one cache instance.

    q [T,Hq,D], k, v [T,Hkv,D]; pos [T,n_axes]; slot [T] destination slots;
    cache_k, cache_v [Hkv, W, D] float64 arrays updated in place with the stored
    (dtype-rounded) values.  Returns the exact float64 transformed q [T,Hq,D].
    The runtime writes k/v into slot t between the qkv and attention steps
    (Youtu-VL-4B port, step 6; HunyuanOCR v1.0 port, section five item 2: the
    cache holds the normalised K).  V is stored unchanged."""
    qr = qk_transform(q, pos, q_norm_w, eps, rope, norm_after_rope)
    kr = qk_transform(k, pos, k_norm_w, eps, rope, norm_after_rope)
    slot = np.asarray(slot)
    W = cache_k.shape[1]
    if np.any(slot < 0) or np.any(slot >= W):
        raise IndexError("slot outside the cache window (context overflow is rejected)")
    for t in range(qr.shape[0]):
        cache_k[:, slot[t], :] = store(kr[t], cache_dtype)
        cache_v[:, slot[t], :] = store(np.asarray(v[t], dtype=F64), cache_dtype)
    return qr


# ----------------------------------------------------------------------------
# Attention
# ----------------------------------------------------------------------------
def attend(q, cache_k, cache_v, allowed, scale=None) -> np.ndarray:
    """o[i,h] = softmax_j(q[i,h] . K[g,j] * scale, j allowed) . V[g,j], g = h // (Hq/Hkv).

    q [Sq, Hq, D]; cache_k, cache_v [Hkv, W, D]; allowed [Sq, W] bool.
    Softmax unrolled as amax -> sub -> exp -> sum -> div (Youtu-VL-4B port,
    implementation difficulty 3).  GQA grouping by repeat-interleave (Penguin-VL
    section 3)."""
    q = np.asarray(q, dtype=F64)
    Sq, Hq, D = q.shape
    Hkv = cache_k.shape[0]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.zeros((Sq, Hq, cache_v.shape[2]), dtype=F64)
    for h in range(Hq):
        g = h // G
        K = np.asarray(cache_k[g], dtype=F64)                # [W, D]
        V = np.asarray(cache_v[g], dtype=F64)
        for i in range(Sq):
            idx = np.nonzero(allowed[i])[0]
            s = (K[idx] @ q[i, h]) * scale                    # logits of the allowed keys
            m = np.max(s)                                     # amax
            e = np.exp(s - m)                                 # sub, exp
            p = e / np.sum(e)                                 # sum, div
            out[i, h] = p @ V[idx]
    return out


def prefill_mask(S: int, kind: str, segment=None) -> np.ndarray:
    """Allowed-key matrix [S, S] in cache-slot order.  'causal': j <= i (the
    additive mask 0 at slots <= t, -1e9 elsewhere: Youtu-VL-4B port, step 7);
    'full': all keys; 'segment': keys of the same window only (block-diagonal mask of
    the windowed vision layers: Youtu-VL-4B port, step 3)."""
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    if kind == "causal":
        return j <= i
    if kind == "full":
        return np.ones((S, S), dtype=bool)
    if kind == "segment":
        seg = np.asarray(segment)
        return seg[:, None] == seg[None, :]
    if kind == "causal_segment":
        # causal, plus every key of the row's own segment: an image span (one segment) is
        # visible as a whole to its rows while text keeps the causal mask (MNN llm_demo
        # walkthrough, section 3.3); a text token is a segment of its own
        seg = np.asarray(segment)
        return (j <= i) | (seg[:, None] == seg[None, :])
    raise ValueError(kind)


def prefill(q_slots, cache_k, cache_v, S: int, kind: str, segment=None, scale=None):
    """Parallel prefill over cache slots 0..S-1; q_slots [S, Hq, D] holds the query
    of the token stored in each slot (Youtu-VL-4B port, step 7)."""
    allowed = np.zeros((S, cache_k.shape[1]), dtype=bool)
    allowed[:, :S] = prefill_mask(S, kind, segment)
    return attend(q_slots, cache_k, cache_v, allowed, scale)


def decode(q, cache_k, cache_v, length: int, scale=None):
    """Single-token decode: q [Hq, D] against the first `length` cache slots (the
    new token's slot included).  Youtu-VL-4B port, step 8; HunyuanOCR v1.0 port,
    section four step 4 (attention consumes the whole window plus the mask)."""
    allowed = np.zeros((1, cache_k.shape[1]), dtype=bool)
    allowed[0, :length] = True
    return attend(np.asarray(q, dtype=F64)[None], cache_k, cache_v, allowed, scale)[0]


# ----------------------------------------------------------------------------
# Speculative-decoding verify block (DFlash)
# ----------------------------------------------------------------------------
def verify_block(q_rows, cache_k, cache_v, length: int, scale=None):
    """One verify forward of a k-token block: q_rows [k, Hq, D] are the queries of the tokens
    stored in the last k valid slots (length - k .. length - 1), and row i attends to the keys
    of slots 0 .. length - k + i (a multi-token causal mask over the existing cache: HunyuanOCR
    v1.5 port, section 3.8, target verification)."""
    q_rows = np.asarray(q_rows, dtype=F64)
    k = q_rows.shape[0]
    if not 1 <= k <= length:
        raise ValueError("block of k tokens needs 1 <= k <= length")
    allowed = np.zeros((k, cache_k.shape[1]), dtype=bool)
    for i in range(k):
        allowed[i, :length - k + i + 1] = True
    return attend(q_rows, cache_k, cache_v, allowed, scale)


def verify_accept(posterior, block_tokens, length: int):
    """Acceptance and commit of a verify block (HunyuanOCR v1.5 port, section 3.8): the block
    holds the current token and k - 1 draft candidates (block_tokens [k], in slots
    length - k .. length - 1); posterior [k] is the target's greedy id after each of them.
    Candidate i + 1 is accepted while posterior[i] equals it, stopping at the first mismatch;
    the target's id after the accepted prefix is kept (the correction, or the next token when
    every candidate matched).  The cache is cut back to the current token plus the accepted
    candidates.  Returns (accepted a, next token, committed length)."""
    posterior = np.asarray(posterior)
    block_tokens = np.asarray(block_tokens)
    k = block_tokens.shape[0]
    a = 0
    while a < k - 1 and posterior[a] == block_tokens[a + 1]:
        a += 1
    return a, int(posterior[a]), length - k + a + 1


# ----------------------------------------------------------------------------
# Greedy lm_head
# ----------------------------------------------------------------------------
def lm_logits(h, W, V: int) -> np.ndarray:
    """z_v = sum_k W[v,k] h[k] for v < V (tied [vocab, hidden] table, row dot
    products: Youtu-VL-4B port, step 6; HunyuanOCR v1.5 port, section 3.4).
    W may be float or raw bf16 bits (uint16), widened exactly."""
    Wf = W
    if W.dtype == np.uint16:
        Wf = (W[:V].astype(np.uint32) << 16).view(np.float32)
    return np.asarray(Wf[:V], dtype=F64) @ np.asarray(h, dtype=F64)


def argmax_lowest(z) -> tuple[int, float, float]:
    """Greedy pick: (id, max logit, top1 - top2 margin).  Ties go to the lowest id
    (reading; numpy.argmax returns the first maximum)."""
    z = np.asarray(z, dtype=F64)
    i = int(np.argmax(z))
    top = z[i]
    rest = np.delete(z, i)
    margin = float(top - np.max(rest)) if rest.size else math.inf
    return i, float(top), margin


def topk_lowest(z, k: int):
    """The k largest entries of z as (ids [k], values [k]), ordered by value descending and, among
    equal values, by id ascending (the argmax tie rule extended to a ranking).  A plain sort on
    (-value, id)."""
    z = np.asarray(z, dtype=F64)
    order = sorted(range(z.shape[0]), key=lambda v: (-z[v], v))[:k]
    return np.asarray(order, dtype=np.int64), z[order]


def lmhead_topk(h, W, V: int, k: int, norm_w=None, eps: float = 1e-6):
    """Greedy step with the final RMSNorm in front of the tied lm_head (Youtu-VL-4B port,
    "decoding and sampling": every step takes final RMSNorm, then lm_head logits over the whole
    vocabulary, then the highest-probability token; step 8), returning the k best ids and their
    logits per row of h [B, H] (top_k is one of the generation options of the published
    interface, HunyuanOCR v1.5 port, section 3.6; k = 1 is the greedy id).  norm_w None skips
    the norm."""
    h = np.atleast_2d(np.asarray(h, dtype=F64))
    if norm_w is not None:
        h = np.stack([rms_norm(row, norm_w, eps) for row in h])
    ids, vals = [], []
    for row in h:
        i, v = topk_lowest(lm_logits(row, W, V), k)
        ids.append(i); vals.append(v)
    return np.stack(ids), np.stack(vals)


def lmhead_argmax(h, W, V: int):
    """For each row of h [B, H]: (ids [B], max [B], margin [B]).  Only the first V
    rows are candidates: the selector clamps the vocab to the logits length
    (Penguin-VL section 4.1)."""
    h = np.atleast_2d(np.asarray(h, dtype=F64))
    ids, mx, mg = [], [], []
    for b in range(h.shape[0]):
        i, m, g = argmax_lowest(lm_logits(h[b], W, V))
        ids.append(i); mx.append(m); mg.append(g)
    return np.asarray(ids, dtype=np.int64), np.asarray(mx), np.asarray(mg)
