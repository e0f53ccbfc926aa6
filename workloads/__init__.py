"""Seeded synthetic inputs for the KV-cache GQA attention step.

This module only draws numbers and lays out positions, slots and segment ids.
It holds none of the method's arithmetic (no norm, no rotation, no softmax,
no dot product) so that both the CUDA path's tests and the CPU oracle can take
their inputs from it without sharing any of the computation.

The five workloads follow the shapes the pages give:
  * Qwen3 attention geometry: 16 query heads, 8 KV heads, head_dim 128,
    hidden 1024, 28 layers, vocab 151936, RoPE theta 1e6, RMSNorm eps 1e-6
    (Penguin-VL ncnn port, section 2.1 "structure parameters").
  * HunyuanOCR image span: 1 + h*(w+1) + 1 rows, 274 = 1 + 16*17 + 1
    (HunyuanOCR v1.0 ncnn port, section five item 4; HunyuanOCR v1.5 ncnn port,
    section 3.1 visual token count Nv = (gh/m)*(gw/m + 1) + 2).
  * Vision tower: 14 x 92 = 1288 patches, 322 merged 2x2 tokens, windows of
    8 x 8 merged patches chosen by a window_index permutation
    (Youtu-VL-4B ncnn port, results section and implementation step 3).

Random draws use numpy's PCG64 generator (numpy.random.default_rng), seeded
per workload; every array records the order it is drawn in, so both sides of a
comparison see identical bytes.
"""
from __future__ import annotations

import dataclasses
import numpy as np

# ----------------------------------------------------------------------------
# Model constants printed by the pages
# ----------------------------------------------------------------------------
QWEN3_N_Q_HEADS = 16
QWEN3_N_KV_HEADS = 8
QWEN3_HEAD_DIM = 128
QWEN3_HIDDEN = 1024
QWEN3_LAYERS = 28
QWEN3_VOCAB = 151936
QWEN3_ROPE_THETA = 1.0e6
QWEN3_RMS_EPS = 1.0e-6
XDROPE_BASE = 1.11588e7          # effective base reported by the HunyuanOCR v1.0 port
XDROPE_SECTIONS = (16, 16, 16, 16)
VISION_GRID = (14, 92)           # patch rows x cols of the 1468x220 banner
VISION_MERGE = 2                 # 2x2 merge -> 7 x 46 merged grid
VISION_WINDOW = 8                # 8 x 8 merged patches per window
VISION_HEAD_DIM = 72
VISION_HEADS = 16


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even) and return the raw
    16-bit patterns.  Used only to store synthetic weights/caches in bf16; inputs are
    finite by construction."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((b >> 16) & 1) + np.uint32(0x7FFF)
    return ((b + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen raw bfloat16 patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# Position / slot / segment builders
# ----------------------------------------------------------------------------
def positions_1d(start: int, count: int) -> np.ndarray:
    """[count, 1] int32 text positions start .. start+count-1."""
    return np.arange(start, start + count, dtype=np.int32)[:, None].copy()


def image_span_positions(text_before: int, grid_h: int, grid_w: int,
                         text_after: int, image_index: int = 0) -> np.ndarray:
    """4-axis position ids [S, 4] for text + one image span + text.

    Layout of the span: one begin row, grid_h rows of (grid_w + 1) cells (the last
    cell of each row is the row separator), one end row, i.e. 1 + h*(w+1) + 1 rows.
    Text rows (and the span's begin/end rows) carry their sequence index on all four
    axes.  Grid cell (r, c) at sequence index p carries (p, r, c, image_index):
    axis 0 = position, 1 = height, 2 = width, 3 = image index.
    """
    rows = []
    p = 0
    for _ in range(text_before):
        rows.append((p, p, p, p)); p += 1
    rows.append((p, p, p, p)); p += 1                    # span begin marker
    for r in range(grid_h):
        for c in range(grid_w + 1):                       # c == grid_w: row separator
            rows.append((p, r, c, image_index)); p += 1
    rows.append((p, p, p, p)); p += 1                    # span end marker
    for _ in range(text_after):
        rows.append((p, p, p, p)); p += 1
    return np.asarray(rows, dtype=np.int32)


def image_span_segments(text_before: int, grid_h: int, grid_w: int, text_after: int) -> np.ndarray:
    """Segment ids [S] for the layout of image_span_positions: every text row (the span's begin
    and end markers included) is a segment of its own (id = its index); the h*(w+1) grid rows
    of the span share one id (the index of the first grid row).  Non-decreasing."""
    S = text_before + 2 + grid_h * (grid_w + 1) + text_after
    seg = np.arange(S, dtype=np.int32)
    g0 = text_before + 1
    g1 = g0 + grid_h * (grid_w + 1)
    seg[g0:g1] = g0
    return seg


@dataclasses.dataclass
class VisionLayout:
    pos_rc: np.ndarray       # [S, 2] int32 (row, col) of each patch, natural row-major order
    slot: np.ndarray         # [S] int32: window-ordered slot of natural token t
    row_of_slot: np.ndarray  # [S] int32: natural token stored in slot i (inverse of slot)
    segment: np.ndarray      # [S] int32: window id of slot i (non-decreasing)
    window_sizes: list


def vision_window_layout(grid=VISION_GRID, merge=VISION_MERGE,
                         window=VISION_WINDOW) -> VisionLayout:
    """Window permutation for windowed vision attention.

    Natural order: patches row-major over the grid.  Merged unit (mr, mc) =
    (r // merge, c // merge); window (wr, wc) = (mr // window, mc // window),
    anchored at (0, 0) so edge windows are ragged.  Window order: windows row-major;
    inside a window, merged units row-major; inside a unit, its patches row-major.
    """
    gh, gw = grid
    mh, mw = gh // merge, gw // merge
    nwr, nwc = -(-mh // window), -(-mw // window)
    order = []
    sizes = []
    seg = []
    for wr in range(nwr):
        for wc in range(nwc):
            n0 = len(order)
            for mr in range(wr * window, min((wr + 1) * window, mh)):
                for mc in range(wc * window, min((wc + 1) * window, mw)):
                    for dr in range(merge):
                        for dc in range(merge):
                            r, c = mr * merge + dr, mc * merge + dc
                            order.append(r * gw + c)
            sizes.append(len(order) - n0)
            seg.extend([len(sizes) - 1] * (len(order) - n0))
    row_of_slot = np.asarray(order, dtype=np.int32)
    slot = np.empty_like(row_of_slot)
    slot[row_of_slot] = np.arange(len(order), dtype=np.int32)
    rr, cc = np.divmod(np.arange(gh * gw, dtype=np.int32), gw)
    pos_rc = np.stack([rr, cc], axis=1).astype(np.int32)
    return VisionLayout(pos_rc, slot, row_of_slot, np.asarray(seg, dtype=np.int32), sizes)


# ----------------------------------------------------------------------------
# Workload recipes
# ----------------------------------------------------------------------------
def _normal(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32)


def norm_weights(rng, d):
    """QK-Norm weight 1 + 0.1*N(0,1) (float32)."""
    return (1.0 + 0.1 * rng.standard_normal(d)).astype(np.float32)


def tiny_fp32(seed: int = 0, n_tokens: int = 80, n_prefill: int = 64):
    """Tiny fp32 single layer: 16/8 heads, D=128, prefill 64 then 16 decode steps.
    Draw order: q, k, v, q_norm_w, k_norm_w."""
    rng = np.random.default_rng(seed)
    Hq, Hkv, D = QWEN3_N_Q_HEADS, QWEN3_N_KV_HEADS, QWEN3_HEAD_DIM
    return dict(
        q=_normal(rng, (n_tokens, Hq, D)), k=_normal(rng, (n_tokens, Hkv, D)),
        v=_normal(rng, (n_tokens, Hkv, D)),
        q_norm_w=norm_weights(rng, D), k_norm_w=norm_weights(rng, D),
        pos=positions_1d(0, n_tokens), n_prefill=n_prefill, eps=QWEN3_RMS_EPS,
        base=QWEN3_ROPE_THETA, capacity=n_tokens)


def qwen3_layers(seed: int = 0, n_layers: int = QWEN3_LAYERS, prompt: int = 512,
                 steps: int = 256, capacity: int = 1024):
    """Qwen3-0.6B-shaped attention for n_layers independent layer instances.
    Draw order: per-layer q_norm_w, k_norm_w; prefill q, k, v [L, prompt, H, D];
    decode q, k, v [steps, L, H, D]."""
    rng = np.random.default_rng(seed)
    Hq, Hkv, D = QWEN3_N_Q_HEADS, QWEN3_N_KV_HEADS, QWEN3_HEAD_DIM
    qw = np.stack([norm_weights(rng, D) for _ in range(n_layers)])
    kw = np.stack([norm_weights(rng, D) for _ in range(n_layers)])
    return dict(
        q_norm_w=qw, k_norm_w=kw,
        q=_normal(rng, (n_layers, prompt, Hq, D)), k=_normal(rng, (n_layers, prompt, Hkv, D)),
        v=_normal(rng, (n_layers, prompt, Hkv, D)),
        dq=_normal(rng, (steps, n_layers, Hq, D)), dk=_normal(rng, (steps, n_layers, Hkv, D)),
        dv=_normal(rng, (steps, n_layers, Hkv, D)),
        prompt=prompt, steps=steps, capacity=capacity, eps=QWEN3_RMS_EPS,
        base=QWEN3_ROPE_THETA)


def lm_head_weights(seed: int = 1, vocab: int = QWEN3_VOCAB, hidden: int = QWEN3_HIDDEN,
                    std: float = 0.02):
    """Tied lm_head table [vocab, hidden] bf16 ~ N(0, std^2), as raw uint16 bits."""
    rng = np.random.default_rng(seed)
    out = np.empty((vocab, hidden), dtype=np.uint16)
    step = 16384
    for r0 in range(0, vocab, step):
        r1 = min(vocab, r0 + step)
        out[r0:r1] = f32_to_bf16_bits(std * _normal(rng, (r1 - r0, hidden)))
    return out


def hidden_states(seed: int, n: int, batch: int = 1, hidden: int = QWEN3_HIDDEN):
    """[n, batch, hidden] float32 ~ N(0,1) hidden vectors fed to the lm_head."""
    rng = np.random.default_rng(seed)
    return _normal(rng, (n, batch, hidden))


def image_span_prefill(seed: int = 0, text_before: int = 20, grid: int = 16,
                       text_after: int = 218, steps: int = 64, capacity: int = 1024):
    """VLM image-span prefill: 20 text + (1 + 16*17 + 1) image rows + 218 text = 512,
    4-axis xdRoPE positions, then `steps` decode tokens at text positions.
    Draw order: q_norm_w, k_norm_w, q, k, v, dq, dk, dv."""
    rng = np.random.default_rng(seed)
    Hq, Hkv, D = QWEN3_N_Q_HEADS, QWEN3_N_KV_HEADS, QWEN3_HEAD_DIM
    pos = image_span_positions(text_before, grid, grid, text_after)
    S = pos.shape[0]
    dpos = np.repeat(np.arange(S, S + steps, dtype=np.int32)[:, None], 4, axis=1)
    qw, kw = norm_weights(rng, D), norm_weights(rng, D)
    return dict(
        q_norm_w=qw, k_norm_w=kw,
        q=_normal(rng, (S, Hq, D)), k=_normal(rng, (S, Hkv, D)), v=_normal(rng, (S, Hkv, D)),
        dq=_normal(rng, (steps, Hq, D)), dk=_normal(rng, (steps, Hkv, D)),
        dv=_normal(rng, (steps, Hkv, D)),
        pos=pos, dpos=dpos, capacity=capacity, eps=QWEN3_RMS_EPS, base=XDROPE_BASE,
        sections=XDROPE_SECTIONS)


def vision_windowed(seed: int = 0):
    """Vision tower windowed attention on the 14x92 grid: 16 heads = 16 KV heads,
    head_dim 72, no QK-Norm, 2D RoPE (row half, col half), base 1e6.
    Draw order: q, k, v (natural token order)."""
    rng = np.random.default_rng(seed)
    lay = vision_window_layout()
    S = lay.pos_rc.shape[0]
    H, D = VISION_HEADS, VISION_HEAD_DIM
    return dict(q=_normal(rng, (S, H, D)), k=_normal(rng, (S, H, D)), v=_normal(rng, (S, H, D)),
                layout=lay, base=QWEN3_ROPE_THETA)


def serving_contexts(seed: int = 0, batch: int = 64, lo: int = 1024, hi: int = 32768):
    """Per-sequence context lengths, uniform integers in [lo, hi]."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=batch).astype(np.int32)


def serving_prefix(seed: int, b: int, ctx: int, n_kv_heads: int = QWEN3_N_KV_HEADS,
                   d: int = QWEN3_HEAD_DIM):
    """Prefix cache contents of sequence b: K, V [Hkv, ctx, D] bf16 bits of N(0,1).
    Each sequence has its own stream (seed, b) so a sample can be drawn alone."""
    rng = np.random.default_rng([seed, 7919, b])
    k = f32_to_bf16_bits(_normal(rng, (n_kv_heads, ctx, d)))
    v = f32_to_bf16_bits(_normal(rng, (n_kv_heads, ctx, d)))
    return k, v


def serving_step_inputs(seed: int, step: int, batch: int = 64):
    """Per decode step of the batched serving workload: q [B,16,128], k,v [B,8,128]
    float32 N(0,1) and the lm_head hidden [B,1024]."""
    rng = np.random.default_rng([seed, 104729, step])
    Hq, Hkv, D = QWEN3_N_Q_HEADS, QWEN3_N_KV_HEADS, QWEN3_HEAD_DIM
    return dict(q=_normal(rng, (batch, Hq, D)), k=_normal(rng, (batch, Hkv, D)),
                v=_normal(rng, (batch, Hkv, D)), h=_normal(rng, (batch, QWEN3_HIDDEN)))


def serving_norm_weights(seed: int = 0):
    rng = np.random.default_rng([seed, 31])
    return norm_weights(rng, QWEN3_HEAD_DIM), norm_weights(rng, QWEN3_HEAD_DIM)
