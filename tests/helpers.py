"""Shared test utilities: tensor marshalling between numpy inputs and the CUDA path, and the
comparison metrics the contract states (per-row relative L2, max abs, cosine)."""
import numpy as np

import workloads as WL


def torch():
    import torch as _t
    return _t


def dev(x, dtype=None):
    """numpy -> CUDA tensor (float32 unless dtype given; uint16 arrays are raw bf16 bits)."""
    t = torch()
    if isinstance(x, np.ndarray) and x.dtype == np.uint16:
        return t.from_numpy(x.view(np.int16).copy()).cuda().view(t.bfloat16)
    a = t.from_numpy(np.ascontiguousarray(x)).cuda()
    return a if dtype is None else a.to(dtype)


def host(t_):
    """CUDA tensor -> float64 numpy (bf16 widened exactly)."""
    t = torch()
    return t_.detach().to(t.float64).cpu().numpy()


def bf16_bits(t_):
    t = torch()
    return t_.detach().view(t.int16).cpu().numpy().view(np.uint16)


def row_rel_err(a, b):
    """Max over rows (last axis) of ||a - b|| / ||b||."""
    a = np.asarray(a, np.float64).reshape(-1, a.shape[-1])
    b = np.asarray(b, np.float64).reshape(-1, b.shape[-1])
    num = np.linalg.norm(a - b, axis=1)
    den = np.maximum(np.linalg.norm(b, axis=1), 1e-300)
    return float(np.max(num / den))


def row_cos_min(a, b):
    a = np.asarray(a, np.float64).reshape(-1, a.shape[-1])
    b = np.asarray(b, np.float64).reshape(-1, b.shape[-1])
    c = np.sum(a * b, axis=1) / (np.linalg.norm(a, axis=1) * np.linalg.norm(b, axis=1) + 1e-12)
    return float(np.min(c))


def max_abs(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))


# Tolerances stated by the contract for this path.
FP32_ROW_REL = 1e-5            # fp32 configs: max relative error per output row
BF16_MAX_ABS = 2e-2            # bf16-cache configs: max abs error on unit-scale outputs
BF16_COS_MIN = 0.9999          # bf16-cache configs: cosine per row
ARGMAX_MARGIN = 1e-3           # argmax must match where top1 - top2 exceeds this


def assert_fp32_close(gpu, ref, what=""):
    e = row_rel_err(gpu, ref)
    assert e <= FP32_ROW_REL, f"{what}: max row rel err {e:.3e} > {FP32_ROW_REL}"


def assert_bf16_close(gpu, ref, what=""):
    ma = max_abs(gpu, ref)
    cs = row_cos_min(gpu, ref)
    assert ma <= BF16_MAX_ABS and cs >= BF16_COS_MIN, f"{what}: max abs {ma:.3e}, min cos {cs:.6f}"


def assert_bf16_store(gpu_bits, exact, what="", slack=2e-6):
    """A value stored in bf16 from an fp32 intermediate: within one bf16 ulp of the exact
    (float64) value plus an absolute slack for the fp32 arithmetic, taken relative to the
    row's RMS (cancellation in x*cos - y*sin can leave an element far below the row scale,
    where a 1e-7 absolute fp32 error spans several bf16 ulps)."""
    g = WL.bf16_bits_to_f32(gpu_bits).astype(np.float64)
    e = np.asarray(exact, np.float64)
    assert g.shape == e.shape, (g.shape, e.shape)
    rms = np.sqrt(np.mean(e * e, axis=-1, keepdims=True))
    ulp = np.ldexp(1.0, np.floor(np.log2(np.maximum(np.abs(e), 1e-300))).astype(int) - 7)
    err = np.abs(g - e)
    bad = err > ulp + slack * rms
    assert not np.any(bad), f"{what}: {int(bad.sum())} stored values off by more than 1 ulp + {slack} rms " \
                            f"(worst {float(np.max(err - ulp - slack * rms)):.3e})"


def bf16_ulp_diff(gpu_bits, ref_vals):
    """Max difference in bf16 ulps between stored bf16 bits and oracle bf16 values."""
    ref_bits = WL.f32_to_bf16_bits(np.asarray(ref_vals, np.float32))
    def key(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return int(np.max(np.abs(key(gpu_bits) - key(ref_bits))))
