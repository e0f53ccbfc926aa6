"""Mutation check of the oracle's pins: each case plants one plausible slip in a scratch copy of
oracle/kv_oracle.py (a dropped term, a wrong sign, index or axis, a swapped order, a transposed
operand, an off-by-one) and runs tests/test_oracle_pins.py against that copy; every slip must
make a pin fail.  CPU only; the planted copies live in a temporary directory."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# name -> (text in the oracle, replacement)
MUTATIONS = {
    "rms_sum_not_mean": ("ms = np.mean(x * x, axis=-1, keepdims=True)", "ms = np.sum(x * x, axis=-1, keepdims=True)"),
    "eps_outside_sqrt": ("np.sqrt(ms + eps)", "(np.sqrt(ms) + eps)"),
    "dropped_norm_weight": ("return x / np.sqrt(ms + eps) * np.asarray(w, dtype=F64)", "return x / np.sqrt(ms + eps)"),
    "rope_sign": ("x1 * c - x2 * s, x2 * c + x1 * s", "x1 * c + x2 * s, x2 * c - x1 * s"),
    "frequency_exponent": ("-2.0 * j / width", "-1.0 * j / width"),
    "norm_rope_order_swapped": ("    if norm_after_rope:\n        return rms_norm(rope_apply(x, pos, rope), w, eps)",
                                "    if not norm_after_rope:\n        return rms_norm(rope_apply(x, pos, rope), w, eps)"),
    "2d_axes_swapped": ("ang = pos[:, b:b + 1] * inv[None, :]", "ang = pos[:, 1 - b:2 - b] * inv[None, :]"),
    "section_axes_reversed": ("axis_of_j = np.repeat(np.arange(len(rope.sections)), rope.sections)",
                              "axis_of_j = np.repeat(np.arange(len(rope.sections))[::-1], rope.sections)"),
    "interleave_order": ("xd = np.concatenate([x[..., 0::2], x[..., 1::2]], axis=-1)",
                         "xd = np.concatenate([x[..., 1::2], x[..., 0::2]], axis=-1)"),
    "subrange_frequencies_of_whole_head": (
        "out[..., o:o + w] = rope_apply(x[..., o:o + w], pos, Rope(rope.kind, rope.base, rope.sections))",
        "out[..., o:o + w] = rope_apply(x, pos, Rope(rope.kind, rope.base, rope.sections))[..., o:o + w]"),
    "gqa_mapping": ("g = h // G", "g = h % Hkv"),
    "strict_causal": ("return j <= i\n", "return j < i + (i == 0)\n"),
    "segment_ignored": ('        return seg[:, None] == seg[None, :]\n    if kind == "causal_segment"',
                        '        return np.ones((S, S), dtype=bool)\n    if kind == "causal_segment"'),
    "dropped_scale": ("s = (K[idx] @ q[i, h]) * scale", "s = (K[idx] @ q[i, h])"),
    "partial_max_subtraction": ("e = np.exp(s - m)", "e = np.exp(s - m * 0.5)"),
    "p_times_k": ("out[i, h] = p @ V[idx]", "out[i, h] = p @ K[idx][:, :V.shape[1]]"),
    "v_normalised_in_cache": ("cache_v[:, slot[t], :] = store(np.asarray(v[t], dtype=F64), cache_dtype)",
                              "cache_v[:, slot[t], :] = store(np.asarray(v[t], dtype=F64) / "
                              "np.linalg.norm(v[t], axis=-1, keepdims=True), cache_dtype)"),
    "truncating_bf16": ("out = np.round(x / scale) * scale", "out = np.trunc(x / scale) * scale"),
    "decode_drops_last_key": ("allowed[0, :length] = True", "allowed[0, :length - 1] = True"),
    "argmax_direction": ("i = int(np.argmax(z))", "i = int(np.argmin(z))"),
    "ties_to_highest_id": ("i = int(np.argmax(z))", "i = int(z.shape[0] - 1 - np.argmax(z[::-1]))"),
    "no_vocab_clamp": ("return np.asarray(Wf[:V], dtype=F64) @ np.asarray(h, dtype=F64)",
                       "return np.asarray(Wf, dtype=F64) @ np.asarray(h, dtype=F64)"),
    "verify_off_by_one": ("allowed[i, :length - k + i + 1] = True", "allowed[i, :length - k + i] = True"),
    "commit_off_by_one": ("return a, int(posterior[a]), length - k + a + 1", "return a, int(posterior[a]), length - k + a"),
    "topk_ties_to_highest_id": ("key=lambda v: (-z[v], v)", "key=lambda v: (-z[v], -v)"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_slip_fails_a_pin(name, tmp_path):
    src = open(os.path.join(ROOT, "oracle", "kv_oracle.py")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"{name}: the oracle text to mutate was not found exactly once"
    os.makedirs(tmp_path / "oracle")
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), tmp_path / "oracle" / "__init__.py")
    (tmp_path / "oracle" / "kv_oracle.py").write_text(src.replace(old, new))
    for d in ("tests", "workloads"):
        shutil.copytree(os.path.join(ROOT, d), tmp_path / d, ignore=shutil.ignore_patterns("__pycache__"))
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-q", "-x", "-m", "not gpu",
                        "-p", "no:cacheprovider"], cwd=tmp_path, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"{name}: every oracle pin still passes with this slip planted"
