"""GB300-native KV-cache GQA attention step: a C-ABI CUDA library (libkv_attn.so, sources in
csrc/, ABI in include/kv_attn.h) and its thin Python binding.

Entry points (same names as the C ABI):
  kv_cache_append_rope_qknorm  fused QK-Norm + RoPE + K/V cache write
  kv_attn_prefill              flash-style parallel prefill (causal / full / window segments)
  kv_attn_decode               split-KV single-token decode
  kv_attn_decode_step          the append of the new token and the decode in one launch
  kv_attn_verify               a speculative-decoding block: k query rows, causal inside the block
  kv_verify_commit             acceptance of the block's draft tokens and the cache-length commit
  lmhead_argmax                tied lm_head GEMV + greedy argmax (lowest id on ties)
  lmhead_topk                  final RMSNorm + lm_head, the k best ids (k = 1: fused greedy argmax)
"""
from .kv_attn import (KVCache, KvaError, Rope, decode_workspace_bytes, kv_attn_decode,  # noqa: F401
                      kv_attn_decode_step, kv_attn_verify, kv_verify_commit, verify_workspace_bytes,
                      kv_attn_prefill, kv_cache_append_rope_qknorm, launch_count, lib,
                      lmhead_argmax, lmhead_topk, lmhead_topk_workspace_bytes, lmhead_workspace_bytes,
                      version, wait_timeouts, workspace_bytes, PreparedCall, prepare_decode_step,
                      prepare_lmhead_argmax)
