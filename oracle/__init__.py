"""CPU oracle (test infrastructure): plain float64 definition of the KV-cache GQA
attention step.  Only tests, the smoke check and the benchmark's CPU baseline use it.

Every function here is pinned by the `-m "not gpu"` tests against closed forms,
invariants, library routines, brute force on tiny inputs and values the pages print.
"""
from .kv_oracle import *  # noqa: F401,F403
