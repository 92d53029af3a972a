"""GB300 (sm_103a) absorbed-MLA attention for the speculative-decoding verify step.

The computation runs in hand-written CUDA kernels behind the C ABI declared in
``include/mla_verify_attn.h``; this package builds that library in-tree and
binds it with ctypes.  ``inputs`` makes seeded synthetic workloads.
"""
from ._lib import (TWO_TERM_MAX_KEYS_DEFAULT, MLAError, forced, last_device_error, load_library,
                   paged_workspace_size, plan, set_timing_events, set_two_term_max_keys, strerror,
                   verify_attn, verify_attn_paged, verify_attn_raw, workspace_size)
from ._build import build

__all__ = ["TWO_TERM_MAX_KEYS_DEFAULT", "MLAError", "build", "forced", "last_device_error", "load_library",
           "paged_workspace_size", "plan", "set_timing_events", "set_two_term_max_keys", "strerror",
           "verify_attn", "verify_attn_paged", "verify_attn_raw", "workspace_size"]
