"""ctypes binding of the C ABI in include/mla_verify_attn.h.

Argument marshalling only: every step of the verify path runs in the CUDA
kernels of libmla_verify_attn.so.  PyTorch is used to allocate device memory
and to supply the current stream.  There is no other implementation to fall
back to: if the library cannot be built or loaded, calls raise.
"""
from __future__ import annotations

import contextlib
import ctypes
import threading

from . import _build

MLA_OK = 0
STATUS_NAMES = {
    0: "MLA_OK", -1: "MLA_ERR_NULLPTR", -2: "MLA_ERR_SHAPE", -3: "MLA_ERR_ALIGN",
    -4: "MLA_ERR_WORKSPACE", -5: "MLA_ERR_UNSUPPORTED_DEVICE", -6: "MLA_ERR_LAUNCH",
    -7: "MLA_ERR_DEVICE_TIMEOUT", -8: "MLA_ERR_SEQLEN", -9: "MLA_ERR_ARG", -10: "MLA_ERR_PAGE",
}
EXPORTED = ("mla_verify_attn", "mla_verify_attn_workspace_size", "mla_verify_attn_last_device_error",
            "mla_verify_attn_strerror", "mla_verify_attn_plan", "mla_verify_attn_paged",
            "mla_verify_attn_paged_workspace_size", "mla_verify_attn_set_timing_events",
            "mla_verify_attn_set_test_controls", "mla_verify_attn_noalloc",
            "mla_verify_attn_set_two_term_max_keys")

_lock = threading.Lock()
_lib = None


class MLAError(RuntimeError):
    def __init__(self, status: int, what: str = "mla_verify_attn"):
        self.status = status
        super().__init__("%s failed: %s" % (what, strerror(status)))


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the in-tree CUDA library."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build() if build_if_missing else _build.LIB_PATH
        lib = ctypes.CDLL(path)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.mla_verify_attn.argtypes = [P, P, P, P, P, I, I, I, I, F, P, P, P, Z, P]
        lib.mla_verify_attn.restype = I
        lib.mla_verify_attn_workspace_size.argtypes = [I, I, I, I]
        lib.mla_verify_attn_workspace_size.restype = Z
        lib.mla_verify_attn_last_device_error.argtypes = [P]
        lib.mla_verify_attn_last_device_error.restype = I
        lib.mla_verify_attn_strerror.argtypes = [I]
        lib.mla_verify_attn_strerror.restype = ctypes.c_char_p
        IP = ctypes.POINTER(ctypes.c_int)
        lib.mla_verify_attn_plan.argtypes = [I, I, I, I, I, IP, IP, IP]
        lib.mla_verify_attn_plan.restype = I
        L = ctypes.c_longlong
        lib.mla_verify_attn_paged.argtypes = [P, P, P, L, P, I, I, P, P, I, I, I, F, P, P, P, Z, P]
        lib.mla_verify_attn_paged.restype = I
        lib.mla_verify_attn_paged_workspace_size.argtypes = [I, I, I, I, I]
        lib.mla_verify_attn_paged_workspace_size.restype = Z
        lib.mla_verify_attn_set_timing_events.argtypes = [P, P]
        lib.mla_verify_attn_set_timing_events.restype = I
        lib.mla_verify_attn_set_test_controls.argtypes = [I, I]
        lib.mla_verify_attn_set_test_controls.restype = I
        lib.mla_verify_attn_set_two_term_max_keys.argtypes = [I]
        lib.mla_verify_attn_set_two_term_max_keys.restype = I
        lib.mla_verify_attn_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, F, P, P, P]
        lib.mla_verify_attn_noalloc.restype = I
        _lib = lib
        return lib


def strerror(status: int) -> str:
    try:
        return load_library().mla_verify_attn_strerror(int(status)).decode()
    except OSError:
        return STATUS_NAMES.get(int(status), "status %d" % status)


def plan(B: int, q_len: int, H: int, Smax: int, max_clusters: int = 0):
    """(n_row_tiles, nsplit, chunk_tiles) the library would use."""
    a, b, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    st = load_library().mla_verify_attn_plan(B, q_len, H, Smax, max_clusters, ctypes.byref(a),
                                             ctypes.byref(b), ctypes.byref(c))
    if st != MLA_OK:
        raise MLAError(st, "mla_verify_attn_plan")
    return a.value, b.value, c.value


def workspace_size(B: int, q_len: int, H: int, Smax: int) -> int:
    return int(load_library().mla_verify_attn_workspace_size(B, q_len, H, Smax))


def paged_workspace_size(B: int, q_len: int, H: int, max_blocks: int, page_size: int) -> int:
    return int(load_library().mla_verify_attn_paged_workspace_size(B, q_len, H, max_blocks, page_size))


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def verify_attn_raw(q_nope_ptr, q_rope_ptr, kv_ptr, seq_lens_ptr, mask_ptr, B, q_len, H, Smax,
                    scale, out_ptr, lse_ptr, workspace_ptr, workspace_bytes, stream_handle) -> int:
    """Direct C-ABI call with integer device pointers; returns the status."""
    return int(load_library().mla_verify_attn(q_nope_ptr, q_rope_ptr, kv_ptr, seq_lens_ptr,
                                              mask_ptr, B, q_len, H, Smax, float(scale), out_ptr,
                                              lse_ptr, workspace_ptr, workspace_bytes,
                                              stream_handle))


def verify_attn(q_nope, q_rope, kv, seq_lens, tree_mask, scale, out=None, lse=None,
                workspace=None, stream=None):
    """Absorbed-MLA verify attention on the current CUDA device.

    q_nope [B,q,H,512] bf16, q_rope [B,q,H,64] bf16, kv [B,Smax,576] bf16,
    seq_lens [B] int32, tree_mask [B,q,ceil(q/32)] int32/uint32 bit words,
    all contiguous CUDA tensors.  Returns (out [B,q,H,512] fp32, lse [B,q,H] fp32).
    """
    import torch
    B, q, H, Dl = q_nope.shape
    Smax = kv.shape[1]
    if Dl != 512 or tuple(q_rope.shape) != (B, q, H, 64) or tuple(kv.shape) != (B, Smax, 576):
        raise ValueError("expected q_nope [B,q,H,512], q_rope [B,q,H,64], kv [B,Smax,576]")
    for name, t, dt in (("q_nope", q_nope, torch.bfloat16), ("q_rope", q_rope, torch.bfloat16),
                        ("kv", kv, torch.bfloat16), ("seq_lens", seq_lens, torch.int32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA %s tensor" % (name, dt))
    if tree_mask.element_size() != 4 or not tree_mask.is_cuda or not tree_mask.is_contiguous():
        raise ValueError("tree_mask must be a contiguous CUDA 32-bit tensor")
    dev = q_nope.device
    if out is None:
        out = torch.empty((B, q, H, 512), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, q, H), dtype=torch.float32, device=dev)
    need = workspace_size(B, q, H, Smax)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = workspace.data_ptr() if workspace is not None else 0
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = verify_attn_raw(q_nope.data_ptr(), q_rope.data_ptr(), kv.data_ptr(), seq_lens.data_ptr(),
                         tree_mask.data_ptr(), B, q, H, Smax, scale, out.data_ptr(),
                         lse.data_ptr(), ws_ptr, ws_bytes, _stream_handle(stream))
    if st != MLA_OK:
        raise MLAError(st)
    return out, lse


def verify_attn_paged(q_nope, q_rope, kv_pool, block_table, page_size, seq_lens, tree_mask, scale,
                      out=None, lse=None, workspace=None, stream=None):
    """verify_attn over a paged cache.

    kv_pool [pool_rows, 576] bf16 (pages of page_size rows), block_table
    [B, max_blocks] int32 (page of each page_size-key block of each stream),
    page_size >= 1 (multiples of 64 are read in place; other sizes are first
    copied into a contiguous cache in the workspace); other arguments as for
    verify_attn.
    """
    import torch
    B, q, H, Dl = q_nope.shape
    pool_rows = kv_pool.shape[0]
    max_blocks = block_table.shape[1]
    if Dl != 512 or tuple(q_rope.shape) != (B, q, H, 64) or kv_pool.dim() != 2 or kv_pool.shape[1] != 576:
        raise ValueError("expected q_nope [B,q,H,512], q_rope [B,q,H,64], kv_pool [rows,576]")
    if tuple(block_table.shape) != (B, max_blocks):
        raise ValueError("expected block_table [B, max_blocks]")
    for name, t, dt in (("q_nope", q_nope, torch.bfloat16), ("q_rope", q_rope, torch.bfloat16),
                        ("kv_pool", kv_pool, torch.bfloat16), ("seq_lens", seq_lens, torch.int32),
                        ("block_table", block_table, torch.int32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA %s tensor" % (name, dt))
    if tree_mask.element_size() != 4 or not tree_mask.is_cuda or not tree_mask.is_contiguous():
        raise ValueError("tree_mask must be a contiguous CUDA 32-bit tensor")
    dev = q_nope.device
    if out is None:
        out = torch.empty((B, q, H, 512), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, q, H), dtype=torch.float32, device=dev)
    need = paged_workspace_size(B, q, H, max_blocks, int(page_size))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = workspace.data_ptr() if workspace is not None else 0
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = int(load_library().mla_verify_attn_paged(
        q_nope.data_ptr(), q_rope.data_ptr(), kv_pool.data_ptr(), pool_rows, block_table.data_ptr(),
        max_blocks, int(page_size), seq_lens.data_ptr(), tree_mask.data_ptr(), B, q, H, float(scale),
        out.data_ptr(), lse.data_ptr(), ws_ptr, ws_bytes, _stream_handle(stream)))
    if st != MLA_OK:
        raise MLAError(st, "mla_verify_attn_paged")
    return out, lse


def set_timing_events(before=None, after=None) -> None:
    """Have every later call record two torch.cuda.Events around its split kernel.

    The events must already exist on the device (record each once first: torch
    creates them lazily).  ``set_timing_events()`` switches recording off.
    """
    b = 0 if before is None else int(before.cuda_event)
    a = 0 if after is None else int(after.cuda_event)
    st = int(load_library().mla_verify_attn_set_timing_events(b or None, a or None))
    if st != MLA_OK:
        raise MLAError(st, "mla_verify_attn_set_timing_events")


TWO_TERM_MAX_KEYS_DEFAULT = 4096


def set_two_term_max_keys(max_keys: int) -> None:
    """Streams of at most ``max_keys`` keys send P as two bf16 terms (exact to
    ~1e-5); longer ones send one term plus the correction of each row's
    largest-score key.  Default 4096; 0 = one term everywhere; 2**31 - 1 = two
    terms everywhere.  Process-wide, for later calls."""
    st = int(load_library().mla_verify_attn_set_two_term_max_keys(int(max_keys)))
    if st != MLA_OK:
        raise MLAError(st, "mla_verify_attn_set_two_term_max_keys")


_controls = [0, 0]   # the values last given to mla_verify_attn_set_test_controls


@contextlib.contextmanager
def forced(nsplit=None, stall=False):
    """Within the block, calls use a forced slice count (``nsplit`` > 0) and/or
    make one work unit withhold a cache load (``stall``); both are restored on
    exit.  For tests of the split/merge and timeout paths."""
    lib = load_library()
    old = list(_controls)
    new = [int(nsplit or 0), 1 if stall else 0]
    st = int(lib.mla_verify_attn_set_test_controls(*new))
    if st != MLA_OK:
        raise MLAError(st, "mla_verify_attn_set_test_controls")
    _controls[:] = new
    try:
        yield
    finally:
        lib.mla_verify_attn_set_test_controls(*old)
        _controls[:] = old


def last_device_error(stream=None) -> int:
    return int(load_library().mla_verify_attn_last_device_error(_stream_handle(stream)))
