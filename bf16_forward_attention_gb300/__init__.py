"""GB300-native bf16 forward attention.

The product is the C ABI in ``include/attn_fwd.h`` (library
``_lib/libattn_fwd.so``, built by ``build.py``). This module is the thin Python
binding: it checks tensors, marshals pointers and sizes, and calls the library on
the current torch stream. Every step of the computation runs in the CUDA kernel;
there is no Python or CPU fallback - if the library is missing, calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os

from .build import lib_path

LAYOUTS = {"bhsd": 0, "bshd": 1}
ROUNDINGS = {"rtne": 0, "rtna": 1, "rtz": 2}

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_MISALIGNED = -3
ATTN_ERR_ALIASING = -4
ATTN_ERR_NO_DEVICE = -5
ATTN_ERR_ARCH = -6
ATTN_ERR_LAUNCH = -7
ATTN_ERR_TIMEOUT = -8
ATTN_ERR_TOO_LARGE = -9
ATTN_ERR_SCRATCH = -10
ATTN_ERR_SEQLENS = -11
ATTN_ERR_DEBUG_CHECK = -12
ATTN_FLAG_CAUSAL = 1
ATTN_FLAG_SPLIT_TAIL = 2

_libs: dict = {}


class AttnError(RuntimeError):
    """A nonzero status from the C library."""

    def __init__(self, status: int, msg: str):
        super().__init__(f"attn_fwd failed ({status}): {msg}")
        self.status = status


def load_library(debug: bool | None = None) -> ctypes.CDLL:
    """Load ``libattn_fwd.so``, or its debug flavour ``libattn_fwd_debug.so`` when
    ``debug`` (default: the environment variable ATTN_FWD_DEBUG=1). Raises if the
    library has not been built."""
    if debug is None:
        debug = os.environ.get("ATTN_FWD_DEBUG") == "1"
    if debug in _libs:
        return _libs[debug]
    path = lib_path(debug)
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library not built: {path} is missing. Run "
            f"`python -m bf16_forward_attention_gb300.build{' --debug' if debug else ''}` (needs nvcc).")
    lib = ctypes.CDLL(path)
    i64 = ctypes.c_int64
    lib.attn_fwd.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, i64, i64, i64, i64, i64,
                                                     ctypes.c_float, ctypes.c_int, ctypes.c_void_p]
    lib.attn_fwd.restype = ctypes.c_int
    lib.attn_status_str.argtypes = [ctypes.c_int]
    lib.attn_status_str.restype = ctypes.c_char_p
    lib.attn_fwd_last_error.argtypes = []
    lib.attn_fwd_last_error.restype = ctypes.c_int
    lib.attn_fwd_version.argtypes = []
    lib.attn_fwd_version.restype = ctypes.c_int
    lib.attn_fwd_timeout_selftest.argtypes = lib.attn_fwd.argtypes + [ctypes.c_uint64, ctypes.c_int]
    lib.attn_fwd_timeout_selftest.restype = ctypes.c_int
    lib.attn_fwd_splitkv.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, i64, i64, i64, i64, i64,
                                                             ctypes.c_float, ctypes.c_int,
                                                             ctypes.c_int, ctypes.c_void_p, i64,
                                                             ctypes.c_void_p]
    lib.attn_fwd_splitkv.restype = ctypes.c_int
    lib.attn_fwd_splitkv_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, ctypes.c_int]
    lib.attn_fwd_splitkv_workspace_bytes.restype = i64
    lib.attn_fwd_split_tail_items.argtypes = [i64, i64, i64, i64]
    lib.attn_fwd_split_tail_items.restype = ctypes.c_int
    lib.attn_fwd_splitkv_num_splits.argtypes = [i64, i64, i64, i64]
    lib.attn_fwd_splitkv_num_splits.restype = ctypes.c_int
    lib.attn_fwd_splitkv_noalloc.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, i64, i64, i64,
                                                                     i64, i64, ctypes.c_float,
                                                                     ctypes.c_int, ctypes.c_int,
                                                                     ctypes.c_void_p]
    lib.attn_fwd_splitkv_noalloc.restype = ctypes.c_int
    lib.attn_fwd_ex.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, i64, i64, i64, i64, i64, i64,
                                                        ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                                        ctypes.c_void_p]
    lib.attn_fwd_ex.restype = ctypes.c_int
    lib.attn_fwd_varlen.argtypes = ([ctypes.c_void_p] * 6 + [i64] * 7
                                    + [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p])
    lib.attn_fwd_varlen.restype = ctypes.c_int
    lib.attn_fwd_host_workspace_bytes.argtypes = [i64] * 6
    lib.attn_fwd_host_workspace_bytes.restype = i64
    lib.attn_fwd_host.argtypes = ([ctypes.c_void_p] * 4 + [ctypes.c_int] + [i64] * 6
                                  + [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, i64,
                                     ctypes.c_void_p])
    lib.attn_fwd_host.restype = ctypes.c_int
    lib.attn_fwd_varlen_host_workspace_bytes.argtypes = [i64] * 6
    lib.attn_fwd_varlen_host_workspace_bytes.restype = i64
    lib.attn_fwd_varlen_host.argtypes = ([ctypes.c_void_p] * 6 + [i64] * 6
                                         + [ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_void_p, i64, ctypes.c_void_p])
    lib.attn_fwd_varlen_host.restype = ctypes.c_int
    lib.attn_fwd_debug_build.argtypes = []
    lib.attn_fwd_debug_build.restype = ctypes.c_int
    lib.attn_fwd_debug_selftest.argtypes = lib.attn_fwd.argtypes
    lib.attn_fwd_debug_selftest.restype = ctypes.c_int
    _libs[debug] = lib
    return lib


def status_str(status: int) -> str:
    return load_library().attn_status_str(int(status)).decode()


def attn_fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, layout: int, B: int, H: int,
                 Sq: int, Sk: int, d: int, scale: float, rounding_mode: int, stream: int) -> int:
    """Direct call of the C entry point ``attn_fwd``; returns its status code."""
    return load_library().attn_fwd(q_ptr, k_ptr, v_ptr, out_ptr, layout, B, H, Sq, Sk, d,
                                   ctypes.c_float(scale), rounding_mode, stream)


def attn_fwd_timeout_selftest_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, layout: int,
                                  B: int, H: int, Sq: int, Sk: int, d: int, scale: float,
                                  rounding_mode: int, stream: int, timeout_ns: int,
                                  flags: int = 0) -> int:
    """Direct call of ``attn_fwd_timeout_selftest`` (a launch whose device-side
    wait must time out; see include/attn_fwd.h)."""
    return load_library().attn_fwd_timeout_selftest(q_ptr, k_ptr, v_ptr, out_ptr, layout, B, H, Sq,
                                                    Sk, d, ctypes.c_float(scale), rounding_mode,
                                                    stream, timeout_ns, flags)


def attn_fwd_splitkv_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, layout: int, B: int,
                         H: int, Sq: int, Sk: int, d: int, scale: float, rounding_mode: int,
                         num_splits: int, workspace_ptr: int, workspace_bytes: int,
                         stream: int) -> int:
    """Direct call of the C entry point ``attn_fwd_splitkv``; returns its status."""
    return load_library().attn_fwd_splitkv(q_ptr, k_ptr, v_ptr, out_ptr, layout, B, H, Sq, Sk, d,
                                           ctypes.c_float(scale), rounding_mode, num_splits,
                                           workspace_ptr, workspace_bytes, stream)


def attn_fwd_splitkv_noalloc_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, layout: int,
                                 B: int, H: int, Sq: int, Sk: int, d: int, scale: float,
                                 rounding_mode: int, num_splits: int, stream: int) -> int:
    """Direct call of ``attn_fwd_splitkv_noalloc``: split-KV whose workspace is the
    library's fixed device scratch array, for callers that cannot allocate device
    memory (see include/attn_fwd.h). Returns its status code."""
    return load_library().attn_fwd_splitkv_noalloc(q_ptr, k_ptr, v_ptr, out_ptr, layout, B, H, Sq,
                                                   Sk, d, ctypes.c_float(scale), rounding_mode,
                                                   num_splits, stream)


def splitkv_workspace_bytes(B: int, H: int, Sq: int, Sk: int, num_splits: int, d: int = 128) -> int:
    n = load_library().attn_fwd_splitkv_workspace_bytes(B, H, Sq, Sk, d, num_splits)
    if n < 0:
        raise AttnError(int(n), status_str(int(n)))
    return int(n)


def splitkv_num_splits(B: int, H: int, Sq: int, Sk: int) -> int:
    n = load_library().attn_fwd_splitkv_num_splits(B, H, Sq, Sk)
    if n < 0:
        raise AttnError(int(n), status_str(int(n)))
    return int(n)


def attn_fwd_splitkv(q, k, v, *, num_splits: int | None = None, layout: str = "bhsd",
                     scale: float | None = None, rounding: str = "rtne", out=None,
                     workspace=None):
    """attn_fwd with the key range split over several CTAs (see include/attn_fwd.h).

    ``workspace``: a CUDA tensor of at least ``splitkv_workspace_bytes(...)`` bytes;
    allocated here if not given (the C entry point itself never allocates).
    """
    import torch

    if layout not in LAYOUTS or rounding not in ROUNDINGS:
        raise ValueError("unknown layout or rounding mode")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a bf16 CUDA tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D tensor")
    B, H, Sq, D = _dims(q, layout)
    Bk, Hk, Sk, Dk = _dims(k, layout)
    if (Bk, Hk, Dk) != (B, H, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on one device")
    if num_splits is None:
        num_splits = splitkv_num_splits(B, H, Sq, Sk)
    need = splitkv_workspace_bytes(B, H, Sq, Sk, num_splits, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_workspace(workspace, q.device)
    if out is None:
        out = torch.empty_like(q)
    _check_out(out, q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with _on_device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        st = attn_fwd_splitkv_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  LAYOUTS[layout], B, H, Sq, Sk, D, float(scale),
                                  ROUNDINGS[rounding], num_splits, workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(), stream)
    if st != ATTN_OK:
        raise AttnError(st, status_str(st))
    return out


def split_tail_items(B: int, Hq: int, Sq: int, Sk: int) -> int:
    """Items of an ``attn_fwd_ex(..., split_tail=True)`` call of this size that run on
    pairs of CTAs on the current device (0: the flag changes nothing), or a negative
    status (see include/attn_fwd.h)."""
    return load_library().attn_fwd_split_tail_items(B, Hq, Sq, Sk)


def attn_fwd_ex_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, layout: int, B: int, Hq: int,
                    Hkv: int, Sq: int, Sk: int, d: int, scale: float, rounding_mode: int,
                    flags: int, stream: int) -> int:
    """Direct call of ``attn_fwd_ex`` (grouped-query heads, causal flag)."""
    return load_library().attn_fwd_ex(q_ptr, k_ptr, v_ptr, out_ptr, layout, B, Hq, Hkv, Sq, Sk, d,
                                      ctypes.c_float(scale), rounding_mode, flags, stream)


def attn_fwd_ex(q, k, v, *, causal: bool = False, layout: str = "bhsd",
                scale: float | None = None, rounding: str = "rtne", out=None,
                split_tail: bool = False):
    """attn_fwd with grouped-query heads (k, v may have fewer heads than q, a divisor
    of q's) and an optional causal mask aligned at the bottom right.

    ``split_tail``: run the items of the last, partial wave on pairs of CTAs, each
    taking half of the key range (ATTN_FLAG_SPLIT_TAIL; no effect with the mask).
    Faster when that wave is short, but an item's bits then depend on the size
    of the call."""
    import torch

    if layout not in LAYOUTS or rounding not in ROUNDINGS:
        raise ValueError("unknown layout or rounding mode")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a bf16 CUDA tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D tensor")
    B, Hq, Sq, D = _dims(q, layout)
    Bk, Hkv, Sk, Dk = _dims(k, layout)
    if (Bk, Dk) != (B, D) or tuple(v.shape) != tuple(k.shape) or Hq % Hkv:
        raise ValueError("shape mismatch")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on one device")
    if out is None:
        out = torch.empty_like(q)
    _check_out(out, q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with _on_device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        st = attn_fwd_ex_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                             LAYOUTS[layout], B, Hq, Hkv, Sq, Sk, D, float(scale),
                             ROUNDINGS[rounding],
                             (ATTN_FLAG_CAUSAL if causal else 0)
                             | (ATTN_FLAG_SPLIT_TAIL if split_tail else 0), stream)
    if st != ATTN_OK:
        raise AttnError(st, status_str(st))
    return out


def attn_fwd_varlen_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, cu_q_ptr: int,
                        cu_k_ptr: int, B: int, Hq: int, Hkv: int, total_q: int, total_k: int,
                        max_seqlen_q: int, d: int, scale: float, rounding_mode: int, flags: int,
                        stream: int) -> int:
    """Direct call of ``attn_fwd_varlen`` (packed variable-length batch)."""
    return load_library().attn_fwd_varlen(q_ptr, k_ptr, v_ptr, out_ptr, cu_q_ptr, cu_k_ptr, B, Hq,
                                          Hkv, total_q, total_k, max_seqlen_q, d,
                                          ctypes.c_float(scale), rounding_mode, flags, stream)


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, *,
                    causal: bool = False, scale: float | None = None, rounding: str = "rtne",
                    out=None):
    """Attention over a packed batch of variable-length sequences.

    q: (total_q, Hq, 128), k and v: (total_k, Hkv, 128), bf16 CUDA tensors packed
    token after token; cu_seqlens_q / cu_seqlens_k: int32 CUDA tensors of B + 1
    offsets; max_seqlen_q: a bound on every sequence's query count. Invalid
    offsets are found on the device: check ``attn_fwd_last_error()`` after a sync.
    """
    import torch

    if rounding not in ROUNDINGS:
        raise ValueError("unknown rounding mode")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a bf16 CUDA tensor")
        if t.dim() != 3 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous (tokens, heads, d) tensor")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if (not isinstance(t, torch.Tensor) or t.dtype != torch.int32 or not t.is_cuda
                or t.dim() != 1 or not t.is_contiguous()):
            raise TypeError(f"{name} must be a contiguous 1-D int32 CUDA tensor")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both have B + 1 >= 2 entries")
    total_q, Hq, D = q.shape
    total_k, Hkv, Dk = k.shape
    if Dk != D or tuple(v.shape) != tuple(k.shape) or Hq % Hkv:
        raise ValueError("shape mismatch")
    if not (q.device == k.device == v.device == cu_seqlens_q.device == cu_seqlens_k.device):
        raise ValueError("q, k, v and the offsets must be on one device")
    if out is None:
        out = torch.empty_like(q)
    _check_out(out, q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with _on_device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        st = attn_fwd_varlen_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                 cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
                                 cu_seqlens_q.numel() - 1, Hq, Hkv, total_q, total_k,
                                 int(max_seqlen_q), D, float(scale), ROUNDINGS[rounding],
                                 ATTN_FLAG_CAUSAL if causal else 0, stream)
    if st != ATTN_OK:
        raise AttnError(st, status_str(st))
    return out


def host_workspace_bytes(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, d: int = 128) -> int:
    """Device workspace attn_fwd_host needs (negative: a status code)."""
    return load_library().attn_fwd_host_workspace_bytes(B, Hq, Hkv, Sq, Sk, d)


def attn_fwd_host_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, layout: int, B: int,
                      Hq: int, Hkv: int, Sq: int, Sk: int, d: int, scale: float,
                      rounding_mode: int, flags: int, workspace_ptr: int, workspace_bytes: int,
                      stream: int) -> int:
    """Direct call of ``attn_fwd_host`` (host buffers, copies overlapped)."""
    return load_library().attn_fwd_host(q_ptr, k_ptr, v_ptr, out_ptr, layout, B, Hq, Hkv, Sq, Sk,
                                        d, ctypes.c_float(scale), rounding_mode, flags,
                                        workspace_ptr, workspace_bytes, stream)


def attn_fwd_host(q, k, v, *, causal: bool = False, layout: str = "bhsd",
                  scale: float | None = None, rounding: str = "rtne", out=None, workspace=None,
                  device=None):
    """attn_fwd_ex on CPU tensors (pinned for overlap): uploads, computes and
    downloads in overlapped chunks on ``device`` and returns ``out`` (a CPU
    tensor, pinned when allocated here). The call is asynchronous on the
    current stream: synchronize before reading ``out``, and keep q, k, v (and a
    caller-given workspace) alive until then."""
    import torch

    if layout not in LAYOUTS or rounding not in ROUNDINGS:
        raise ValueError("unknown layout or rounding mode")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.is_cuda:
            raise TypeError(f"{name} must be a bf16 CPU tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D tensor")
    B, Hq, Sq, D = _dims(q, layout)
    Bk, Hkv, Sk, Dk = _dims(k, layout)
    if (Bk, Dk) != (B, D) or tuple(v.shape) != tuple(k.shape) or Hq % Hkv:
        raise ValueError("shape mismatch")
    if out is not None:
        _check_out(out, q)
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    need = host_workspace_bytes(B, Hq, Hkv, Sq, Sk, D)
    if need < 0:
        raise AttnError(need, status_str(need))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    _check_workspace(workspace, torch.device(device))
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    _check_out(out, q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with _on_device(device):
        stream = torch.cuda.current_stream(device).cuda_stream
        st = attn_fwd_host_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               LAYOUTS[layout], B, Hq, Hkv, Sq, Sk, D, float(scale),
                               ROUNDINGS[rounding], ATTN_FLAG_CAUSAL if causal else 0,
                               workspace.data_ptr(), workspace.numel(), stream)
    if st != ATTN_OK:
        raise AttnError(st, status_str(st))
    return out


def attn_fwd_varlen_host(q, k, v, cu_seqlens_q, cu_seqlens_k, *, causal: bool = False,
                         scale: float | None = None, rounding: str = "rtne", out=None,
                         workspace=None, device=None):
    """attn_fwd_varlen on CPU tensors (pinned for overlap): q (total_q, Hq, 128),
    k and v (total_k, Hkv, 128) bf16, cu_seqlens_q / cu_seqlens_k int32 CPU
    tensors of B + 1 offsets. Uploads, computes and downloads in overlapped chunks
    of whole sequences on ``device``; returns ``out`` (CPU). Asynchronous on the
    current stream: synchronize before reading ``out``."""
    import torch

    if rounding not in ROUNDINGS:
        raise ValueError("unknown rounding mode")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.is_cuda:
            raise TypeError(f"{name} must be a bf16 CPU tensor")
        if t.dim() != 3 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous (tokens, heads, d) tensor")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if (not isinstance(t, torch.Tensor) or t.dtype != torch.int32 or t.is_cuda
                or t.dim() != 1 or not t.is_contiguous()):
            raise TypeError(f"{name} must be a contiguous 1-D int32 CPU tensor")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both have B + 1 >= 2 entries")
    total_q, Hq, D = q.shape
    total_k, Hkv, Dk = k.shape
    if Dk != D or tuple(v.shape) != tuple(k.shape) or Hq % Hkv:
        raise ValueError("shape mismatch")
    if out is not None:
        _check_out(out, q)
    B = cu_seqlens_q.numel() - 1
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    need = load_library().attn_fwd_varlen_host_workspace_bytes(B, Hq, Hkv, total_q, total_k, D)
    if need < 0:
        raise AttnError(int(need), status_str(int(need)))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    _check_workspace(workspace, torch.device(device))
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with _on_device(device):
        stream = torch.cuda.current_stream(device).cuda_stream
        st = load_library().attn_fwd_varlen_host(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), cu_seqlens_q.data_ptr(),
            cu_seqlens_k.data_ptr(), B, Hq, Hkv, total_q, total_k, D, ctypes.c_float(float(scale)),
            ROUNDINGS[rounding], ATTN_FLAG_CAUSAL if causal else 0, workspace.data_ptr(),
            workspace.numel(), stream)
    if st != ATTN_OK:
        raise AttnError(st, status_str(st))
    return out


def attn_fwd_last_error() -> int:
    return load_library().attn_fwd_last_error()


def _on_device(device):
    """The device context for a library call: none when `device` is already the
    current CUDA device (entering torch.cuda.device costs a few microseconds, a
    noticeable share of a small call)."""
    import contextlib

    import torch

    if torch.cuda.current_device() == device.index:
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def _dims(x, layout):
    if layout == "bhsd":
        B, H, S, D = x.shape
    else:
        B, S, H, D = x.shape
    return B, H, S, D


def _check_out(out, q):
    """The C library writes through out's pointer: it must be a contiguous bf16
    tensor shaped like q, on q's device (CUDA or host)."""
    import torch

    if (not isinstance(out, torch.Tensor) or out.dtype != torch.bfloat16
            or out.shape != q.shape or not out.is_contiguous() or out.device != q.device):
        raise ValueError("out must be a contiguous bf16 tensor shaped like q on q's device")


def _check_workspace(ws, device):
    import torch

    if not isinstance(ws, torch.Tensor) or not ws.is_cuda or ws.device != device or not ws.is_contiguous():
        raise ValueError(f"workspace must be a contiguous CUDA tensor on {device}")


def attn_fwd(q, k, v, *, layout: str = "bhsd", scale: float | None = None,
             rounding: str = "rtne", out=None):
    """O = softmax(Q K^T * scale) V on bf16 CUDA tensors (head_dim 128).

    q: (B, H, Sq, 128) for "bhsd" or (B, Sq, H, 128) for "bshd"; k, v likewise with
    Sk. Returns ``out`` (allocated like q if not given) in the same layout, rounded
    to bf16 per ``rounding`` ("rtne", "rtna", "rtz"). Runs on the current stream.
    """
    import torch

    if layout not in LAYOUTS:
        raise ValueError(f"layout must be one of {sorted(LAYOUTS)}")
    if rounding not in ROUNDINGS:
        raise ValueError(f"rounding must be one of {sorted(ROUNDINGS)}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a bf16 CUDA tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D tensor")
    B, H, Sq, D = _dims(q, layout)
    Bk, Hk, Sk, Dk = _dims(k, layout)
    if (Bk, Hk, Dk) != (B, H, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on one device")
    if out is None:
        out = torch.empty_like(q)
    elif (out.dtype != torch.bfloat16 or out.shape != q.shape or not out.is_contiguous()
          or out.device != q.device):
        raise ValueError("out must be a contiguous bf16 tensor shaped like q on q's device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with _on_device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        st = attn_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                          LAYOUTS[layout], B, H, Sq, Sk, D, float(scale), ROUNDINGS[rounding],
                          stream)
    if st != ATTN_OK:
        raise AttnError(st, status_str(st))
    return out


__all__ = ["attn_fwd", "attn_fwd_raw", "attn_fwd_last_error", "attn_fwd_timeout_selftest_raw",
           "attn_fwd_splitkv", "attn_fwd_splitkv_raw", "splitkv_workspace_bytes",
           "splitkv_num_splits", "attn_fwd_splitkv_noalloc_raw", "attn_fwd_ex", "attn_fwd_ex_raw",
           "attn_fwd_varlen", "attn_fwd_varlen_raw", "ATTN_ERR_SEQLENS",
           "attn_fwd_host", "attn_fwd_host_raw", "host_workspace_bytes", "attn_fwd_varlen_host", "status_str", "load_library",
           "AttnError", "LAYOUTS", "ROUNDINGS", "lib_path", "ATTN_ERR_DEBUG_CHECK",
           "ATTN_FLAG_CAUSAL", "ATTN_FLAG_SPLIT_TAIL", "split_tail_items"]
