"""ctypes binding of libfa_fwd.so: argument marshalling only.

Each function has the name of the C entry point it calls (include/fa_fwd.h).
The ``*_raw`` forms take integer device addresses and sizes exactly as the
C ABI does; the plain forms take torch tensors, check them, and pass their
pointers, shapes and the current CUDA stream. Every step of the attention
computation runs in the library's CUDA kernels; there is no fallback. If the
library is not built, the first call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa_fwd.so")
_lock = threading.Lock()
_lib = None

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4

EXPORTED = ("fa_fwd", "fa_fwd_f32", "fa_get_device_status", "fa_status_string", "fa_last_error",
            "fa_fwd_noalloc", "fa_fwd_splitkv", "fa_fwd_splitkv_workspace_bytes", "fa_fwd_splitkv_suggest",
            "fa_fwd_host", "fa_fwd_host_workspace_bytes", "fa_selftest_wait_timeout", "fa_bwd",
            "fa_bwd_workspace_bytes", "fa_fwd_f32x3", "fa_fwd_f32x3_workspace_bytes")


class FaError(RuntimeError):
    """A non-OK status from libfa_fwd.so."""

    def __init__(self, status: int, where: str):
        self.status = status
        lib = load_library()
        name = lib.fa_status_string(status).decode()
        detail = lib.fa_last_error().decode()
        super().__init__(f"{where}: {name}: {detail}")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Loads libfa_fwd.so (once) and declares the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is not built; run `python -m flashattention_fa_fwd_gb300.build` "
                "(or __graft_entry__.build()) with the CUDA 13 toolkit first")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        for name in ("fa_fwd", "fa_fwd_f32", "fa_fwd_noalloc"):
            fn = getattr(lib, name)
            fn.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, ctypes.c_float, ctypes.c_int, vp]
            fn.restype = ctypes.c_int
        lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, ctypes.c_float, ctypes.c_int,
                                        ctypes.c_int, vp, i64, vp]
        lib.fa_fwd_splitkv.restype = ctypes.c_int
        lib.fa_fwd_splitkv_workspace_bytes.argtypes = [i64, i64, i64, i64, ctypes.c_int]
        lib.fa_fwd_splitkv_workspace_bytes.restype = i64
        lib.fa_fwd_splitkv_suggest.argtypes = [i64, i64, i64, i64, ctypes.c_int]
        lib.fa_fwd_splitkv_suggest.restype = ctypes.c_int
        lib.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, ctypes.c_float, ctypes.c_int,
                                    i64, vp, i64, vp]
        lib.fa_fwd_host.restype = ctypes.c_int
        lib.fa_fwd_host_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, i64]
        lib.fa_fwd_host_workspace_bytes.restype = i64
        lib.fa_bwd.argtypes = [vp] * 9 + [i64] * 5 + [ctypes.c_float, ctypes.c_int, vp, i64, vp]
        lib.fa_bwd.restype = ctypes.c_int
        lib.fa_bwd_workspace_bytes.argtypes = [i64, i64, i64]
        lib.fa_bwd_workspace_bytes.restype = i64
        lib.fa_fwd_f32x3.argtypes = [vp] * 5 + [i64] * 5 + [ctypes.c_float, ctypes.c_int, vp, i64, vp]
        lib.fa_fwd_f32x3.restype = ctypes.c_int
        lib.fa_fwd_f32x3_workspace_bytes.argtypes = [i64, i64, i64, i64]
        lib.fa_fwd_f32x3_workspace_bytes.restype = i64
        lib.fa_selftest_wait_timeout.argtypes = [i64, vp]
        lib.fa_selftest_wait_timeout.restype = ctypes.c_int
        lib.fa_get_device_status.argtypes = [vp]
        lib.fa_get_device_status.restype = ctypes.c_int
        lib.fa_status_string.argtypes = [ctypes.c_int]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_last_error.argtypes = []
        lib.fa_last_error.restype = ctypes.c_char_p
        _lib = lib
        return lib


# ------------------------------------------------------------------ raw ABI

def fa_fwd_raw(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, M: int, N: int, D: int,
               scale: float, causal: bool, stream: int = 0) -> int:
    """Calls fa_fwd with raw device addresses; returns the status code."""
    return load_library().fa_fwd(q, k, v, o, lse, B, H, M, N, D, float(scale), int(bool(causal)), stream)


def fa_fwd_f32_raw(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, M: int, N: int, D: int,
                   scale: float, causal: bool, stream: int = 0) -> int:
    """Calls fa_fwd_f32 with raw device addresses; returns the status code."""
    return load_library().fa_fwd_f32(q, k, v, o, lse, B, H, M, N, D, float(scale), int(bool(causal)), stream)


def fa_fwd_f32x3_raw(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, M: int, N: int, D: int,
                     scale: float, causal: bool, workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    """Calls fa_fwd_f32x3 (fp32 on the tensor cores, three TF32 products)
    with raw device addresses; returns the status code."""
    return load_library().fa_fwd_f32x3(q, k, v, o, lse, B, H, M, N, D, float(scale), int(bool(causal)),
                                       workspace, int(workspace_bytes), stream)


def fa_fwd_f32x3_workspace_bytes(B: int, H: int, N: int, D: int) -> int:
    return load_library().fa_fwd_f32x3_workspace_bytes(B, H, N, D)


def fa_fwd_noalloc_raw(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, M: int, N: int, D: int,
                       scale: float, causal: bool, stream: int = 0) -> int:
    """Calls fa_fwd_noalloc (the bf16 forward whose scratch is a static
    device array, for callers that cannot allocate); returns the status.

    Calls that overlap on the GPU share that array and race. A pipeline
    timeout of this entry point stays recorded in the array's status word
    until fa_get_device_status() reads it, as for fa_fwd."""
    return load_library().fa_fwd_noalloc(q, k, v, o, lse, B, H, M, N, D, float(scale), int(bool(causal)), stream)


def fa_fwd_splitkv_raw(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, M: int, N: int, D: int,
                       scale: float, causal: bool, num_splits: int, workspace: int, workspace_bytes: int,
                       stream: int = 0) -> int:
    """Calls fa_fwd_splitkv with raw device addresses; returns the status."""
    return load_library().fa_fwd_splitkv(q, k, v, o, lse, B, H, M, N, D, float(scale), int(bool(causal)),
                                         int(num_splits), workspace, int(workspace_bytes), stream)


def fa_fwd_splitkv_workspace_bytes(B: int, H: int, M: int, D: int, num_splits: int) -> int:
    return load_library().fa_fwd_splitkv_workspace_bytes(B, H, M, D, num_splits)


def fa_fwd_splitkv_suggest(B: int, H: int, M: int, N: int, causal: bool) -> int:
    return load_library().fa_fwd_splitkv_suggest(B, H, M, N, int(bool(causal)))


def fa_fwd_host_raw(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, M: int, N: int, D: int,
                    scale: float, causal: bool, heads_per_chunk: int, workspace: int, workspace_bytes: int,
                    stream: int = 0) -> int:
    """Calls fa_fwd_host with raw host addresses and a device workspace; returns the status."""
    return load_library().fa_fwd_host(q, k, v, o, lse, B, H, M, N, D, float(scale), int(bool(causal)),
                                      int(heads_per_chunk), workspace, int(workspace_bytes), stream)


def fa_fwd_host_workspace_bytes(B: int, H: int, M: int, N: int, D: int, heads_per_chunk: int = 0) -> int:
    return load_library().fa_fwd_host_workspace_bytes(B, H, M, N, D, heads_per_chunk)


def fa_selftest_wait_timeout(limit_us: int = 20000, stream: int = 0) -> int:
    """Launches the bounded-wait self-test (a wait that nothing satisfies
    gives up after ``limit_us``); returns the launch status. Read the outcome
    with :func:`fa_get_device_status`, which should give FA_ERR_TIMEOUT."""
    return load_library().fa_selftest_wait_timeout(int(limit_us), stream)


def fa_bwd_raw(q: int, k: int, v: int, o: int, lse: int, dout: int, dq: int, dk: int, dv: int, B: int, H: int,
               M: int, N: int, D: int, scale: float, causal: bool, workspace: int, workspace_bytes: int,
               stream: int = 0) -> int:
    """Calls fa_bwd with raw device addresses; returns the status."""
    return load_library().fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, M, N, D, float(scale),
                                 int(bool(causal)), workspace, int(workspace_bytes), stream)


def fa_bwd_workspace_bytes(B: int, H: int, M: int) -> int:
    return load_library().fa_bwd_workspace_bytes(B, H, M)


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(status).decode()


def fa_last_error() -> str:
    return load_library().fa_last_error().decode()


# ------------------------------------------------------------ torch tensors

def _shape4(t, name):
    if t.dim() == 2:
        return (1, 1) + tuple(t.shape)
    if t.dim() == 4:
        return tuple(t.shape)
    raise ValueError(f"{name} must be [M, D] or [B, H, M, D], got {tuple(t.shape)}")


def _marshal(q, k, v, o, lse, dtype):
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 CUDA tensor")
    B, H, M, D = _shape4(q, "q")
    Bk, Hk, N, Dk = _shape4(k, "k")
    if (Bk, Hk, Dk) != (B, H, D) or _shape4(v, "v") != (B, H, N, D):
        raise ValueError("k and v must be [B, H, N, D] matching q's B, H and D")
    if _shape4(o, "o") != (B, H, M, D):
        raise ValueError("o must have q's shape")
    if lse.numel() != B * H * M:
        raise ValueError("lse must hold B*H*M values")
    devs = {t.device for t in (q, k, v, o, lse)}
    if len(devs) != 1:
        raise ValueError("all tensors must be on the same device")
    return B, H, M, N, D


def _stream_of(t, stream):
    import torch

    if stream is None:
        return torch.cuda.current_stream(t.device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def fa_fwd(q, k, v, o, lse, scale: float, causal: bool = False, stream=None) -> None:
    """bf16 attention forward: writes ``o`` (bf16) and ``lse`` (fp32).

    q [B, H, M, D] (or [M, D]), k and v [B, H, N, D], o like q, lse with
    B*H*M fp32 values; all contiguous CUDA tensors on one device. Runs on
    ``stream`` (default: the current torch stream) and does not synchronise.
    """
    import torch

    B, H, M, N, D = _marshal(q, k, v, o, lse, torch.bfloat16)
    with torch.cuda.device(q.device):
        st = fa_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        B, H, M, N, D, scale, causal, _stream_of(q, stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd")


def fa_fwd_f32(q, k, v, o, lse, scale: float, causal: bool = False, stream=None) -> None:
    """fp32 attention forward (CUDA cores, exact fp32): writes ``o`` and ``lse``."""
    import torch

    B, H, M, N, D = _marshal(q, k, v, o, lse, torch.float32)
    with torch.cuda.device(q.device):
        st = fa_fwd_f32_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            B, H, M, N, D, scale, causal, _stream_of(q, stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_f32")


def fa_fwd_f32x3(q, k, v, o, lse, scale: float, causal: bool = False, workspace=None, stream=None) -> None:
    """fp32 attention forward on the tensor cores (three TF32 products per
    matrix product): writes ``o`` and ``lse``. ``workspace`` is a CUDA tensor
    of at least fa_fwd_f32x3_workspace_bytes(B, H, N, D) bytes (allocated
    here with torch when None)."""
    import torch

    B, H, M, N, D = _marshal(q, k, v, o, lse, torch.float32)
    with torch.cuda.device(q.device):
        need = fa_fwd_f32x3_workspace_bytes(B, H, N, D)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        st = fa_fwd_f32x3_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              B, H, M, N, D, scale, causal, workspace.data_ptr(),
                              workspace.numel() * workspace.element_size(), _stream_of(q, stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_f32x3")


def fa_fwd_splitkv(q, k, v, o, lse, scale: float, causal: bool = False, num_splits: int = 0,
                   workspace=None, stream=None) -> None:
    """Split-KV bf16 forward (same result as :func:`fa_fwd`). ``num_splits``
    0 asks the library for a split count; ``workspace`` is a CUDA tensor of at
    least fa_fwd_splitkv_workspace_bytes(...) bytes (allocated here with torch
    when None)."""
    import torch

    B, H, M, N, D = _marshal(q, k, v, o, lse, torch.bfloat16)
    with torch.cuda.device(q.device):
        if num_splits == 0:
            num_splits = fa_fwd_splitkv_suggest(B, H, M, N, causal)
        need = fa_fwd_splitkv_workspace_bytes(B, H, M, D, num_splits)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        st = fa_fwd_splitkv_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                B, H, M, N, D, scale, causal, num_splits, workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(), _stream_of(q, stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_splitkv")


def fa_fwd_noalloc(q, k, v, o, lse, scale: float, causal: bool = False, stream=None) -> None:
    """bf16 forward like :func:`fa_fwd`, for callers that cannot allocate
    device memory: the library allocates nothing, not even on the first call
    (the kernel's scratch is a static device array shared by all calls, so
    overlapping calls on the GPU race). Make the first call on each device
    before any stream capture."""
    import torch

    B, H, M, N, D = _marshal(q, k, v, o, lse, torch.bfloat16)
    with torch.cuda.device(q.device):
        st = fa_fwd_noalloc_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                B, H, M, N, D, scale, causal, _stream_of(q, stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_noalloc")


def fa_get_device_status(stream=None, device=None) -> int:
    """Synchronises the stream and returns (and clears) the device status."""
    import torch

    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        s = torch.cuda.current_stream(dev).cuda_stream if stream is None else (
            stream if isinstance(stream, int) else stream.cuda_stream)
        return load_library().fa_get_device_status(s)


def fa_fwd_host(q, k, v, o, lse, scale: float, causal: bool = False, heads_per_chunk: int = 0,
                workspace=None, device=None, stream=None) -> None:
    """bf16 attention forward on host tensors, copies overlapped with compute.

    q, k, v, o, lse as in :func:`fa_fwd` but contiguous CPU tensors (pinned
    for the copies to overlap). ``workspace`` is a CUDA uint8 tensor of at
    least fa_fwd_host_workspace_bytes(...) bytes (allocated here with torch
    when None) on ``device`` (default: the current device). Asynchronous on
    ``stream`` (default: that device's current torch stream): synchronise it
    before reading o and lse.
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be a bfloat16 torch.Tensor")
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    if lse.dtype != torch.float32 or lse.is_cuda or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 CPU tensor")
    B, H, M, D = _shape4(q, "q")
    Bk, Hk, N, Dk = _shape4(k, "k")
    if (Bk, Hk, Dk) != (B, H, D) or _shape4(v, "v") != (B, H, N, D) or _shape4(o, "o") != (B, H, M, D):
        raise ValueError("k, v must be [B, H, N, D] and o [B, H, M, D], matching q")
    if lse.numel() != B * H * M:
        raise ValueError("lse must hold B*H*M values")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        need = fa_fwd_host_workspace_bytes(B, H, M, N, D, heads_per_chunk)
        if workspace is None:
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        s = torch.cuda.current_stream(dev).cuda_stream if stream is None else (
            stream if isinstance(stream, int) else stream.cuda_stream)
        st = fa_fwd_host_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                             B, H, M, N, D, scale, causal, heads_per_chunk, workspace.data_ptr(),
                             workspace.numel(), s)
    if st != FA_OK:
        raise FaError(st, "fa_fwd_host")


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, scale: float, causal: bool = False, workspace=None,
           stream=None) -> None:
    """Gradients of :func:`fa_fwd`: writes fp32 ``dq``, ``dk``, ``dv`` from the
    bf16 inputs ``q``, ``k``, ``v``, the forward's ``o`` (bf16) and ``lse``
    (fp32), and the bf16 output gradient ``dout``. ``workspace`` is a CUDA
    tensor of at least fa_bwd_workspace_bytes(B, H, M) bytes (allocated here
    when None)."""
    import torch

    B, H, M, N, D = _marshal(q, k, v, o, lse, torch.bfloat16)
    if dout.dtype != torch.bfloat16 or not dout.is_cuda or not dout.is_contiguous() or _shape4(dout, "dout") != (B, H, M, D):
        raise ValueError("dout must be a contiguous bf16 CUDA tensor shaped like q")
    for name, t, rows in (("dq", dq, M), ("dk", dk, N), ("dv", dv, N)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or _shape4(t, name) != (B, H, rows, D):
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of shape [B, H, {rows}, D]")
    with torch.cuda.device(q.device):
        need = fa_bwd_workspace_bytes(B, H, M)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        st = fa_bwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, M, N, D, scale, causal,
                        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_of(q, stream))
    if st != FA_OK:
        raise FaError(st, "fa_bwd")
