"""Thin Python binding of the C ABI in include/fa.h (argument marshalling only).

Every step of the attention forward pass runs in the CUDA library
``libfa.so``; this module only checks tensor metadata, passes raw device
pointers and the current CUDA stream, and turns status codes into
exceptions. There is no fallback: if the library is missing, every call
raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4

#: every symbol include/fa.h declares
EXPORTED = ("fa_fwd", "fa_get_device_status", "fa_status_string", "fa_last_cuda_error", "fa_fwd_fault_test",
            "fa_naive_fwd", "fa_naive_workspace_bytes", "fa_naive_fwd_noalloc", "fa_bwd", "fa_bwd_workspace_bytes",
            "fa_bwd_fault_test", "fa_fwd_kv", "fa_fwd_kv_num_splits", "fa_fwd_kv_workspace_bytes",
            "fa_fwd_kv_fault_test", "fa_merge_partials", "fa_fwd_host", "fa_fwd_host_workspace_bytes",
            "fa_fwd_kv_f32", "fa_fwd_kv_f32_workspace_bytes", "fa_fwd_launch_shape")

_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {fa_status_string(status)}"
        if status == FA_ERR_CUDA:
            msg += f" (cudaError {fa_last_cuda_error()})"
        super().__init__(msg)


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libfa.so (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with exact_io_aware_34_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i, f, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_ulonglong
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, vp]
    lib.fa_fwd.restype = i
    lib.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, ctypes.c_size_t, vp]
    lib.fa_fwd_host.restype = i
    lib.fa_fwd_host_workspace_bytes.argtypes = [i, i, i, i]
    lib.fa_fwd_host_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_fwd_fault_test.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, u64, vp]
    lib.fa_fwd_fault_test.restype = i
    lib.fa_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
    lib.fa_get_device_status.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_last_cuda_error.argtypes = []
    lib.fa_last_cuda_error.restype = i
    lib.fa_naive_workspace_bytes.argtypes = [i, i, i]
    lib.fa_naive_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_naive_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, vp, ctypes.c_size_t, vp]
    lib.fa_naive_fwd.restype = i
    lib.fa_naive_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, vp]
    lib.fa_naive_fwd_noalloc.restype = i
    lib.fa_bwd_workspace_bytes.argtypes = [i, i, i]
    lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, vp, ctypes.c_size_t, vp]
    lib.fa_bwd.restype = i
    lib.fa_bwd_fault_test.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, vp, ctypes.c_size_t, i, u64,
                                      vp]
    lib.fa_bwd_fault_test.restype = i
    lib.fa_fwd_kv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, ctypes.c_size_t, vp]
    lib.fa_fwd_kv.restype = i
    lib.fa_fwd_kv_fault_test.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, ctypes.c_size_t, i, u64, vp]
    lib.fa_fwd_kv_fault_test.restype = i
    lib.fa_fwd_kv_num_splits.argtypes = [i, i, i, i, i, i]
    lib.fa_fwd_kv_num_splits.restype = i
    lib.fa_fwd_kv_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
    lib.fa_fwd_kv_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_fwd_kv_f32.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, ctypes.c_size_t, vp]
    lib.fa_fwd_kv_f32.restype = i
    lib.fa_fwd_kv_f32_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
    lib.fa_fwd_kv_f32_workspace_bytes.restype = ctypes.c_size_t
    ip = ctypes.POINTER(ctypes.c_int)
    lib.fa_fwd_launch_shape.argtypes = [i, i, i, i, ip, ip, ip]
    lib.fa_fwd_launch_shape.restype = i
    lib.fa_merge_partials.argtypes = [vp, vp, vp, vp, i, ctypes.c_longlong, i, vp]
    lib.fa_merge_partials.restype = i
    _lib = lib
    return lib


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def fa_last_cuda_error() -> int:
    return int(load_library().fa_last_cuda_error())


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check_qkv(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16, got {t.dtype}")
        if t.dim() != 4:
            raise ValueError(f"{name} must be [B, H, N, d]")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if not (q.shape == k.shape == v.shape):
        raise ValueError(f"q, k, v shapes differ: {tuple(q.shape)} {tuple(k.shape)} {tuple(v.shape)}")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on the same device")


def fa_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor | None = None,
           lse: torch.Tensor | None = None, scale: float | None = None, stream=None):
    """O = softmax(scale * q k^T) v and LSE, by one launch of the fused kernel.

    q, k, v: bf16 CUDA tensors [B, H, N, d], contiguous. ``o`` (bf16 [B,H,N,d])
    and ``lse`` (float32 [B,H,N]) are allocated with torch when not given.
    ``scale`` defaults to 1/sqrt(d). Enqueued on ``stream`` (default: torch's
    current stream for q's device). Returns (o, lse).
    """
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if o.dtype != torch.bfloat16 or o.shape != q.shape or not o.is_contiguous() or o.device != q.device:
        raise ValueError("o must be a contiguous bf16 tensor shaped like q on q's device")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous() \
            or lse.device != q.device:
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor on q's device")
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        B, H, N, d, float(scale), _stream_handle(stream, q.device))
    if st != FA_OK:
        raise FaError(st, "fa_fwd")
    return o, lse


def fa_fwd_host_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().fa_fwd_host_workspace_bytes(int(B), int(H), int(N), int(d)))


def fa_fwd_host(qh: torch.Tensor, kh: torch.Tensor, vh: torch.Tensor, oh: torch.Tensor | None = None,
                lseh: torch.Tensor | None = None, scale: float | None = None, num_chunks: int = 0, workspace=None,
                device=None, stream=None):
    """fa_fwd on host tensors, end to end (upload, kernel, download, pipelined
    over head groups by the library).

    qh, kh, vh: bf16 CPU tensors [B, H, N, d], contiguous (pinned for full copy
    bandwidth). ``oh`` / ``lseh`` (CPU, allocated pinned when not given) receive
    O and LSE. ``workspace``: a CUDA uint8 tensor of at least
    fa_fwd_host_workspace_bytes(B, H, N, d) bytes on ``device`` (default: the
    current CUDA device), allocated with torch when None. The call is
    asynchronous on ``stream``: synchronise it before reading ``oh`` and
    ``lseh``. Returns (oh, lseh).
    """
    for x in (qh, kh, vh):
        if x.device.type != "cpu" or x.dtype != torch.bfloat16 or not x.is_contiguous() or x.dim() != 4:
            raise ValueError("qh, kh, vh must be contiguous bf16 CPU tensors [B, H, N, d]")
    if not (qh.shape == kh.shape == vh.shape):
        raise ValueError("qh, kh, vh must have the same shape")
    B, H, N, d = qh.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if oh is None:
        oh = torch.empty(qh.shape, dtype=torch.bfloat16).pin_memory()
    if lseh is None:
        lseh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    if oh.device.type != "cpu" or oh.dtype != torch.bfloat16 or oh.shape != qh.shape or not oh.is_contiguous():
        raise ValueError("oh must be a contiguous bf16 CPU tensor shaped like qh")
    if lseh.device.type != "cpu" or lseh.dtype != torch.float32 or tuple(lseh.shape) != (B, H, N) \
            or not lseh.is_contiguous():
        raise ValueError("lseh must be a contiguous float32 CPU tensor [B, H, N]")
    need = fa_fwd_host_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    lib = load_library()
    with torch.cuda.device(dev):
        st = lib.fa_fwd_host(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), oh.data_ptr(), lseh.data_ptr(), B, H, N, d,
                             float(scale), int(num_chunks), workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), _stream_handle(stream, dev))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_host")
    return oh, lseh


def fa_naive_workspace_bytes(B: int, H: int, N: int) -> int:
    return int(load_library().fa_naive_workspace_bytes(int(B), int(H), int(N)))


def fa_naive_fwd(q, k, v, o=None, lse=None, scale: float | None = None, workspace=None, stream=None):
    """Standard attention with S and P materialised in ``workspace`` (the
    comparator of the fused kernel). ``workspace`` is a CUDA tensor of at least
    fa_naive_workspace_bytes(B, H, N) bytes; allocated with torch when None.
    Returns (o, lse)."""
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    need = fa_naive_workspace_bytes(B, H, N)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.fa_naive_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                              float(scale), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                              _stream_handle(stream, q.device))
    if st != FA_OK:
        raise FaError(st, "fa_naive_fwd")
    return o, lse


def fa_fwd_launch_shape(B: int, H: int, N: int, d: int) -> tuple:
    """(grid, cluster, whole_units) of the launch fa_fwd makes for these sizes
    on the current device: cluster is 1, or 2 when CTA pairs share the units
    of the last, partial round."""
    grid, cluster, whole = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    st = load_library().fa_fwd_launch_shape(int(B), int(H), int(N), int(d), ctypes.byref(grid),
                                            ctypes.byref(cluster), ctypes.byref(whole))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_launch_shape")
    return grid.value, cluster.value, whole.value


def fa_fwd_kv_num_splits(B: int, H: int, H_kv: int, N_q: int, N_kv: int, d: int) -> int:
    return int(load_library().fa_fwd_kv_num_splits(int(B), int(H), int(H_kv), int(N_q), int(N_kv), int(d)))


def fa_fwd_kv_workspace_bytes(B: int, H: int, H_kv: int, N_q: int, N_kv: int, d: int, num_splits: int = 0) -> int:
    return int(load_library().fa_fwd_kv_workspace_bytes(int(B), int(H), int(H_kv), int(N_q), int(N_kv), int(d),
                                                         int(num_splits)))


def _check_kv(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4 \
                or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor [B, heads, N, d]")
    if k.shape != v.shape or q.shape[0] != k.shape[0] or q.shape[3] != k.shape[3]:
        raise ValueError(f"shapes do not match: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on the same device")


def fa_fwd_kv(q, k, v, o=None, lse=None, scale: float | None = None, num_splits: int = 0, workspace=None,
              stream=None):
    """O = softmax(scale q k^T) v with shared K/V heads and any N_q, N_kv.

    q: bf16 [B, H, N_q, d]; k, v: bf16 [B, H_kv, N_kv, d] with H a multiple of
    H_kv (query head h uses K/V head h // (H // H_kv)). Returns (o, lse).
    ``num_splits`` = 0 lets the library choose the key split (none when the
    fused forward kernel fills the device; see :func:`fa_fwd_kv_num_splits`),
    1 forbids one; the workspace is allocated with torch when needed and not
    given.
    """
    _check_kv(q, k, v)
    B, H, N_q, d = q.shape
    H_kv, N_kv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N_q), dtype=torch.float32, device=q.device)
    need = fa_fwd_kv_workspace_bytes(B, H, H_kv, N_q, N_kv, d, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.fa_fwd_kv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, H_kv, N_q,
                           N_kv, d, float(scale), int(num_splits), ws_ptr, ws_bytes, _stream_handle(stream, q.device))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_kv")
    return o, lse


def fa_fwd_kv_f32_workspace_bytes(B: int, H: int, H_kv: int, N_q: int, N_kv: int, d: int,
                                  num_splits: int = 0) -> int:
    return int(load_library().fa_fwd_kv_f32_workspace_bytes(int(B), int(H), int(H_kv), int(N_q), int(N_kv), int(d),
                                                             int(num_splits)))


def fa_fwd_kv_f32(q, k, v, o=None, lse=None, scale: float | None = None, num_splits: int = 0, workspace=None,
                  stream=None):
    """:func:`fa_fwd_kv` with o returned in float32 (normalised, not rounded):
    the partial result of one key shard that a sequence split exchanges.
    Returns (o float32 [B, H, N_q, d], lse float32 [B, H, N_q])."""
    _check_kv(q, k, v)
    B, H, N_q, d = q.shape
    H_kv, N_kv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty((B, H, N_q, d), dtype=torch.float32, device=q.device)
    if o.dtype != torch.float32 or tuple(o.shape) != (B, H, N_q, d) or not o.is_contiguous():
        raise ValueError("o must be a contiguous float32 [B, H, N_q, d] tensor")
    if lse is None:
        lse = torch.empty((B, H, N_q), dtype=torch.float32, device=q.device)
    need = fa_fwd_kv_f32_workspace_bytes(B, H, H_kv, N_q, N_kv, d, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.fa_fwd_kv_f32(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, H_kv,
                               N_q, N_kv, d, float(scale), int(num_splits), ws_ptr, ws_bytes,
                               _stream_handle(stream, q.device))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_kv_f32")
    return o, lse


def fa_fwd_kv_fault_test(q, k, v, o, lse, scale: float, num_splits: int, workspace, drop_load: int,
                         timeout_ns: int, stream=None) -> int:
    """Test hook of the C ABI (see include/fa.h): returns the raw status code."""
    _check_kv(q, k, v)
    B, H, N_q, d = q.shape
    lib = load_library()
    with torch.cuda.device(q.device):
        return int(lib.fa_fwd_kv_fault_test(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, k.shape[1], N_q, k.shape[2],
            d, float(scale), int(num_splits), workspace.data_ptr() if workspace is not None else None,
            workspace.numel() * workspace.element_size() if workspace is not None else 0, int(drop_load),
            int(timeout_ns), _stream_handle(stream, q.device)))


def fa_merge_partials(o_parts: torch.Tensor, lse_parts: torch.Tensor, o=None, lse=None, stream=None):
    """Merge partial results over disjoint key sets (see include/fa.h).

    o_parts: float32 CUDA [P, ..., d]; lse_parts: float32 CUDA [P, ...] with the
    same leading shape. Returns (o bf16 [..., d], lse float32 [...]).
    """
    for name, t in (("o_parts", o_parts), ("lse_parts", lse_parts)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    if o_parts.shape[:-1] != lse_parts.shape or o_parts.dim() < 3:
        raise ValueError(f"shapes do not match: {tuple(o_parts.shape)} vs {tuple(lse_parts.shape)}")
    P, d = o_parts.shape[0], o_parts.shape[-1]
    out_shape = tuple(o_parts.shape[1:])
    rows = int(lse_parts[0].numel())
    if o is None:
        o = torch.empty(out_shape, dtype=torch.bfloat16, device=o_parts.device)
    if lse is None:
        lse = torch.empty(out_shape[:-1], dtype=torch.float32, device=o_parts.device)
    lib = load_library()
    with torch.cuda.device(o_parts.device):
        st = lib.fa_merge_partials(o_parts.data_ptr(), lse_parts.data_ptr(), o.data_ptr(), lse.data_ptr(), int(P), rows,
                                   int(d), _stream_handle(stream, o_parts.device))
    if st != FA_OK:
        raise FaError(st, "fa_merge_partials")
    return o, lse


def fa_bwd_workspace_bytes(B: int, H: int, N: int) -> int:
    return int(load_library().fa_bwd_workspace_bytes(int(B), int(H), int(N)))


def fa_bwd(q, k, v, o, do, lse, dq=None, dk=None, dv=None, scale: float | None = None, workspace=None,
           stream=None):
    """Gradients (dq, dk, dv) of <do, o> for o = softmax(scale * q k^T) v, with
    the probabilities rebuilt from the forward's ``lse`` and ``o``.

    q, k, v, o, do: bf16 CUDA tensors [B, H, N, d], contiguous; lse: float32
    [B, H, N]. Outputs (bf16, shaped like q) and the workspace (at least
    fa_bwd_workspace_bytes(B, H, N) bytes) are allocated with torch when not
    given. ``scale`` defaults to 1/sqrt(d). Returns (dq, dk, dv).
    """
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    for name, t in (("o", o), ("do", do)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.shape != q.shape \
                or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q on q's device")
    if not isinstance(lse, torch.Tensor) or lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) \
            or not lse.is_contiguous() or lse.device != q.device:
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor on q's device")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    outs = []
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        if t is None:
            t = torch.empty_like(q)
        elif t.dtype != torch.bfloat16 or t.shape != q.shape or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q on q's device")
        outs.append(t)
    need = fa_bwd_workspace_bytes(B, H, N)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                        outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(), B, H, N, d, float(scale),
                        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                        _stream_handle(stream, q.device))
    if st != FA_OK:
        raise FaError(st, "fa_bwd")
    return tuple(outs)


def fa_bwd_fault_test(q, k, v, o, do, lse, dq, dk, dv, scale: float, workspace, drop_load: int, timeout_ns: int,
                      stream=None) -> int:
    """Test hook of the C ABI (see include/fa.h): returns the raw status code."""
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    lib = load_library()
    with torch.cuda.device(q.device):
        return int(lib.fa_bwd_fault_test(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                         lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                                         float(scale), workspace.data_ptr(),
                                         workspace.numel() * workspace.element_size(), int(drop_load),
                                         int(timeout_ns), _stream_handle(stream, q.device)))


def fa_fwd_fault_test(q, k, v, o, lse, scale: float, drop_load: int, timeout_ns: int, stream=None) -> int:
    """Test hook of the C ABI (see include/fa.h): returns the raw status code."""
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    lib = load_library()
    with torch.cuda.device(q.device):
        return int(lib.fa_fwd_fault_test(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                         B, H, N, d, float(scale), int(drop_load), int(timeout_ns),
                                         _stream_handle(stream, q.device)))


def fa_get_device_status(stream=None, device=None):
    """Synchronise the stream and read/clear the device status word: (status, info[4])."""
    lib = load_library()
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    info = (ctypes.c_uint * 4)()
    with torch.cuda.device(device):
        st = lib.fa_get_device_status(_stream_handle(stream, device), info)
    return int(st), [int(x) for x in info]
