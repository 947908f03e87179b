"""ctypes binding of libssd_scan.so (argument marshalling only).

Every function here has the name of the C entry point it calls (include/ssd_scan.h).  Torch
is used for device memory and the current stream; all computation happens in the library's
CUDA kernels.  If the library is missing the import of a function fails loudly: there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssd_scan.so")

SSD_F32, SSD_BF16 = 0, 1
SSD_OK, SSD_ERR_INVALID, SSD_ERR_UNSUPPORTED, SSD_ERR_CUDA, SSD_ERR_TIMEOUT, SSD_ERR_WORKSPACE = range(6)
SSD_PATH_AUTO, SSD_PATH_CHUNKED, SSD_PATH_TC = -1, 0, 1
PATH_NAMES = {SSD_PATH_CHUNKED: "chunked", SSD_PATH_TC: "tc"}

_lib = None
_lock = threading.Lock()


class ssd_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("nheads", ctypes.c_int64), ("headdim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
                ("dtype", ctypes.c_int32)]


class SSDError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {ssd_scan_strerror(code)} (code {code})")


def load_library(path: str = LIB_PATH):
    """Load libssd_scan.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"libssd_scan.so not built at {path}; run __graft_entry__.build() "
                              "or python -m mamba_ssd_scan_05_b300.build")
        lib = ctypes.CDLL(path)
        vp, sz, i32, fp = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p
        dims_p = ctypes.POINTER(ssd_dims)
        lib.ssd_scan_resolve_path.argtypes = [dims_p, i32, i32]
        lib.ssd_scan_resolve_path.restype = i32
        lib.ssd_scan_workspace_bytes.argtypes = [dims_p, i32, i32]
        lib.ssd_scan_workspace_bytes.restype = sz
        lib.ssd_scan_kernels_per_call.argtypes = [dims_p, i32, i32]
        lib.ssd_scan_kernels_per_call.restype = i32
        fwd_args = [dims_p, vp, vp, fp, vp, vp, fp, fp, i32, vp, fp, vp, sz, vp]
        lib.ssd_scan_fwd.argtypes = fwd_args
        lib.ssd_scan_fwd.restype = i32
        lib.ssd_scan_fwd_path.argtypes = fwd_args + [i32]
        lib.ssd_scan_fwd_path.restype = i32
        lib.ssd_scan_host_arena_bytes.argtypes = [dims_p, i32]
        lib.ssd_scan_host_arena_bytes.restype = sz
        lib.ssd_scan_fwd_host.argtypes = fwd_args
        lib.ssd_scan_fwd_host.restype = i32
        lib.ssd_step_fwd.argtypes = [dims_p, vp, vp, fp, vp, vp, fp, fp, fp, vp, vp]
        lib.ssd_step_fwd.restype = i32
        i64 = ctypes.c_int64
        lib.ssd_causal_conv1d_fwd.argtypes = [i64, i64, i64, i32, i32, vp, fp, fp, vp, vp, i32,
                                              vp, vp]
        lib.ssd_causal_conv1d_fwd.restype = i32
        lib.ssd_gated_rmsnorm_fwd.argtypes = [i64, i64, i64, i32, vp, vp, fp, ctypes.c_float,
                                              vp, vp]
        lib.ssd_gated_rmsnorm_fwd.restype = i32
        cu_p = ctypes.POINTER(ctypes.c_int64)
        lib.ssd_scan_varlen_workspace_bytes.argtypes = [dims_p, cu_p, i64, i32, i32]
        lib.ssd_scan_varlen_workspace_bytes.restype = sz
        lib.ssd_scan_fwd_varlen.argtypes = [dims_p, cu_p, i64, vp, vp, fp, vp, vp, fp, fp, i32,
                                            vp, fp, vp, sz, vp, i32]
        lib.ssd_scan_fwd_varlen.restype = i32
        lib.ssd_scan_get_status.argtypes = [vp, vp]
        lib.ssd_scan_get_status.restype = i32
        lib.ssd_scan_gated_workspace_bytes.argtypes = [dims_p, i32, i64]
        lib.ssd_scan_gated_workspace_bytes.restype = sz
        lib.ssd_scan_fwd_gated.argtypes = [dims_p, vp, vp, fp, vp, vp, fp, fp, i32, vp, fp,
                                           ctypes.c_float, i64, vp, fp, vp, sz, vp]
        lib.ssd_scan_fwd_gated.restype = i32
        lib.ssd_scan_set_wait_cycles.argtypes = [ctypes.c_int64]
        lib.ssd_block_get_status.argtypes = [ctypes.c_void_p]
        lib.ssd_block_get_status.restype = i32
        lib.ssd_scan_set_wait_cycles.restype = ctypes.c_int64
        lib.ssd_scan_strerror.argtypes = [i32]
        lib.ssd_scan_strerror.restype = ctypes.c_char_p
        lib.ssd_scan_version.argtypes = []
        lib.ssd_scan_version.restype = i32
        _lib = lib
        return lib


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return SSD_F32
    if t == torch.bfloat16:
        return SSD_BF16
    raise TypeError(f"ssd_scan: unsupported element type {t} (float32 or bfloat16)")


def make_dims(x: torch.Tensor, B: torch.Tensor) -> ssd_dims:
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    return ssd_dims(b, L, H, P, N, G, _dtype_code(x.dtype))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def ssd_scan_strerror(code: int) -> str:
    return load_library().ssd_scan_strerror(int(code)).decode()


def ssd_scan_version() -> int:
    return load_library().ssd_scan_version()


def ssd_scan_resolve_path(dims: ssd_dims, chunk_size: int, path: int = SSD_PATH_AUTO) -> int:
    return load_library().ssd_scan_resolve_path(ctypes.byref(dims), int(chunk_size), int(path))


def ssd_scan_workspace_bytes(dims: ssd_dims, chunk_size: int, path: int = SSD_PATH_AUTO) -> int:
    return load_library().ssd_scan_workspace_bytes(ctypes.byref(dims), int(chunk_size), int(path))


def ssd_scan_kernels_per_call(dims: ssd_dims, chunk_size: int, path: int = SSD_PATH_AUTO) -> int:
    """Kernels one ssd_scan_fwd call enqueues on the current device (negative: an SSD_ERR_*)."""
    return load_library().ssd_scan_kernels_per_call(ctypes.byref(dims), int(chunk_size), int(path))


def _check_inputs(x, dt, A, B, C, D, initial_state):
    if x.dim() != 4 or dt.dim() != 3 or B.dim() != 4 or C.dim() != 4:
        raise ValueError("ssd_scan: x [b,L,H,P], dt [b,L,H], B/C [b,L,G,N] expected")
    b, L, H, P = x.shape
    if dt.shape != (b, L, H) or B.shape[:2] != (b, L) or C.shape != B.shape:
        raise ValueError("ssd_scan: inconsistent shapes")
    for name, t in (("dt", dt), ("B", B), ("C", C)):
        if t.dtype != x.dtype:
            raise TypeError(f"ssd_scan: {name} must have x's dtype {x.dtype}")
    if A.shape != (H,) or A.dtype != torch.float32:
        raise ValueError("ssd_scan: A must be float32 [H]")
    if D is not None and (D.shape != (H,) or D.dtype != torch.float32):
        raise ValueError("ssd_scan: D must be float32 [H]")
    N = B.shape[3]
    if initial_state is not None and (initial_state.shape != (b, H, P, N)
                                      or initial_state.dtype != torch.float32):
        raise ValueError("ssd_scan: initial_state must be float32 [b,H,P,N]")
    for t in (x, dt, A, B, C, D, initial_state):
        if t is not None and not t.is_contiguous():
            raise ValueError("ssd_scan: tensors must be contiguous")


def ssd_scan_fwd(x, dt, A, B, C, D=None, initial_state=None, chunk_size: int = 256,
                 path: int = SSD_PATH_AUTO, y=None, final_state=None, workspace=None,
                 return_final_state: bool = True):
    """y, final_state = scan(x, dt, A, B, C, D, initial_state) on x's CUDA device.

    Enqueued on torch's current stream; outputs (and the workspace, unless given) are
    allocated with torch.  A given workspace smaller than ssd_scan_workspace_bytes raises
    SSDError(SSD_ERR_WORKSPACE).  Raises SSDError on any non-zero return code.
    """
    _check_inputs(x, dt, A, B, C, D, initial_state)
    if not x.is_cuda:
        raise ValueError("ssd_scan_fwd: tensors must be on a CUDA device (see ssd_scan_fwd_host)")
    lib = load_library()
    dims = make_dims(x, B)
    b, L, H, P = x.shape
    N = B.shape[3]
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_final_state:
        final_state = torch.empty((b, H, P, N), dtype=torch.float32, device=x.device)
    need = lib.ssd_scan_workspace_bytes(ctypes.byref(dims), int(chunk_size), int(path))
    if need == 0:
        rc = lib.ssd_scan_resolve_path(ctypes.byref(dims), int(chunk_size), int(path))
        raise SSDError(-rc if rc < 0 else SSD_ERR_INVALID, "ssd_scan_workspace_bytes")
    # a workspace the caller passes is used as it is: one that is too small comes back from
    # the library as SSD_ERR_WORKSPACE (replacing it would hide the call's status word)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    args = (ctypes.byref(dims), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
            _ptr(initial_state), int(chunk_size), _ptr(y), _ptr(final_state), _ptr(workspace),
            workspace.numel(), _stream_handle(x.device))
    if path == SSD_PATH_AUTO:
        rc = lib.ssd_scan_fwd(*args)
    else:
        rc = lib.ssd_scan_fwd_path(*args, int(path))
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_scan_fwd")
    return y, final_state


def ssd_scan_gated_workspace_bytes(dims: ssd_dims, chunk_size: int, group_size: int) -> int:
    return load_library().ssd_scan_gated_workspace_bytes(ctypes.byref(dims), int(chunk_size),
                                                         int(group_size))


def ssd_scan_fwd_gated(x, dt, A, B, C, z, D=None, initial_state=None, norm_weight=None,
                       eps: float = 1e-5, group_size=None, chunk_size: int = 256, out=None,
                       final_state=None, workspace=None, return_final_state: bool = True):
    """out, final_state = gated_rmsnorm(scan(x, dt, A, B, C, D, initial_state), z).

    out[..., f] = y / sqrt(mean over f's group of y^2 + eps) * norm_weight[f] * silu(z), with
    f = h * P + p and groups of ``group_size`` consecutive features (default: one head,
    ``P``).  Fused into the scan kernel where it can be (see include/ssd_scan.h).
    """
    _check_inputs(x, dt, A, B, C, D, initial_state)
    if not x.is_cuda:
        raise ValueError("ssd_scan_fwd_gated: tensors must be on a CUDA device")
    if z.shape != x.shape or z.dtype != x.dtype or not z.is_contiguous():
        raise ValueError("ssd_scan_fwd_gated: z must be shaped, typed and laid out like x")
    b, L, H, P = x.shape
    N = B.shape[3]
    if norm_weight is not None and (norm_weight.shape != (H * P,)
                                    or norm_weight.dtype != torch.float32
                                    or not norm_weight.is_contiguous()):
        raise ValueError("ssd_scan_fwd_gated: norm_weight must be contiguous float32 [H * P]")
    g = P if group_size is None else int(group_size)
    lib = load_library()
    dims = make_dims(x, B)
    if out is None:
        out = torch.empty_like(x)
    if final_state is None and return_final_state:
        final_state = torch.empty((b, H, P, N), dtype=torch.float32, device=x.device)
    need = lib.ssd_scan_gated_workspace_bytes(ctypes.byref(dims), int(chunk_size), g)
    if need == 0:
        raise SSDError(SSD_ERR_INVALID, "ssd_scan_gated_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    rc = lib.ssd_scan_fwd_gated(ctypes.byref(dims), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                _ptr(D), _ptr(initial_state), int(chunk_size), _ptr(z),
                                _ptr(norm_weight), float(eps), g, _ptr(out), _ptr(final_state),
                                _ptr(workspace), workspace.numel(), _stream_handle(x.device))
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_scan_fwd_gated")
    return out, final_state


def _cu_array(cu_seqlens):
    vals = [int(v) for v in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    return (ctypes.c_int64 * len(vals))(*vals), len(vals) - 1


def ssd_scan_varlen_workspace_bytes(dims: ssd_dims, cu_seqlens, chunk_size: int,
                                    path: int = SSD_PATH_AUTO) -> int:
    cu, nseq = _cu_array(cu_seqlens)
    return load_library().ssd_scan_varlen_workspace_bytes(ctypes.byref(dims), cu, nseq,
                                                          int(chunk_size), int(path))


def ssd_scan_fwd_varlen(x, dt, A, B, C, cu_seqlens, D=None, initial_states=None,
                        chunk_size: int = 256, path: int = SSD_PATH_AUTO, y=None,
                        final_states=None, workspace=None, return_final_states: bool = True):
    """The scan over a packed batch: x [1, total, H, P] (and dt, B, C alike) holds the
    sequences back to back, sequence i being tokens cu_seqlens[i] .. cu_seqlens[i+1] - 1 (a
    host list or CPU tensor).  Each sequence starts from initial_states[i] (or zeros).
    Returns (y, final_states [nseq, H, P, N])."""
    if x.dim() != 4 or x.shape[0] != 1:
        raise ValueError("ssd_scan_fwd_varlen: x must be [1, total, H, P]")
    _check_inputs(x, dt, A, B, C, D, None)
    if not x.is_cuda:
        raise ValueError("ssd_scan_fwd_varlen: tensors must be on a CUDA device")
    cu, nseq = _cu_array(cu_seqlens)
    _, L, H, P = x.shape
    N = B.shape[3]
    if initial_states is not None and (initial_states.shape != (nseq, H, P, N)
                                       or initial_states.dtype != torch.float32
                                       or not initial_states.is_contiguous()):
        raise ValueError("ssd_scan_fwd_varlen: initial_states must be float32 [nseq,H,P,N]")
    lib = load_library()
    dims = make_dims(x, B)
    if y is None:
        y = torch.empty_like(x)
    if final_states is None and return_final_states:
        final_states = torch.empty((nseq, H, P, N), dtype=torch.float32, device=x.device)
    need = lib.ssd_scan_varlen_workspace_bytes(ctypes.byref(dims), cu, nseq, int(chunk_size),
                                               int(path))
    if need == 0:
        raise SSDError(SSD_ERR_INVALID, "ssd_scan_varlen_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    rc = lib.ssd_scan_fwd_varlen(ctypes.byref(dims), cu, nseq, _ptr(x), _ptr(dt), _ptr(A),
                                 _ptr(B), _ptr(C), _ptr(D), _ptr(initial_states),
                                 int(chunk_size), _ptr(y), _ptr(final_states), _ptr(workspace),
                                 workspace.numel(), _stream_handle(x.device), int(path))
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_scan_fwd_varlen")
    return y, final_states


def ssd_step_fwd(x, dt, A, B, C, D=None, state=None, state_out=None, y=None):
    """One recurrent step (a single token per sequence) on x's CUDA device.

    x [b,1,H,P] or [b,H,P]; dt [b,1,H] or [b,H]; B, C [b,1,G,N] or [b,G,N]; A, D float32 [H];
    state float32 [b,H,P,N] or None (zeros).  The new state goes to ``state_out``: by default
    ``state`` itself (updated in place), or a new tensor when ``state`` is None.  Returns
    (y, state_out) with y shaped like x.  Enqueued on torch's current stream.
    """
    squeeze = x.dim() == 3
    if squeeze:
        x, dt, B, C = x.unsqueeze(1), dt.unsqueeze(1), B.unsqueeze(1), C.unsqueeze(1)
    _check_inputs(x, dt, A, B, C, D, state)
    if x.shape[1] != 1:
        raise ValueError("ssd_step_fwd: one token per sequence (seqlen 1)")
    if not x.is_cuda:
        raise ValueError("ssd_step_fwd: tensors must be on a CUDA device")
    b, _, H, P = x.shape
    N = B.shape[3]
    if state_out is None:
        state_out = state if state is not None else torch.empty(
            (b, H, P, N), dtype=torch.float32, device=x.device)
    elif (state_out.shape != (b, H, P, N) or state_out.dtype != torch.float32
          or not state_out.is_contiguous()):
        raise ValueError("ssd_step_fwd: state_out must be contiguous float32 [b,H,P,N]")
    if y is None:
        y = torch.empty_like(x)
    rc = load_library().ssd_step_fwd(ctypes.byref(make_dims(x, B)), _ptr(x), _ptr(dt), _ptr(A),
                                     _ptr(B), _ptr(C), _ptr(D), _ptr(state), _ptr(state_out),
                                     _ptr(y), _stream_handle(x.device))
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_step_fwd")
    return (y.squeeze(1) if squeeze else y), state_out


def ssd_causal_conv1d_fwd(x, weight, bias=None, state=None, silu: bool = True,
                          return_state: bool = False, out=None, state_out=None):
    """Depthwise causal conv1d (+ SiLU) over x [b, L, C] on its CUDA device.

    weight float32 [C, K] (K <= 8), bias float32 [C] or None, state [b, K-1, C] (x's dtype) or
    None (zeros).  Returns out [b, L, C], or (out, state_out) with ``return_state``.
    """
    if x.dim() != 3 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("ssd_causal_conv1d_fwd: x must be a contiguous CUDA tensor [b, L, C]")
    b, L, C = x.shape
    if weight.dim() != 2 or weight.shape[0] != C or weight.dtype != torch.float32:
        raise ValueError("ssd_causal_conv1d_fwd: weight must be float32 [C, K]")
    K = weight.shape[1]
    if bias is not None and (bias.shape != (C,) or bias.dtype != torch.float32):
        raise ValueError("ssd_causal_conv1d_fwd: bias must be float32 [C]")
    if state is not None and (state.shape != (b, K - 1, C) or state.dtype != x.dtype):
        raise ValueError("ssd_causal_conv1d_fwd: state must be [b, K-1, C] of x's dtype")
    for t in (weight, bias, state):
        if t is not None and not t.is_contiguous():
            raise ValueError("ssd_causal_conv1d_fwd: tensors must be contiguous")
    if out is None:
        out = torch.empty_like(x)
    if return_state and state_out is None:
        state_out = torch.empty((b, K - 1, C), dtype=x.dtype, device=x.device)
    rc = load_library().ssd_causal_conv1d_fwd(b, L, C, K, _dtype_code(x.dtype), _ptr(x),
                                              _ptr(weight), _ptr(bias), _ptr(state),
                                              _ptr(state_out), int(bool(silu)), _ptr(out),
                                              _stream_handle(x.device))
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_causal_conv1d_fwd")
    return (out, state_out) if return_state else out


def ssd_gated_rmsnorm_fwd(y, z=None, weight=None, eps: float = 1e-5, group_size=None, out=None):
    """rmsnorm(y) * weight * silu(z) over the last dimension (in groups of ``group_size``)."""
    if not y.is_cuda or not y.is_contiguous():
        raise ValueError("ssd_gated_rmsnorm_fwd: y must be a contiguous CUDA tensor")
    D = y.shape[-1]
    rows = y.numel() // D if D else 0
    if z is not None and (z.shape != y.shape or z.dtype != y.dtype or not z.is_contiguous()):
        raise ValueError("ssd_gated_rmsnorm_fwd: z must match y")
    if weight is not None and (weight.shape != (D,) or weight.dtype != torch.float32):
        raise ValueError("ssd_gated_rmsnorm_fwd: weight must be float32 [D]")
    g = D if group_size is None else int(group_size)
    if out is None:
        out = torch.empty_like(y)
    rc = load_library().ssd_gated_rmsnorm_fwd(rows, D, g, _dtype_code(y.dtype), _ptr(y), _ptr(z),
                                              _ptr(weight), float(eps), _ptr(out),
                                              _stream_handle(y.device))
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_gated_rmsnorm_fwd")
    return out


def ssd_scan_get_status(workspace, device=None) -> int:
    """Synchronise the current stream and return (and clear) the workspace status word."""
    lib = load_library()
    return lib.ssd_scan_get_status(_ptr(workspace), _stream_handle(device or workspace.device))


def ssd_block_get_status(device=None) -> int:
    """Synchronise the current stream of ``device`` and return (and clear) the status word of the
    streaming conv1d / RMSNorm kernels (SSD_OK, or SSD_ERR_TIMEOUT after a wait gave up)."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    return lib.ssd_block_get_status(_stream_handle(dev))


def ssd_scan_set_wait_cycles(cycles: int) -> int:
    """Limit of each device-side wait of the tensor-core kernels, in SM cycles (<= 0: the
    default).  Process-wide; returns the previous limit."""
    return load_library().ssd_scan_set_wait_cycles(int(cycles))


def ssd_scan_host_arena_bytes(dims: ssd_dims, chunk_size: int) -> int:
    return load_library().ssd_scan_host_arena_bytes(ctypes.byref(dims), int(chunk_size))


def ssd_scan_fwd_host(x, dt, A, B, C, D=None, initial_state=None, chunk_size: int = 256,
                      y=None, final_state=None, arena=None, device=None):
    """The host-buffer entry point: CPU tensors in and out (pinned memory recommended).

    Copies in, scans and copies out on the current stream of ``device`` and synchronises it
    before returning.  ``arena`` (a CUDA uint8 tensor) is used when given; one smaller than
    ssd_scan_host_arena_bytes raises SSDError(SSD_ERR_WORKSPACE).
    """
    _check_inputs(x, dt, A, B, C, D, initial_state)
    if x.is_cuda:
        raise ValueError("ssd_scan_fwd_host: tensors must be host tensors")
    device = torch.device(device or "cuda")
    lib = load_library()
    dims = make_dims(x, B)
    b, L, H, P = x.shape
    N = B.shape[3]
    if y is None:
        y = torch.empty_like(x, pin_memory=True)
    if final_state is None:
        final_state = torch.empty((b, H, P, N), dtype=torch.float32, pin_memory=True)
    need = lib.ssd_scan_host_arena_bytes(ctypes.byref(dims), int(chunk_size))
    if need == 0:
        raise SSDError(SSD_ERR_INVALID, "ssd_scan_host_arena_bytes")
    if arena is None:
        arena = torch.empty(need, dtype=torch.uint8, device=device)
    stream = _stream_handle(device)
    rc = lib.ssd_scan_fwd_host(ctypes.byref(dims), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                               _ptr(D), _ptr(initial_state), int(chunk_size), _ptr(y),
                               _ptr(final_state), _ptr(arena), arena.numel(), stream)
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_scan_fwd_host")
    torch.cuda.current_stream(device).synchronize()
    return y, final_state
