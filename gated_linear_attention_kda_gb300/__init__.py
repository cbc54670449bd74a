"""KDA (Kimi Delta Attention) chunked forward pass for GB300 -- Python binding.

Argument marshalling only: every step of the computation runs in the CUDA
library ``libkda.so`` (built from ``csrc/``) through its C ABI
(``include/kda.h``). PyTorch supplies device memory and the current stream.
There is no fallback: importing this package fails when the library is
missing, and every call raises when the library reports an error.

The call follows the tensor contract of "FlashKDA Input Tensor Shapes and
DTypes: Complete Specification for the Forward Pass": bf16 q, k, v, g
``[B, T, H, 128]``, bf16 beta logits ``[B, T, H]``, fp32 ``A_log [H]`` and
``dt_bias [H, 128]``, ``lower_bound`` in [-5, 0], optional bf16/fp32 states
``[B|N, H, 128, 128]``, optional int64 ``cu_seqlens [N+1]`` with B = 1, and
contiguous CUDA tensors.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# KDA_DEBUG_BUILD=1 loads the bounds-checked build of the same sources (libkda_debug.so), which
# reports an out-of-bounds access through check_device_status instead of faulting
DEBUG_BUILD = os.environ.get("KDA_DEBUG_BUILD", "") == "1"
LIB_PATH = os.path.join(_PKG, "libkda_debug.so" if DEBUG_BUILD else "libkda.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{os.path.basename(LIB_PATH)} is not built; run `python gated_linear_attention_kda_gb300/_build.py` "
        "(or __graft_entry__.build()) first")

_lib = ctypes.CDLL(LIB_PATH)

STATUS = {0: "KDA_OK", 1: "KDA_ERR_NULL", 2: "KDA_ERR_SHAPE", 3: "KDA_ERR_DTYPE", 4: "KDA_ERR_RANGE",
          5: "KDA_ERR_STATE_MISMATCH", 6: "KDA_ERR_ALIGN", 7: "KDA_ERR_LAUNCH", 8: "KDA_ERR_DEVICE"}
DTYPE_NONE, DTYPE_BF16, DTYPE_FP32 = 0, 1, 2
FLAG_QK_L2NORM = 1  # KDA_FLAG_QK_L2NORM: q and k L2-normalised per (token, head) inside the kernel
FLAG_CHUNK32 = 2    # KDA_FLAG_CHUNK32: 32-token chunks (the chunk-size ablation)
_P, _F, _I64, _I = ctypes.c_void_p, ctypes.c_float, ctypes.c_int64, ctypes.c_int
FWD_ARGTYPES = [_P, _P, _P, _P, _P, _F, _P, _P, _P, _F, _P, _I, _P, _I, _P, _I64, _I64, _I64, _I64, _I64, _I64, _P]
_lib.kda_fwd.argtypes = FWD_ARGTYPES
_lib.kda_fwd.restype = _I
_lib.kda_fwd_host.argtypes = FWD_ARGTYPES
_lib.kda_fwd_host.restype = _I
_lib.kda_fwd_flat.argtypes = FWD_ARGTYPES
_lib.kda_fwd_flat.restype = _I
FWD_EX_ARGTYPES = FWD_ARGTYPES[:-1] + [ctypes.c_uint32, _P]
_lib.kda_fwd_ex.argtypes = FWD_EX_ARGTYPES
_lib.kda_fwd_ex.restype = _I
_lib.kda_fwd_ws.argtypes = FWD_ARGTYPES[:-1] + [ctypes.c_uint32, _P, ctypes.c_size_t, _P]
_lib.kda_fwd_ws.restype = _I
_lib.kda_fwd_workspace_bytes.argtypes = [_I64, _I64, ctypes.c_uint32, ctypes.POINTER(ctypes.c_size_t)]
_lib.kda_fwd_workspace_bytes.restype = _I
_lib.kda_fwd_static.argtypes = FWD_EX_ARGTYPES
_lib.kda_fwd_static.restype = _I
STATIC_SCRATCH_STATES = 80  # KDA_STATIC_SCRATCH_STATES


class FwdArgs(ctypes.Structure):
    """ctypes mirror of ``kda_fwd_args`` (include/kda.h), field for field."""
    _fields_ = [("q", _P), ("k", _P), ("v", _P), ("g", _P), ("beta", _P), ("out", _P),
                ("A_log", _P), ("dt_bias", _P), ("initial_state", _P), ("final_state", _P),
                ("cu_seqlens", _P), ("initial_dtype", _I), ("final_dtype", _I),
                ("scale", _F), ("lower_bound", _F),
                ("N", _I64), ("B", _I64), ("T", _I64), ("H", _I64), ("K", _I64), ("V", _I64),
                ("flags", ctypes.c_uint32)]


_lib.kda_fwd_packed.argtypes = [ctypes.POINTER(FwdArgs), _P]
_lib.kda_fwd_packed.restype = _I
_lib.kda_decode.argtypes = [_P, _P, _P, _P, _P, _F, _P, _P, _P, _F, _P, _I, _I64, _I64, _I64, _I64, _P]
_lib.kda_decode.restype = _I
_lib.kda_decode_ex.argtypes = [_P, _P, _P, _P, _P, _F, _P, _P, _P, _F, _P, _I, _I64, _I64, _I64, _I64, ctypes.c_uint32, _P]
_lib.kda_decode_ex.restype = _I
_lib.kda_probe_chunk.argtypes = [_P, _P, _P, _P, _P, _P, _F, _I, _P, _P, _P, _P, _P, _P]
_lib.kda_probe_chunk.restype = _I
_lib.kda_probe_wait_timeout.argtypes = [_I, _P, _P]
_lib.kda_probe_wait_timeout.restype = _I
_lib.kda_probe_bounds.argtypes = [_P, _P]
_lib.kda_probe_bounds.restype = _I
_lib.kda_debug_build.argtypes = []
_lib.kda_debug_build.restype = _I
_lib.kda_probe_slots.argtypes = [_P, _P, _P, _P, _P, _F, _P, _P, _P, _F, ctypes.c_int64, _P, _I, _P]
_lib.kda_probe_slots.restype = _I
_lib.kda_probe_slot_bytes.argtypes = []
_lib.kda_probe_slot_bytes.restype = _I
_lib.kda_last_error.restype = ctypes.c_char_p
_lib.kda_check_device_status.argtypes = [_P]
_lib.kda_check_device_status.restype = _I
_lib.kda_gate_scale.argtypes = [_F]
_lib.kda_gate_scale.restype = _F
_lib.kda_plan.argtypes = [_I64, _I, ctypes.POINTER(_I), ctypes.POINTER(_I64)]
_lib.kda_plan.restype = _I
_lib.kda_version.restype = _I


class KDAError(RuntimeError):
    def __init__(self, status: int):
        self.status = status
        self.name = STATUS.get(status, str(status))
        msg = _lib.kda_last_error().decode(errors="replace")
        super().__init__(f"{self.name}: {msg}")


def _raise(status: int):
    if status != 0:
        if status in (1, 2, 3, 4, 5, 6):
            raise ValueError(str(KDAError(status)))
        raise KDAError(status)


def _state_code(t):
    if t is None:
        return DTYPE_NONE
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_FP32
    raise ValueError(f"state tensors must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(name, t, dtype, shape, cuda=True):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not cuda and t.is_cuda:
        raise ValueError(f"{name} must be a CPU tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _validate(q, k, v, g, beta, out, A_log, dt_bias, initial_state, final_state, cu_seqlens, cuda):
    if not isinstance(q, torch.Tensor) or q.dim() != 4 or not isinstance(v, torch.Tensor) or v.dim() != 4:
        raise ValueError("q, k, g must be [B, T, H, K] and v, out [B, T, H, V]")
    B, T, H, K = q.shape
    V = v.shape[-1]
    for name, t, shp in (("q", q, (B, T, H, K)), ("k", k, (B, T, H, K)), ("g", g, (B, T, H, K)),
                         ("v", v, (B, T, H, V)), ("out", out, (B, T, H, V)), ("beta", beta, (B, T, H))):
        if t is None:
            raise ValueError(f"{name} is required")
        _check(name, t, torch.bfloat16, shp, cuda)
    _check("A_log", A_log, torch.float32, (H,), cuda)
    _check("dt_bias", dt_bias, torch.float32, (H, K), cuda)
    N = 0
    if cu_seqlens is not None:
        _check("cu_seqlens", cu_seqlens, torch.int64, None, cuda)
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
            raise ValueError("cu_seqlens must be [N+1] with N >= 1")
        N = cu_seqlens.numel() - 1
    S = N if cu_seqlens is not None else B
    for name, t in (("initial_state", initial_state), ("final_state", final_state)):
        _check(name, t, None, (S, H, V, K), cuda)
    _same_device(q.device, (("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out), ("A_log", A_log),
                            ("dt_bias", dt_bias), ("initial_state", initial_state), ("final_state", final_state),
                            ("cu_seqlens", cu_seqlens)))
    return B, T, H, K, V, N


def _flags(qk_l2norm, chunk):
    if chunk not in (16, 32):
        raise ValueError(f"chunk must be 16 or 32, got {chunk}")
    return (FLAG_QK_L2NORM if qk_l2norm else 0) | (FLAG_CHUNK32 if chunk == 32 else 0)


def _same_device(dev, named):
    """Every given tensor must live on ``dev`` (q's device): the library launches on that device
    and dereferences every pointer there, so a tensor on another GPU is rejected here."""
    for name, t in named:
        if t is not None and t.device != dev:
            raise ValueError(f"{name} is on {t.device}, but q is on {dev}: all tensors must share one device")


def fwd(q, k, v, g, beta, scale, out, A_log=None, dt_bias=None, lower_bound=-5.0,
        initial_state=None, final_state=None, cu_seqlens=None, qk_l2norm=False, chunk=16):
    """Chunked KDA forward on the current CUDA stream. Writes ``out`` (and
    ``final_state`` if given) in place and returns ``(out, final_state)``.
    ``qk_l2norm=True`` L2-normalises q and k per (token, head) inside the
    kernel (``KDA_FLAG_QK_L2NORM``); ``chunk=32`` runs 32-token chunks
    (``KDA_FLAG_CHUNK32``). Either goes through ``kda_fwd_ex``, the plain
    call through ``kda_fwd``."""
    flags = _flags(qk_l2norm, chunk)
    B, T, H, K, V, N = _validate(q, k, v, g, beta, out, A_log, dt_bias, initial_state, final_state,
                                 cu_seqlens, cuda=True)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out),
            _ptr(A_log), _ptr(dt_bias), float(lower_bound),
            _ptr(initial_state), _state_code(initial_state),
            _ptr(final_state), _state_code(final_state),
            _ptr(cu_seqlens), N, B, T, H, K, V)
    with torch.cuda.device(q.device):
        stream = ctypes.c_void_p(torch.cuda.current_stream(q.device).cuda_stream)
        if flags:
            st = _lib.kda_fwd_ex(*args, flags, stream)
        else:
            st = _lib.kda_fwd(*args, stream)
    _raise(st)
    return out, final_state


def workspace_bytes(states, H, qk_l2norm=False, chunk=16) -> int:
    """Bytes of workspace ``fwd_ws`` uses for ``states`` sequences x ``H`` heads on the current
    device (0 when the call's plan does not split the state)."""
    n = ctypes.c_size_t(0)
    _raise(_lib.kda_fwd_workspace_bytes(int(states), int(H), _flags(qk_l2norm, chunk), ctypes.byref(n)))
    return int(n.value)


def fwd_ws(q, k, v, g, beta, scale, out, A_log=None, dt_bias=None, lower_bound=-5.0,
           initial_state=None, final_state=None, cu_seqlens=None, qk_l2norm=False, chunk=16, workspace=None):
    """``fwd`` through ``kda_fwd_ws``: with a workspace of ``workspace_bytes`` bytes (a CUDA uint8
    tensor), a split state's chunk preparation is shared by the CTAs of the state. Results equal
    ``fwd``'s bit for bit."""
    flags = _flags(qk_l2norm, chunk)
    B, T, H, K, V, N = _validate(q, k, v, g, beta, out, A_log, dt_bias, initial_state, final_state,
                                 cu_seqlens, cuda=True)
    nbytes = 0
    if workspace is not None:
        if workspace.dtype != torch.uint8 or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous uint8 tensor")
        _same_device(q.device, [("workspace", workspace)])
        nbytes = workspace.numel()
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out),
            _ptr(A_log), _ptr(dt_bias), float(lower_bound),
            _ptr(initial_state), _state_code(initial_state),
            _ptr(final_state), _state_code(final_state),
            _ptr(cu_seqlens), N, B, T, H, K, V)
    with torch.cuda.device(q.device):
        stream = ctypes.c_void_p(torch.cuda.current_stream(q.device).cuda_stream)
        st = _lib.kda_fwd_ws(*args, flags, _ptr(workspace), ctypes.c_size_t(nbytes), stream)
    _raise(st)
    return out, final_state


def fwd_static(q, k, v, g, beta, scale, out, A_log=None, dt_bias=None, lower_bound=-5.0,
               initial_state=None, final_state=None, cu_seqlens=None, qk_l2norm=False, chunk=16):
    """``fwd`` through ``kda_fwd_static``: the shared chunk preparation of ``fwd_ws`` with the
    library's own scratch (room for ``STATIC_SCRATCH_STATES`` states, no allocation). Calls that
    overlap in time on one device share that scratch: issue them on one stream."""
    flags = _flags(qk_l2norm, chunk)
    B, T, H, K, V, N = _validate(q, k, v, g, beta, out, A_log, dt_bias, initial_state, final_state,
                                 cu_seqlens, cuda=True)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out),
            _ptr(A_log), _ptr(dt_bias), float(lower_bound),
            _ptr(initial_state), _state_code(initial_state),
            _ptr(final_state), _state_code(final_state),
            _ptr(cu_seqlens), N, B, T, H, K, V)
    with torch.cuda.device(q.device):
        stream = ctypes.c_void_p(torch.cuda.current_stream(q.device).cuda_stream)
        st = _lib.kda_fwd_static(*args, flags, stream)
    _raise(st)
    return out, final_state


def fwd_flat(q, k, v, g, beta, scale, out, A_log=None, dt_bias=None, lower_bound=-5.0,
             initial_state=None, final_state=None, cu_seqlens=None):
    """``fwd`` through the ``kda_fwd_flat`` entry point (the same C call under its second name)."""
    B, T, H, K, V, N = _validate(q, k, v, g, beta, out, A_log, dt_bias, initial_state, final_state,
                                 cu_seqlens, cuda=True)
    with torch.cuda.device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        st = _lib.kda_fwd_flat(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out),
                               _ptr(A_log), _ptr(dt_bias), float(lower_bound),
                               _ptr(initial_state), _state_code(initial_state),
                               _ptr(final_state), _state_code(final_state),
                               _ptr(cu_seqlens), N, B, T, H, K, V, ctypes.c_void_p(stream))
    _raise(st)
    return out, final_state


def fwd_packed(q, k, v, g, beta, scale, out, A_log=None, dt_bias=None, lower_bound=-5.0,
               initial_state=None, final_state=None, cu_seqlens=None, qk_l2norm=False, chunk=16):
    """``fwd`` through the argument-struct entry point ``kda_fwd_packed``."""
    flags = _flags(qk_l2norm, chunk)
    B, T, H, K, V, N = _validate(q, k, v, g, beta, out, A_log, dt_bias, initial_state, final_state,
                                 cu_seqlens, cuda=True)
    a = FwdArgs()
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out), ("A_log", A_log),
                    ("dt_bias", dt_bias), ("initial_state", initial_state), ("final_state", final_state),
                    ("cu_seqlens", cu_seqlens)):
        setattr(a, name, None if t is None else t.data_ptr())
    a.initial_dtype, a.final_dtype = _state_code(initial_state), _state_code(final_state)
    a.scale, a.lower_bound = float(scale), float(lower_bound)
    a.N, a.B, a.T, a.H, a.K, a.V = N, B, T, H, K, V
    a.flags = flags
    with torch.cuda.device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        st = _lib.kda_fwd_packed(ctypes.byref(a), ctypes.c_void_p(stream))
    _raise(st)
    return out, final_state




def decode(q, k, v, g, beta, scale, out, state, A_log=None, dt_bias=None, lower_bound=-5.0, qk_l2norm=False):
    """One token per (sequence, head) on the current CUDA stream, ``state`` updated in place:
    ``q, k, v, g, out`` bf16 ``[S, H, 128]`` (or ``[S, 1, H, 128]``), ``beta`` bf16 ``[S, H]``
    (or ``[S, 1, H]``), ``state`` bf16/fp32 ``[S, H, 128, 128]`` (kda_fwd's final_state).
    ``qk_l2norm=True`` L2-normalises q and k inside the kernel (``kda_decode_ex``).
    Returns ``(out, state)``."""
    if not isinstance(q, torch.Tensor) or q.dim() not in (3, 4):
        raise ValueError("q must be [S, H, 128] or [S, 1, H, 128]")
    if q.dim() == 4 and q.shape[1] != 1:
        raise ValueError("decode takes one token per sequence (T = 1)")
    S, H, K = q.shape[0], q.shape[-2], q.shape[-1]
    V = v.shape[-1]
    for name, t, shp in (("q", q, q.shape), ("k", k, q.shape), ("g", g, q.shape), ("v", v, q.shape[:-1] + (V,)),
                         ("out", out, q.shape[:-1] + (V,)), ("beta", beta, q.shape[:-1])):
        _check(name, t, torch.bfloat16, shp, True)
    _check("A_log", A_log, torch.float32, (H,), True)
    _check("dt_bias", dt_bias, torch.float32, (H, K), True)
    _check("state", state, None, (S, H, V, K), True)
    _same_device(q.device, (("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out), ("A_log", A_log),
                            ("dt_bias", dt_bias), ("state", state)))
    with torch.cuda.device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        st = _lib.kda_decode_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out),
                                _ptr(A_log), _ptr(dt_bias), float(lower_bound), _ptr(state), _state_code(state),
                                S, H, K, V, FLAG_QK_L2NORM if qk_l2norm else 0, ctypes.c_void_p(stream))
    _raise(st)
    return out, state

def probe_chunk(q, k, g, beta, A_log=None, dt_bias=None, lower_bound=-5.0, rows=16):
    """Test hook: one chunk of one head (``q, k, g`` bf16 [16, 128], ``beta`` bf16 [16] logits,
    ``A_log`` fp32 [1] or None, ``dt_bias`` fp32 [128] or None, all on the GPU) through the
    per-chunk steps. Returns fp32 ``G2`` [16, 128] (log2 units, cumsum), ``beta`` [16] and
    ``A``, ``P``, ``T`` [16, 16]."""
    for name, t, dt, shp in (("q", q, torch.bfloat16, (16, 128)), ("k", k, torch.bfloat16, (16, 128)),
                             ("g", g, torch.bfloat16, (16, 128)), ("beta", beta, torch.bfloat16, (16,))):
        _check(name, t, dt, shp, True)
    _check("A_log", A_log, torch.float32, (1,), True)
    _check("dt_bias", dt_bias, torch.float32, (128,), True)
    o = {n: torch.empty(shp, dtype=torch.float32, device=q.device)
         for n, shp in (("G2", (16, 128)), ("beta", (16,)), ("A", (16, 16)), ("P", (16, 16)), ("T", (16, 16)))}
    with torch.cuda.device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        st = _lib.kda_probe_chunk(_ptr(q), _ptr(k), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(dt_bias),
                                  float(lower_bound), int(rows), _ptr(o["G2"]), _ptr(o["beta"]), _ptr(o["A"]),
                                  _ptr(o["P"]), _ptr(o["T"]), ctypes.c_void_p(stream))
    _raise(st)
    return o

def probe_wait_timeout(polls, device=None):
    """Test hook: run the kernels' bounded pipeline wait out on purpose (``kda_probe_wait_timeout``)
    with ``polls`` polls. Returns the three result words: (wait 0 succeeded, wait 1 succeeded,
    abort flag). The device error word then carries the timeout bit for ``check_device_status``."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    res = torch.full((3,), -1, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        st = _lib.kda_probe_wait_timeout(int(polls), _ptr(res), ctypes.c_void_p(stream))
    _raise(st)
    return [int(x) for x in res.cpu()]


def probe_bounds(device=None):
    """Test hook: run the bounds checks on a shared address and a global index that are out of
    range, without accessing them (``kda_probe_bounds``). Returns [shared check passed, global
    check passed]: [0, 0] in the bounds-checked build (which also flags the device error word),
    [1, 1] in the product build."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    res = torch.full((2,), -1, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        st = _lib.kda_probe_bounds(_ptr(res), ctypes.c_void_p(stream))
    _raise(st)
    return [int(x) for x in res.cpu()]


def probe_slots(q, k, v, g, beta, scale, A_log=None, dt_bias=None, lower_bound=-5.0, nchunks=None):
    """Test hook: one head of T tokens (``q, k, v, g`` bf16 [T, 128], ``beta`` bf16 [T], ``A_log``
    fp32 [1] or None, ``dt_bias`` fp32 [128] or None; CUDA) through the tcgen05 kernel, returning
    the prep slot of each of the first ``nchunks`` chunks as the tensor core reads it: uint8
    [nchunks, kda_probe_slot_bytes()] (layout in include/kda.h), and the outputs [T, 128]."""
    T = q.shape[0]
    for name, t, shp in (("q", q, (T, 128)), ("k", k, (T, 128)), ("v", v, (T, 128)), ("g", g, (T, 128)),
                         ("beta", beta, (T,))):
        _check(name, t, torch.bfloat16, shp, True)
    _check("A_log", A_log, torch.float32, (1,), True)
    _check("dt_bias", dt_bias, torch.float32, (128,), True)
    n = (T + 15) // 16 if nchunks is None else int(nchunks)
    dump = torch.zeros((n, _lib.kda_probe_slot_bytes()), dtype=torch.uint8, device=q.device)
    out = torch.empty_like(v)
    with torch.cuda.device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        st = _lib.kda_probe_slots(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out),
                                  _ptr(A_log), _ptr(dt_bias), float(lower_bound), T, _ptr(dump), n,
                                  ctypes.c_void_p(stream))
    _raise(st)
    return dump, out


def debug_build() -> bool:
    """True when the loaded library is the bounds-checked build (``KDA_DEBUG_BUILD=1``)."""
    return bool(_lib.kda_debug_build())


def fwd_host(q, k, v, g, beta, scale, out, A_log=None, dt_bias=None, lower_bound=-5.0,
             initial_state=None, final_state=None, cu_seqlens=None, device=None):
    """Same operation on CPU tensors (pin them for fast copies): the library
    copies inputs to the GPU, runs, copies ``out``/``final_state`` back and
    synchronises before returning."""
    B, T, H, K, V, N = _validate(q, k, v, g, beta, out, A_log, dt_bias, initial_state, final_state,
                                 cu_seqlens, cuda=False)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        st = _lib.kda_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out),
                               _ptr(A_log), _ptr(dt_bias), float(lower_bound),
                               _ptr(initial_state), _state_code(initial_state),
                               _ptr(final_state), _state_code(final_state),
                               _ptr(cu_seqlens), N, B, T, H, K, V, ctypes.c_void_p(stream))
    _raise(st)
    return out, final_state


def check_device_status(device=None, stream=None):
    """Synchronise ``stream`` (default: the current stream of ``device``) and raise if a kernel on
    that device flagged an error. ``device`` is a ``torch.device``, an index or a tensor (its
    device); by default the current device. The error word is shared by every call on the device
    and is read and cleared in one step, so a flag is reported once, by the first check after it."""
    if isinstance(device, torch.Tensor):
        device = device.device
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if dev.type == "cuda" and dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        s = torch.cuda.current_stream(dev).cuda_stream if stream is None else stream
        _raise(_lib.kda_check_device_status(ctypes.c_void_p(s)))


def gate_scale(lower_bound: float) -> float:
    return _lib.kda_gate_scale(float(lower_bound))


def plan(units: int, num_sms: int):
    vs, grid = _I(), _I64()
    _raise(_lib.kda_plan(int(units), int(num_sms), ctypes.byref(vs), ctypes.byref(grid)))
    return vs.value, grid.value


def version() -> int:
    return _lib.kda_version()


def library():
    """The loaded ctypes handle of libkda.so (for direct C-ABI calls)."""
    return _lib
