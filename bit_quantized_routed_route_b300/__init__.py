"""Python binding of libds4g, the B300 (sm_103a) routed-MoE expert layer over
low-bit quantized experts.

Argument marshalling only: every step of the layer runs in the CUDA kernels of
``libds4g.so`` behind the C ABI declared in ``include/ds4g.h``.  PyTorch is
used for device memory and streams.  Importing this package on a machine
where the library is missing raises immediately; there is no fallback.

Entry points (same names as the C ABI, without the ``ds4g_`` prefix):
  route_topk, q2k_dequant, cb2_dequant, q4k_dequant, q5k_dequant, q6k_dequant, mxfp4_dequant,
  moe_workspace_bytes, moe_forward,
  moe_forward_host, moe_routing_view, status_string, abi_version.
Each returns the raw status code; ``check(status)`` turns a non-zero status
into ``DS4GError``.  ``Layer`` is a convenience holder for device-resident
expert weights and their descriptor.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(HERE, "libds4g.so")

(OK, ERR_INVALID, ERR_SHAPE, ERR_LAYOUT, ERR_WORKSPACE, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT,
 ERR_RANGE) = range(9)
SCORE_SOFTMAX, SCORE_SIGMOID = 0, 1
FMT_Q2K, FMT_CB2, FMT_Q4K, FMT_Q5K, FMT_Q6K, FMT_MXFP4 = 0, 1, 2, 3, 4, 5
F32, F16, BF16 = 0, 1, 2
FORCE_GEMV, FORCE_TC, DEBUG_STALL = 1, 2, 256

EXPORTED = (
    "ds4g_route_topk", "ds4g_q2k_dequant", "ds4g_cb2_dequant", "ds4g_q4k_dequant",
    "ds4g_q5k_dequant", "ds4g_q6k_dequant", "ds4g_mxfp4_dequant", "ds4g_moe_workspace_bytes",
    "ds4g_moe_forward", "ds4g_moe_forward_host", "ds4g_moe_routing_view",
    "ds4g_moe_forward_phased", "ds4g_moe_forward_launches", "ds4g_moe_device_status",
    "ds4g_status_string", "ds4g_abi_version", "ds4g_last_cuda_error",
    "ds4g_moe_forward_noalloc", "ds4g_moe_noalloc_status", "ds4g_expert_cache_create", "ds4g_expert_cache_workspace_bytes",
    "ds4g_expert_cache_forward", "ds4g_expert_cache_stats", "ds4g_expert_cache_destroy",
)


class DS4GError(RuntimeError):
    def __init__(self, status: int):
        msg = f"ds4g status {status}: {status_string(status)}"
        if status == ERR_CUDA:
            msg += f" (cudaError {_lib.ds4g_last_cuda_error()})"
        super().__init__(msg)
        self.status = status


class MoeDesc(ctypes.Structure):
    """Mirror of ``ds4g_moe_desc``."""
    _fields_ = [
        ("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
        ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
        ("score", ctypes.c_int32), ("format", ctypes.c_int32),
        ("flags", ctypes.c_int32), ("tc_min_tokens", ctypes.c_int32),
        ("down_format", ctypes.c_int32), ("n_slots", ctypes.c_int32),
        ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
        ("gate_up_row_bytes", ctypes.c_int64), ("down_row_bytes", ctypes.c_int64),
        ("gate_up_expert_stride", ctypes.c_int64), ("down_expert_stride", ctypes.c_int64),
        ("codebook", ctypes.c_void_p), ("expert_slot", ctypes.c_void_p),
    ]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIBRARY):
        raise ImportError(
            f"libds4g.so is not built ({LIBRARY}); run `python -m "
            "bit_quantized_routed_route_b300.build` (needs nvcc for sm_103a)")
    lib = ctypes.CDLL(LIBRARY)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    pdesc = ctypes.POINTER(MoeDesc)
    sig = {
        "ds4g_route_topk": (i32, [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]),
        "ds4g_q2k_dequant": (i32, [vp, i64, vp, i32, vp]),
        "ds4g_cb2_dequant": (i32, [vp, i64, vp, vp, i32, vp]),
        "ds4g_q4k_dequant": (i32, [vp, i64, vp, i32, vp]),
        "ds4g_q5k_dequant": (i32, [vp, i64, vp, i32, vp]),
        "ds4g_q6k_dequant": (i32, [vp, i64, vp, i32, vp]),
        "ds4g_mxfp4_dequant": (i32, [vp, i64, vp, i32, vp]),
        "ds4g_moe_noalloc_status": (i32, [ctypes.POINTER(MoeDesc), i32, ctypes.POINTER(i32), vp]),
        "ds4g_expert_cache_create": (i32, [ctypes.POINTER(MoeDesc), i32, ctypes.POINTER(vp)]),
        "ds4g_expert_cache_workspace_bytes": (ctypes.c_size_t, [vp, i32]),
        "ds4g_expert_cache_forward": (i32, [vp, vp, vp, i32, vp, vp, ctypes.c_size_t, vp]),
        "ds4g_expert_cache_stats": (i32, [vp, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                          ctypes.POINTER(i64)]),
        "ds4g_expert_cache_destroy": (None, [vp]),
        "ds4g_moe_workspace_bytes": (sz, [pdesc, i32]),
        "ds4g_moe_forward": (i32, [pdesc, vp, vp, i32, vp, vp, sz, vp]),
        "ds4g_moe_forward_host": (i32, [pdesc, vp, vp, i32, vp, vp, sz, vp]),
        "ds4g_moe_routing_view": (i32, [pdesc, i32, vp, sz, vp, vp, vp, vp, vp]),
        "ds4g_moe_forward_phased": (i32, [pdesc, vp, vp, i32, vp, vp, sz, vp,
                                          ctypes.POINTER(ctypes.c_void_p), i32]),
        "ds4g_moe_forward_launches": (i32, [pdesc, i32]),
        "ds4g_moe_device_status": (i32, [pdesc, i32, vp, sz, ctypes.POINTER(i32), vp]),
        "ds4g_status_string": (ctypes.c_char_p, [i32]),
        "ds4g_abi_version": (i32, []),
        "ds4g_last_cuda_error": (i32, []),
        "ds4g_moe_forward_noalloc": (i32, [pdesc, vp, vp, i32, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def lib() -> ctypes.CDLL:
    return _lib


def _ptr(t) -> Optional[int]:
    """Raw address of a torch tensor, a numpy array, an int, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        return t.ctypes.data
    raise TypeError(f"cannot pass {type(t)} as a pointer")


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def check(status: int) -> None:
    if status != OK:
        raise DS4GError(status)


def status_string(status: int) -> str:
    return _lib.ds4g_status_string(status).decode()


def abi_version() -> int:
    return _lib.ds4g_abi_version()


def route_topk(logits, T, E, k, score, ids, weights, counts=None, offsets=None, perm=None,
               stream=None) -> int:
    return _lib.ds4g_route_topk(_ptr(logits), T, E, k, score, _ptr(ids), _ptr(weights),
                                _ptr(counts), _ptr(offsets), _ptr(perm), _stream(stream))


def q2k_dequant(blocks, n_blocks, out, out_dtype, stream=None) -> int:
    return _lib.ds4g_q2k_dequant(_ptr(blocks), n_blocks, _ptr(out), out_dtype, _stream(stream))


def q4k_dequant(blocks, n_blocks, out, out_dtype, stream=None) -> int:
    return _lib.ds4g_q4k_dequant(_ptr(blocks), n_blocks, _ptr(out), out_dtype, _stream(stream))


def q5k_dequant(blocks, n_blocks, out, out_dtype, stream=None) -> int:
    return _lib.ds4g_q5k_dequant(_ptr(blocks), n_blocks, _ptr(out), out_dtype, _stream(stream))


def q6k_dequant(blocks, n_blocks, out, out_dtype, stream=None) -> int:
    return _lib.ds4g_q6k_dequant(_ptr(blocks), n_blocks, _ptr(out), out_dtype, _stream(stream))


def mxfp4_dequant(blocks, n_blocks, out, out_dtype, stream=None) -> int:
    return _lib.ds4g_mxfp4_dequant(_ptr(blocks), n_blocks, _ptr(out), out_dtype, _stream(stream))


def cb2_dequant(blocks, n_blocks, codebook, out, out_dtype, stream=None) -> int:
    return _lib.ds4g_cb2_dequant(_ptr(blocks), n_blocks, _ptr(codebook), _ptr(out), out_dtype,
                                 _stream(stream))


def moe_workspace_bytes(desc: MoeDesc, T: int) -> int:
    return _lib.ds4g_moe_workspace_bytes(ctypes.byref(desc), T)


def moe_forward(desc: MoeDesc, x, logits, T, y, workspace, ws_bytes=None, stream=None) -> int:
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    return _lib.ds4g_moe_forward(ctypes.byref(desc), _ptr(x), _ptr(logits), T, _ptr(y),
                                 _ptr(workspace), ws_bytes, _stream(stream))


def moe_forward_host(desc: MoeDesc, x_host, logits_host, T, y_host, workspace, ws_bytes=None,
                     stream=None) -> int:
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    return _lib.ds4g_moe_forward_host(ctypes.byref(desc), _ptr(x_host), _ptr(logits_host), T,
                                      _ptr(y_host), _ptr(workspace), ws_bytes, _stream(stream))


def moe_forward_phased(desc: MoeDesc, x, logits, T, y, workspace, events, ws_bytes=None,
                       stream=None) -> int:
    """``events``: five cudaEvent_t handles (ints) recorded at the phase
    boundaries (before routing, after routing, after gate/up, after down,
    after combine)."""
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    arr = (ctypes.c_void_p * len(events))(*events)
    return _lib.ds4g_moe_forward_phased(ctypes.byref(desc), _ptr(x), _ptr(logits), T, _ptr(y),
                                        _ptr(workspace), ws_bytes, _stream(stream), arr,
                                        len(events))


def moe_forward_launches(desc: MoeDesc, T: int) -> int:
    return _lib.ds4g_moe_forward_launches(ctypes.byref(desc), T)


def moe_forward_noalloc(desc: MoeDesc, x, logits, T, y, stream=None) -> int:
    """The layer without a caller workspace (a static device array of
    NOALLOC_SCRATCH_BYTES per GPU); for callers that cannot allocate."""
    return _lib.ds4g_moe_forward_noalloc(ctypes.byref(desc), _ptr(x), _ptr(logits), T, _ptr(y),
                                         _stream(stream))


NOALLOC_SCRATCH_BYTES = 32 << 20


def moe_device_status(desc: MoeDesc, T: int, workspace, ws_bytes=None, stream=None):
    """(status of the call, device status word of the last forward)."""
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    v = ctypes.c_int32(-1)
    st = _lib.ds4g_moe_device_status(ctypes.byref(desc), T, _ptr(workspace), ws_bytes,
                                     ctypes.byref(v), _stream(stream))
    return st, v.value


def moe_routing_view(desc: MoeDesc, T: int, workspace, ws_bytes=None):
    """(status, dict of device addresses: ids, weights, counts, offsets, perm)."""
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    out = [ctypes.c_void_p() for _ in range(5)]
    st = _lib.ds4g_moe_routing_view(ctypes.byref(desc), T, _ptr(workspace), ws_bytes,
                                    *[ctypes.byref(o) for o in out])
    names = ("ids", "weights", "counts", "offsets", "perm")
    return st, {n: (o.value or 0) for n, o in zip(names, out)}


def moe_noalloc_status(desc: MoeDesc, T: int, stream=None):
    """(status, device status word of the last ds4g_moe_forward_noalloc)."""
    v = ctypes.c_int32(-1)
    st = _lib.ds4g_moe_noalloc_status(ctypes.byref(desc), T, ctypes.byref(v), _stream(stream))
    return st, v.value


class Layer:
    """Device-resident expert weights of one layer plus their descriptor.

    ``weights`` holds uint8 tensors [E x N x row_bytes] (any device tensors
    the caller keeps alive); the descriptor points at them.  ``fmt`` is the
    format of W_gate and W_up, ``down_fmt`` that of W_down (default: fmt)."""

    def __init__(self, hidden, inter, n_experts, top_k, score, fmt, w_gate, w_up, w_down,
                 codebook=None, flags=0, tc_min_tokens=0, down_fmt=None):
        self.tensors = (w_gate, w_up, w_down, codebook)
        d = MoeDesc()
        d.hidden, d.inter, d.n_experts, d.top_k = hidden, inter, n_experts, top_k
        d.score, d.format, d.flags, d.tc_min_tokens = score, fmt, flags, tc_min_tokens
        d.down_format = fmt if down_fmt is None else down_fmt
        d.n_slots = 0
        d.w_gate, d.w_up, d.w_down = _ptr(w_gate), _ptr(w_up), _ptr(w_down)
        d.gate_up_row_bytes = w_gate.shape[-1]
        d.down_row_bytes = w_down.shape[-1]
        d.gate_up_expert_stride = w_gate.shape[-2] * w_gate.shape[-1]
        d.down_expert_stride = w_down.shape[-2] * w_down.shape[-1]
        d.codebook = _ptr(codebook)
        self.desc = d

    def with_flags(self, flags: int, tc_min_tokens: Optional[int] = None) -> "Layer":
        other = object.__new__(Layer)
        other.tensors = self.tensors
        d = MoeDesc.from_buffer_copy(self.desc)
        d.flags = flags
        if tc_min_tokens is not None:
            d.tc_min_tokens = tc_min_tokens
        other.desc = d
        return other

    def workspace_bytes(self, T: int) -> int:
        return moe_workspace_bytes(self.desc, T)

    def forward(self, x, logits, y, workspace, stream=None) -> None:
        check(moe_forward(self.desc, x, logits, x.shape[0], y, workspace, stream=stream))


class ExpertCache:
    """ds4g_expert_cache: a layer whose expert weights live in host memory
    (page-locked uint8 tensors [E x N x row_bytes]), ``n_slots`` experts of
    it resident on the current device and uploaded on misses.  ``forward``
    returns the raw status (DS4G_ERR_UNSUPPORTED when a call routes to more
    experts than there are slots)."""

    def __init__(self, hidden, inter, n_experts, top_k, score, fmt, w_gate, w_up, w_down,
                 n_slots, codebook=None, flags=0, down_fmt=None):
        self.host = Layer(hidden, inter, n_experts, top_k, score, fmt, w_gate, w_up, w_down,
                          codebook, flags=flags, down_fmt=down_fmt)
        h = ctypes.c_void_p()
        check(_lib.ds4g_expert_cache_create(ctypes.byref(self.host.desc), n_slots, ctypes.byref(h)))
        self.handle = h

    def workspace_bytes(self, T: int) -> int:
        return _lib.ds4g_expert_cache_workspace_bytes(self.handle, T)

    def forward(self, x, logits, y, workspace, ws_bytes=None, stream=None) -> int:
        if ws_bytes is None:
            ws_bytes = workspace.numel() * workspace.element_size()
        return _lib.ds4g_expert_cache_forward(self.handle, _ptr(x), _ptr(logits), x.shape[0],
                                              _ptr(y), _ptr(workspace), ws_bytes, _stream(stream))

    def stats(self):
        """(hits, misses, bytes uploaded) since creation."""
        v = [ctypes.c_int64() for _ in range(3)]
        check(_lib.ds4g_expert_cache_stats(self.handle, *[ctypes.byref(o) for o in v]))
        return tuple(o.value for o in v)

    def close(self) -> None:
        if getattr(self, "handle", None) is not None and self.handle.value:
            _lib.ds4g_expert_cache_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # pragma: no cover - interpreter shutdown
            pass
