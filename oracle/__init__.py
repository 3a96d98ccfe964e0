"""ds4g reference oracle -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.

A thin ctypes wrapper over ``ds4g_oracle.c``: a plain single-threaded C
restatement of the routed-MoE expert layer over 2-bit quantized experts
(fp32 dequantization from the block definitions, fp64 accumulation, top-k
with ties broken by the lower expert id).  The CUDA library shares no code
with it.  Only the tests, the package smoke check and the benchmark's CPU
baseline leg may import this module.

What each function restates, and which passage of the pages it follows, is
written beside the C functions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "ds4g_oracle.c")
LIBRARY = os.path.join(HERE, "libds4g_oracle.so")

SCORE_SOFTMAX = 0
SCORE_SIGMOID = 1
FMT_Q2K = 0
FMT_CB2 = 1
QK = 256
Q2K_BYTES = 84
CB2_BYTES = 70
Q4K_BYTES, Q5K_BYTES, Q6K_BYTES, MXFP4_BYTES = 144, 176, 210, 136

CFLAGS = ["-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared"]


def build(source: str = SOURCE, out: str = LIBRARY) -> str:
    """Compiles the oracle with gcc (plain C99, no FMA contraction)."""
    cmd = ["gcc", *CFLAGS, "-o", out, source, "-lm"]
    subprocess.run(cmd, check=True)
    return out


class _Layer(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
        ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
        ("score", ctypes.c_int32), ("format", ctypes.c_int32),
        ("down_format", ctypes.c_int32),
        ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p),
        ("w_down", ctypes.c_void_p),
        ("gate_up_row_bytes", ctypes.c_int64), ("down_row_bytes", ctypes.c_int64),
        ("gate_up_expert_stride", ctypes.c_int64), ("down_expert_stride", ctypes.c_int64),
        ("codebook", ctypes.c_void_p),
    ]


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


class Oracle:
    """Handle on one compiled oracle library (the committed one, or a test
    copy with a planted mistake)."""

    def __init__(self, path: str = LIBRARY):
        if path == LIBRARY and not os.path.exists(path):
            build()
        self.path = path
        lib = ctypes.CDLL(path)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_half_to_double.restype = ctypes.c_double
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_double.restype = ctypes.c_double
        lib.orc_q2k_dequant.argtypes = [vp, i64, vp]
        lib.orc_q2k_dequant.restype = None
        lib.orc_cb2_dequant.argtypes = [vp, i64, vp, vp]
        lib.orc_cb2_dequant.restype = None
        for name in ("orc_q4k_dequant", "orc_q5k_dequant", "orc_q6k_dequant", "orc_mxfp4_dequant"):
            getattr(lib, name).argtypes = [vp, i64, vp]
            getattr(lib, name).restype = None
        lib.orc_route.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp]
        lib.orc_route.restype = ctypes.c_int
        lib.orc_moe_forward.argtypes = [ctypes.POINTER(_Layer), vp, vp, i32, vp, i32,
                                        vp, vp, vp]
        lib.orc_moe_forward.restype = ctypes.c_int
        lib.orc_expert_ffn.argtypes = [ctypes.POINTER(_Layer), i32, vp, vp]
        lib.orc_expert_ffn.restype = ctypes.c_int
        self.lib = lib

    # -- scalar formats ---------------------------------------------------
    def half_to_double(self, bits: int) -> float:
        return self.lib.orc_half_to_double(bits)

    def bf16_to_double(self, bits: int) -> float:
        return self.lib.orc_bf16_to_double(bits)

    # -- dequantization ---------------------------------------------------
    def q2k_dequant(self, blocks: np.ndarray) -> np.ndarray:
        """blocks: uint8 [..., 84*n] -> float32 [n*256]."""
        b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
        assert b.size % Q2K_BYTES == 0
        n = b.size // Q2K_BYTES
        out = np.empty(n * QK, dtype=np.float32)
        self.lib.orc_q2k_dequant(_ptr(b), n, _ptr(out))
        return out

    def _kquant(self, fn, bb: int, blocks: np.ndarray) -> np.ndarray:
        b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
        assert b.size % bb == 0
        n = b.size // bb
        out = np.empty(n * QK, dtype=np.float32)
        fn(_ptr(b), n, _ptr(out))
        return out

    def q4k_dequant(self, blocks: np.ndarray) -> np.ndarray:
        """blocks: uint8 [..., 144*n] -> float32 [n*256]."""
        return self._kquant(self.lib.orc_q4k_dequant, Q4K_BYTES, blocks)

    def q5k_dequant(self, blocks: np.ndarray) -> np.ndarray:
        """blocks: uint8 [..., 176*n] -> float32 [n*256]."""
        return self._kquant(self.lib.orc_q5k_dequant, Q5K_BYTES, blocks)

    def q6k_dequant(self, blocks: np.ndarray) -> np.ndarray:
        """blocks: uint8 [..., 210*n] -> float32 [n*256]."""
        return self._kquant(self.lib.orc_q6k_dequant, Q6K_BYTES, blocks)

    def mxfp4_dequant(self, blocks: np.ndarray) -> np.ndarray:
        """blocks: uint8 [..., 136*n] (eight 17-byte MXFP4 blocks per 256 weights)."""
        return self._kquant(self.lib.orc_mxfp4_dequant, MXFP4_BYTES, blocks)

    def cb2_dequant(self, blocks: np.ndarray, codebook: np.ndarray) -> np.ndarray:
        b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
        cb = np.ascontiguousarray(codebook, dtype=np.int8).reshape(-1)
        assert b.size % CB2_BYTES == 0 and cb.size == 256 * 8
        n = b.size // CB2_BYTES
        out = np.empty(n * QK, dtype=np.float32)
        self.lib.orc_cb2_dequant(_ptr(b), n, _ptr(cb), _ptr(out))
        return out

    # -- routing ----------------------------------------------------------
    def route(self, logits: np.ndarray, k: int, score: int):
        lg = np.ascontiguousarray(logits, dtype=np.float32)
        T, E = lg.shape
        ids = np.empty((T, k), dtype=np.int32)
        w = np.empty((T, k), dtype=np.float64)
        counts = np.empty(E, dtype=np.int32)
        offsets = np.empty(E + 1, dtype=np.int32)
        perm = np.empty(T * k, dtype=np.int32)
        rc = self.lib.orc_route(_ptr(lg), T, E, k, score, _ptr(ids), _ptr(w),
                                _ptr(counts), _ptr(offsets), _ptr(perm))
        if rc != 0:
            raise ValueError(f"orc_route rejected its arguments (code {rc})")
        return dict(ids=ids, weights=w, counts=counts, offsets=offsets, perm=perm)

    # -- the layer --------------------------------------------------------
    @staticmethod
    def _layer(layer) -> _Layer:
        L = _Layer()
        L.hidden, L.inter = layer["hidden"], layer["inter"]
        L.n_experts, L.top_k = layer["n_experts"], layer["top_k"]
        L.score, L.format = layer["score"], layer["format"]
        # the down projection may use another format (the shipping mix)
        L.down_format = layer.get("down_format", layer["format"])
        for name in ("w_gate", "w_up", "w_down"):
            arr = layer[name]
            assert arr.dtype == np.uint8 and arr.flags["C_CONTIGUOUS"]
            setattr(L, name, arr.ctypes.data)
        L.gate_up_row_bytes = layer["gate_up_row_bytes"]
        L.down_row_bytes = layer["down_row_bytes"]
        L.gate_up_expert_stride = layer["gate_up_expert_stride"]
        L.down_expert_stride = layer["down_expert_stride"]
        cb = layer.get("codebook")
        L.codebook = cb.ctypes.data if cb is not None else None
        return L

    def moe_forward(self, layer, x_bf16: np.ndarray, logits: np.ndarray,
                    tokens: Optional[np.ndarray] = None):
        """Returns (y fp64 [n x H], ids [n x k], weights fp64 [n x k]) for the
        listed tokens (all when tokens is None)."""
        x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
        lg = np.ascontiguousarray(logits, dtype=np.float32)
        T = lg.shape[0]
        H, k = layer["hidden"], layer["top_k"]
        tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
        n = T if tok is None else tok.size
        y = np.empty((n, H), dtype=np.float64)
        ids = np.empty((n, k), dtype=np.int32)
        w = np.empty((n, k), dtype=np.float64)
        L = self._layer(layer)
        rc = self.lib.orc_moe_forward(ctypes.byref(L), _ptr(x), _ptr(lg), T, _ptr(tok), n,
                                      _ptr(y), _ptr(ids), _ptr(w))
        if rc != 0:
            raise ValueError(f"orc_moe_forward rejected its arguments (code {rc})")
        return y, ids, w

    def expert_ffn(self, layer, e: int, x_row_bf16: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x_row_bf16, dtype=np.uint16)
        o = np.empty(layer["hidden"], dtype=np.float64)
        L = self._layer(layer)
        rc = self.lib.orc_expert_ffn(ctypes.byref(L), e, _ptr(x), _ptr(o))
        if rc != 0:
            raise ValueError(f"orc_expert_ffn rejected its arguments (code {rc})")
        return o


_default: Optional[Oracle] = None


def get() -> Oracle:
    """The committed oracle, compiled on first use."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
