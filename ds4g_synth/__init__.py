"""Seeded synthetic inputs for the routed-MoE expert layer.

Shared by the tests, the oracle runs and the benchmark.  This module holds
input recipes only (random draws, bf16 rounding of activations, router-logit
recipes, the encoders that turn drawn fp32 weights into 2-bit blocks); it
computes no step of the layer.  The heavy lifting is in ``synth.c``
(counter-based splitmix64 streams, threaded; bytes independent of the thread
count).

Workloads (the layer shapes of the five synthetic configurations):

=============  =====  ====  ===  ==  ====  ========  =======  ====
name           H      I     E    k   T     format    score    seed
=============  =====  ====  ===  ==  ====  ========  =======  ====
tiny           256    128   8    2   4     Q2_K      softmax  0
decode_1tok    4096   1536  64   6   1     Q2_K      softmax  1
decode_32tok   7168   2048  256  8   32    Q2_K      sigmoid  2
prefill_2048   7168   2048  256  8   2048  Q2_K      sigmoid  3
codebook_512   7168   2048  256  8   512   codebook  sigmoid  4
mixed_2048     7168   2048  256  8   2048  mixed     sigmoid  5
kquant_32tok   7168   2048  256  8   32    Q4_K/Q6K  sigmoid  6
mxfp4_32tok    7168   2048  256  8   32    MXFP4     sigmoid  7
mxfp4_2048     7168   2048  256  8   2048  MXFP4     sigmoid  8
=============  =====  ====  ===  ==  ====  ========  =======  ====

mixed_2048 is the shipping mix of the ds4 weights (codebook-2-bit gate/up,
Q2_K down) on the prefill layer with the prefill routing recipe.
kquant_32tok is a higher-bit routed layer (Q4_K gate/up, Q6_K down; the
ds4f-q2-q4 / ds4f-q4 downloads and the routed K-quant formats the ds4
README names) at the 32-token decode batch; mxfp4_32tok the same layer with
MXFP4 routed experts (the ds4f-mxfp4 download), and mxfp4_2048 those experts
on the prefill layer with the prefill routing recipe.

Rows are stored packed (ceil(K/256) blocks back to back) for Q2_K; the
codebook rows (70-byte blocks) are padded to a multiple of 16 bytes so that
the tensor-core path can stage them with TMA (1960 -> 1968 bytes).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
from typing import Dict, Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "synth.c")
LIBRARY = os.path.join(HERE, "libds4g_synth.so")

QK = 256
FMT_Q2K, FMT_CB2, FMT_Q4K, FMT_Q5K, FMT_Q6K, FMT_MXFP4 = 0, 1, 2, 3, 4, 5
# bytes per 256 weights (MXFP4: eight 17-byte blocks of 32)
BLOCK_BYTES = {FMT_Q2K: 84, FMT_CB2: 70, FMT_Q4K: 144, FMT_Q5K: 176, FMT_Q6K: 210,
               FMT_MXFP4: 136}
SCORE_SOFTMAX, SCORE_SIGMOID = 0, 1
LOGITS_NORMAL, LOGITS_UNIFORM, LOGITS_BIASED, LOGITS_ZIPF = 0, 1, 2, 3
TENSOR_GATE, TENSOR_UP, TENSOR_DOWN = 3, 4, 5
WEIGHT_SD = 0.02
MARGIN = 1e-3
ZIPF_S = 1.1


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    hidden: int
    inter: int
    n_experts: int
    top_k: int
    tokens: int
    format: int
    score: int
    logits: int
    seed: int
    row_align: int = 1
    down_format: Optional[int] = None      # W_down's format when it differs (mixed layers)

    @property
    def dn_format(self) -> int:
        return self.format if self.down_format is None else self.down_format

    @property
    def block_bytes(self) -> int:
        """Bytes of one W_gate / W_up super-block."""
        return BLOCK_BYTES[self.format]

    @property
    def down_block_bytes(self) -> int:
        return BLOCK_BYTES[self.dn_format]

    def row_bytes(self, K: int, align: Optional[int] = None, fmt: Optional[int] = None) -> int:
        """Row stride: ceil(K/256) blocks of `fmt` (default: the gate/up
        format), padded up to `align` bytes (default: the configuration's
        own row alignment)."""
        align = self.row_align if align is None else align
        fmt = self.format if fmt is None else fmt
        logical = -(-K // QK) * BLOCK_BYTES[fmt]
        return -(-logical // align) * align


CONFIGS: Dict[str, Config] = {
    c.name: c for c in [
        Config("tiny", 256, 128, 8, 2, 4, FMT_Q2K, SCORE_SOFTMAX, LOGITS_NORMAL, 0),
        Config("decode_1tok", 4096, 1536, 64, 6, 1, FMT_Q2K, SCORE_SOFTMAX, LOGITS_NORMAL, 1),
        Config("decode_32tok", 7168, 2048, 256, 8, 32, FMT_Q2K, SCORE_SIGMOID, LOGITS_UNIFORM, 2),
        Config("prefill_2048", 7168, 2048, 256, 8, 2048, FMT_Q2K, SCORE_SIGMOID, LOGITS_BIASED, 3),
        Config("codebook_512", 7168, 2048, 256, 8, 512, FMT_CB2, SCORE_SIGMOID, LOGITS_ZIPF, 4,
               row_align=16),
        Config("mixed_2048", 7168, 2048, 256, 8, 2048, FMT_CB2, SCORE_SIGMOID, LOGITS_BIASED, 5,
               row_align=16, down_format=FMT_Q2K),
        Config("kquant_32tok", 7168, 2048, 256, 8, 32, FMT_Q4K, SCORE_SIGMOID, LOGITS_UNIFORM, 6,
               down_format=FMT_Q6K),
        Config("mxfp4_32tok", 7168, 2048, 256, 8, 32, FMT_MXFP4, SCORE_SIGMOID, LOGITS_UNIFORM, 7),
        Config("mxfp4_2048", 7168, 2048, 256, 8, 2048, FMT_MXFP4, SCORE_SIGMOID, LOGITS_BIASED, 8),
    ]
}


def build(source: str = SOURCE, out: str = LIBRARY) -> str:
    cmd = ["gcc", "-O3", "-std=gnu99", "-ffp-contract=off", "-fPIC", "-shared",
           "-pthread", "-o", out, source, "-lm"]
    subprocess.run(cmd, check=True)
    return out


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIBRARY):
            build()
        L = ctypes.CDLL(LIBRARY)
        u64, i32, i64, vp, dbl = (ctypes.c_uint64, ctypes.c_int32, ctypes.c_int64,
                                  ctypes.c_void_p, ctypes.c_double)
        L.syn_key.argtypes = [u64, u64, u64]
        L.syn_key.restype = u64
        L.syn_uniform.argtypes = [u64, u64]
        L.syn_uniform.restype = dbl
        L.syn_normal.argtypes = [u64, u64]
        L.syn_normal.restype = dbl
        L.syn_draw.argtypes = [u64, u64]
        L.syn_draw.restype = u64
        L.syn_f32_to_bf16.argtypes = [ctypes.c_float]
        L.syn_f32_to_bf16.restype = ctypes.c_uint16
        L.syn_double_to_half.argtypes = [dbl]
        L.syn_double_to_half.restype = ctypes.c_uint16
        L.syn_q2k_encode_block.argtypes = [vp, vp]
        L.syn_q2k_encode_block.restype = None
        L.syn_cb2_encode_block.argtypes = [vp, vp, vp]
        L.syn_cb2_encode_block.restype = None
        for fn in ("syn_q4k_encode_block", "syn_q5k_encode_block", "syn_q6k_encode_block",
                   "syn_mxfp4_encode_block"):
            getattr(L, fn).argtypes = [vp, vp]
            getattr(L, fn).restype = None
        L.syn_make_codebook.argtypes = [u64, vp]
        L.syn_make_codebook.restype = None
        L.syn_make_experts.argtypes = [u64, i32, i32, i32, i32, i32, i64, dbl, vp, vp, i32]
        L.syn_make_experts.restype = ctypes.c_int
        L.syn_make_x.argtypes = [u64, i32, i32, vp]
        L.syn_make_x.restype = None
        L.syn_make_logits.argtypes = [u64, i32, i32, i32, i32, dbl, dbl, vp]
        L.syn_make_logits.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bits (uint16), round to nearest even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = ((u & 0x7F800000) == 0x7F800000) & ((u & 0x007FFFFF) != 0)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = 0x7FC0
    return r


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def q2k_encode(w: np.ndarray) -> np.ndarray:
    """Encodes fp32 weights (multiple of 256) into Q2_K blocks."""
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(-1, QK)
    out = np.zeros((w.shape[0], 84), dtype=np.uint8)
    for b in range(w.shape[0]):
        lib().syn_q2k_encode_block(_p(w[b]), _p(out[b]))
    return out


def kquant_encode(w: np.ndarray, fmt: int) -> np.ndarray:
    """Encodes fp32 weights (multiple of 256) into Q4_K / Q5_K / Q6_K blocks."""
    fn = {FMT_Q4K: "syn_q4k_encode_block", FMT_Q5K: "syn_q5k_encode_block",
          FMT_Q6K: "syn_q6k_encode_block", FMT_MXFP4: "syn_mxfp4_encode_block"}[fmt]
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(-1, QK)
    out = np.zeros((w.shape[0], BLOCK_BYTES[fmt]), dtype=np.uint8)
    f = getattr(lib(), fn)
    for b in range(w.shape[0]):
        f(_p(w[b]), _p(out[b]))
    return out


def cb2_encode(w: np.ndarray, codebook: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(-1, QK)
    cb = np.ascontiguousarray(codebook, dtype=np.int8)
    out = np.zeros((w.shape[0], 70), dtype=np.uint8)
    for b in range(w.shape[0]):
        lib().syn_cb2_encode_block(_p(w[b]), _p(cb), _p(out[b]))
    return out


def make_codebook(seed: int) -> np.ndarray:
    cb = np.empty((256, 8), dtype=np.int8)
    lib().syn_make_codebook(seed, _p(cb))
    return cb


def make_experts(seed: int, tensor: int, E: int, N: int, K: int, fmt: int,
                 row_bytes: int, codebook: Optional[np.ndarray] = None,
                 sd: float = WEIGHT_SD, out: Optional[np.ndarray] = None,
                 n_threads: Optional[int] = None) -> np.ndarray:
    """E x N x row_bytes uint8: N(0, sd) weights encoded row by row."""
    if out is None:
        out = np.empty((E, N, row_bytes), dtype=np.uint8)
    assert out.shape == (E, N, row_bytes) and out.dtype == np.uint8 and out.flags["C_CONTIGUOUS"]
    cbp = _p(codebook) if codebook is not None else None
    rc = lib().syn_make_experts(seed, tensor, E, N, K, fmt, row_bytes, sd, cbp, _p(out),
                                n_threads or threads())
    if rc != 0:
        raise ValueError("syn_make_experts rejected its arguments")
    return out


def make_x(seed: int, T: int, H: int) -> np.ndarray:
    x = np.empty((T, H), dtype=np.uint16)
    lib().syn_make_x(seed, T, H, _p(x))
    return x


def make_logits(seed: int, kind: int, T: int, E: int, k: int,
                margin: float = MARGIN, zipf_s: float = ZIPF_S) -> np.ndarray:
    out = np.empty((T, E), dtype=np.float32)
    rc = lib().syn_make_logits(seed, kind, T, E, k, margin, zipf_s, _p(out))
    if rc != 0:
        raise ValueError("syn_make_logits rejected its arguments")
    return out


def make_layer(cfg: Config, tokens: Optional[int] = None, seed: Optional[int] = None,
               align: Optional[int] = None) -> dict:
    """All inputs of one configuration as host numpy arrays.

    Returns a dict with the layer description (hidden, inter, n_experts,
    top_k, score, format (W_gate / W_up), down_format, strides) plus w_gate /
    w_up / w_down (uint8 [E x N x row_bytes]), codebook (int8 [256 x 8] or
    None), x (bf16 bits [T x H]) and logits (fp32 [T x E]).
    """
    seed = cfg.seed if seed is None else seed
    T = cfg.tokens if tokens is None else tokens
    H, I, E, k = cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k
    codebook = make_codebook(seed) if FMT_CB2 in (cfg.format, cfg.dn_format) else None
    gu_rb = cfg.row_bytes(H, align)
    dn_rb = cfg.row_bytes(I, align, cfg.dn_format)
    layer = dict(
        name=cfg.name, hidden=H, inter=I, n_experts=E, top_k=k, score=cfg.score,
        format=cfg.format, down_format=cfg.dn_format, tokens=T,
        gate_up_row_bytes=gu_rb, down_row_bytes=dn_rb,
        gate_up_expert_stride=I * gu_rb, down_expert_stride=H * dn_rb,
        codebook=codebook,
    )
    layer["w_gate"] = make_experts(seed, TENSOR_GATE, E, I, H, cfg.format, gu_rb, codebook)
    layer["w_up"] = make_experts(seed, TENSOR_UP, E, I, H, cfg.format, gu_rb, codebook)
    layer["w_down"] = make_experts(seed, TENSOR_DOWN, E, H, I, cfg.dn_format, dn_rb, codebook)
    layer["x"] = make_x(seed, T, H)
    layer["logits"] = make_logits(seed, cfg.logits, T, E, k)
    return layer


def make_tokens(cfg: Config, T: int, seed: int) -> dict:
    """Fresh activations and logits (for a new batch over the same layer)."""
    return dict(x=make_x(seed, T, cfg.hidden),
                logits=make_logits(seed, cfg.logits, T, cfg.n_experts, cfg.top_k))
