"""Pins for the reference oracle: checks against things other than the oracle
itself -- hand-derived worked blocks (tests/golden), exhaustive comparison of
the scalar decoders with numpy's own fp16 / fp32 types, independently written
vectorised dequantizers, brute-force routing, dense numpy fp64 matmuls, and
invariants of the layer (zero scales, power-of-two scaling, expert
relabelling, the k = 1 reduction).

Every pin takes an ``oracle.Oracle`` handle so that the same checks run on
the committed oracle and on copies with a planted mistake
(tests/test_oracle_mutants.py).  A pin raises AssertionError when it fails.
"""
from __future__ import annotations

import math
import os

import numpy as np

import ds4g_synth as S

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


# ---------------------------------------------------------------------------
# independent numpy dequantizers (vectorised; written from the block
# definitions, sharing nothing with the C oracle)
# ---------------------------------------------------------------------------

def np_q2k_dequant(blocks: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1, 84)
    n = b.shape[0]
    scales = b[:, :16]
    qs = b[:, 16:80].reshape(n, 2, 1, 32)                      # [block, half, 1, lane]
    shifts = np.array([0, 2, 4, 6], dtype=np.uint8).reshape(1, 1, 4, 1)
    q = ((qs >> shifts) & 3).reshape(n, 256).astype(np.float32)  # j = 128 half + 32 g + lane
    d = b[:, 80:82].copy().view(np.float16).astype(np.float32)   # [n, 1]
    dmin = b[:, 82:84].copy().view(np.float16).astype(np.float32)
    sc = np.repeat((scales & 15).astype(np.float32), 16, axis=1)
    mn = np.repeat((scales >> 4).astype(np.float32), 16, axis=1)
    return ((d * sc) * q - dmin * mn).reshape(-1)


def np_cb2_dequant(blocks: np.ndarray, codebook: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1, 70)
    n = b.shape[0]
    cb = np.asarray(codebook, dtype=np.int8).reshape(256, 8)
    entries = cb[b[:, :32].astype(np.int64)].astype(np.float32)          # [n, 32, 8]
    bits = (b[:, 32:64, None] >> np.arange(8, dtype=np.uint8)) & 1       # [n, 32, 8]
    nib = np.stack([b[:, 64:68] & 15, b[:, 64:68] >> 4], axis=2).reshape(n, 8)
    s = np.repeat(nib.astype(np.float32), 32, axis=1).reshape(n, 32, 8)
    d = b[:, 68:70].copy().view(np.float16).astype(np.float32).reshape(n, 1, 1)
    v = (d * s) * entries
    return np.where(bits == 1, -v, v).reshape(-1)


def _np_k4_scales(p: np.ndarray):
    """[n, 12] packed bytes -> ([n, 8] scales, [n, 8] mins) as integers."""
    p = p.astype(np.int64)
    sc = np.concatenate([p[:, 0:4] & 63, (p[:, 8:12] & 15) | ((p[:, 0:4] >> 6) << 4)], axis=1)
    mn = np.concatenate([p[:, 4:8] & 63, (p[:, 8:12] >> 4) | ((p[:, 4:8] >> 6) << 4)], axis=1)
    return sc, mn


def _np_half(b: np.ndarray) -> np.ndarray:
    return b.copy().view(np.float16).astype(np.float32)


def np_q4k_dequant(blocks: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1, 144)
    n = b.shape[0]
    d, dmin = _np_half(b[:, 0:2]), _np_half(b[:, 2:4])
    sc, mn = _np_k4_scales(b[:, 4:16])
    qs = b[:, 16:144].reshape(n, 4, 1, 32)
    q = np.concatenate([qs & 15, qs >> 4], axis=2).reshape(n, 256).astype(np.float32)
    scf = np.repeat(sc.astype(np.float32), 32, axis=1)
    mnf = np.repeat(mn.astype(np.float32), 32, axis=1)
    return ((d * scf) * q - dmin * mnf).reshape(-1)


def np_q5k_dequant(blocks: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1, 176)
    n = b.shape[0]
    d, dmin = _np_half(b[:, 0:2]), _np_half(b[:, 2:4])
    sc, mn = _np_k4_scales(b[:, 4:16])
    qh = b[:, 16:48]
    high = ((qh[:, None, :] >> np.arange(8, dtype=np.uint8)[None, :, None]) & 1).reshape(n, 256)
    qs = b[:, 48:176].reshape(n, 4, 1, 32)
    low = np.concatenate([qs & 15, qs >> 4], axis=2).reshape(n, 256)
    q = (low.astype(np.int64) + 16 * high.astype(np.int64)).astype(np.float32)
    scf = np.repeat(sc.astype(np.float32), 32, axis=1)
    mnf = np.repeat(mn.astype(np.float32), 32, axis=1)
    return ((d * scf) * q - dmin * mnf).reshape(-1)


def np_q6k_dequant(blocks: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1, 210)
    n = b.shape[0]
    ql = b[:, 0:128].reshape(n, 2, 1, 2, 32)                     # [n, half, nibble, v, lane]
    low = np.concatenate([ql & 15, ql >> 4], axis=2).reshape(n, 2, 4, 32)   # u = 2 nibble + v
    qh = b[:, 128:192].reshape(n, 2, 1, 32)
    high = (qh >> (2 * np.arange(4, dtype=np.uint8)).reshape(1, 1, 4, 1)) & 3
    q = (low.astype(np.int64) + 16 * high.astype(np.int64) - 32).reshape(n, 256).astype(np.float32)
    sc = np.repeat(b[:, 192:208].copy().view(np.int8).astype(np.float32), 16, axis=1)
    d = _np_half(b[:, 208:210])
    return ((d * sc) * q).reshape(-1)


def np_mxfp4_dequant(blocks: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1, 8, 17)
    e = b[:, :, 0].astype(np.int64)
    qs = b[:, :, 1:17]
    codes = np.concatenate([qs & 15, qs >> 4], axis=2).astype(np.int64)     # [n, 8, 32]
    mag = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])[codes & 7]
    val = np.where(codes & 8, -mag, mag)
    with np.errstate(over="ignore", invalid="ignore"):
        scale = np.where(e == 255, np.nan, np.ldexp(1.0, e - 127))
        return (scale[:, :, None] * val).astype(np.float32).reshape(-1)


_NP_BLOCK = {S.FMT_Q2K: 84, S.FMT_CB2: 70, S.FMT_Q4K: 144, S.FMT_Q5K: 176, S.FMT_Q6K: 210,
             S.FMT_MXFP4: 136}


def np_dense_weights(layer, name: str, K: int) -> np.ndarray:
    """[E, N, K] fp32 weights of one tensor, dequantized with the numpy
    routines above."""
    W = layer[name]
    E, N, rb = W.shape
    fmt = layer.get("down_format", layer["format"]) if name == "w_down" else layer["format"]
    bb = _NP_BLOCK[fmt]
    nblk = -(-K // 256)
    raw = np.ascontiguousarray(W[:, :, :nblk * bb]).reshape(-1)
    if fmt == S.FMT_Q2K:
        w = np_q2k_dequant(raw)
    elif fmt == S.FMT_CB2:
        w = np_cb2_dequant(raw, layer["codebook"])
    else:
        w = {S.FMT_Q4K: np_q4k_dequant, S.FMT_Q5K: np_q5k_dequant,
             S.FMT_Q6K: np_q6k_dequant, S.FMT_MXFP4: np_mxfp4_dequant}[fmt](raw)
    return w.reshape(E, N, nblk * 256)[:, :, :K]


def np_route(logits: np.ndarray, k: int, score: int):
    """Brute force: sort each row by (-logit, id) with NaN as -inf."""
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    for t in range(T):
        vals = [(-math.inf if math.isnan(v) else float(v)) for v in logits[t]]
        order = sorted(range(E), key=lambda e: (-vals[e], e))[:k]
        ids[t] = order
        sel = [vals[e] for e in order]
        if score == S.SCORE_SOFTMAX:
            ex = [math.exp(v - sel[0]) for v in sel]
        else:
            ex = [1.0 / (1.0 + math.exp(-v)) for v in sel]
        tot = sum(ex)
        w[t] = [v / tot for v in ex]
    return ids, w


def np_forward(layer, x_bf16, logits) -> np.ndarray:
    """Dense fp64 reference: y_t = sum_i w_ti W_down[e] (SiLU(W_gate[e] x) * W_up[e] x)."""
    H, I, k = layer["hidden"], layer["inter"], layer["top_k"]
    Wg = np_dense_weights(layer, "w_gate", H).astype(np.float64)
    Wu = np_dense_weights(layer, "w_up", H).astype(np.float64)
    Wd = np_dense_weights(layer, "w_down", I).astype(np.float64)
    x = S.bf16_to_f32(x_bf16).astype(np.float64)
    ids, w = np_route(logits, k, layer["score"])
    y = np.zeros((x.shape[0], H))
    for t in range(x.shape[0]):
        for i in range(k):
            e = ids[t, i]
            g = Wg[e] @ x[t]
            u = Wu[e] @ x[t]
            h = g / (1.0 + np.exp(-g)) * u
            y[t] += w[t, i] * (Wd[e] @ h)
    return y


def small_layer(seed=11, H=512, I=320, E=6, k=3, T=5, fmt=S.FMT_Q2K, score=S.SCORE_SOFTMAX,
                logits_kind=S.LOGITS_NORMAL, align=1, down_fmt=None):
    cfg = S.Config("pin", H, I, E, k, T, fmt, score, logits_kind, seed, row_align=align,
                   down_format=down_fmt)
    return S.make_layer(cfg)


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_half_decode(orc):
    """All 65536 fp16 bit patterns against numpy's float16."""
    ref = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(i) for i in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_bf16_decode(orc):
    """All 65536 bf16 bit patterns against the upper half of a numpy float32."""
    with np.errstate(invalid="ignore"):
        ref = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    got = np.array([orc.bf16_to_double(i) for i in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_q2k_onehot(orc):
    for B, val, j, w in _rows("q2k_onehot.txt"):
        blk = np.zeros(84, dtype=np.uint8)
        blk[:16] = 0x01
        blk[80:82] = [0x00, 0x3C]
        blk[16 + int(B)] = int(val, 16)
        out = orc.q2k_dequant(blk)
        exp = np.zeros(256, dtype=np.float32)
        exp[int(j)] = float(w)
        assert np.array_equal(out, exp), (B, val, np.nonzero(out))


def pin_q2k_scale_min(orc):
    for s, sb, fill, dbits, mbits, val in _rows("q2k_scale_min.txt"):
        blk = np.zeros(84, dtype=np.uint8)
        blk[16:80] = int(fill, 16)
        blk[int(s)] = int(sb, 16)
        d, m = int(dbits, 16), int(mbits, 16)
        blk[80:84] = [d & 0xFF, d >> 8, m & 0xFF, m >> 8]
        out = orc.q2k_dequant(blk)
        exp = np.zeros(256, dtype=np.float32)
        exp[16 * int(s):16 * int(s) + 16] = float(val)
        assert np.array_equal(out, exp), (s, sb, out[16 * int(s)])


def _random_q2k_blocks(rng, n):
    blk = rng.integers(0, 256, size=(n, 84), dtype=np.uint8)
    # finite d / dmin: fp16 exponent field below 31
    for off in (80, 82):
        h = rng.integers(0, 0x7C00, size=n).astype(np.uint16)
        h |= (rng.integers(0, 2, size=n).astype(np.uint16) << 15)
        blk[:, off:off + 2] = h.view(np.uint8).reshape(n, 2)
    return blk


def pin_q2k_zero_scale(orc):
    rng = np.random.default_rng(1)
    blk = _random_q2k_blocks(rng, 64)
    blk[:, :16] = 0
    out = orc.q2k_dequant(blk)
    assert np.all(out == 0.0)


def pin_q2k_numpy(orc):
    """Random blocks: bit-exact agreement with the independent numpy decoder."""
    rng = np.random.default_rng(2)
    blk = _random_q2k_blocks(rng, 512)
    got = orc.q2k_dequant(blk)
    ref = np_q2k_dequant(blk)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def _put_half(blk, off, bits):
    blk[off] = bits & 0xFF
    blk[off + 1] = bits >> 8


def pin_q4k_worked(orc):
    for s, p, fill, dbits, mbits, val in _rows("q4k_worked.txt"):
        blk = np.zeros(144, dtype=np.uint8)
        _put_half(blk, 0, int(dbits, 16))
        _put_half(blk, 2, int(mbits, 16))
        blk[4:16] = np.frombuffer(bytes.fromhex(p), dtype=np.uint8)
        blk[16:] = int(fill, 16)
        out = orc.q4k_dequant(blk)
        exp = np.zeros(256, dtype=np.float32)
        exp[32 * int(s):32 * int(s) + 32] = float(val)
        assert np.array_equal(out, exp), (s, out[32 * int(s)], np.nonzero(out)[0][:4])


def pin_q5k_worked(orc):
    for s, p, qsf, qhf, dbits, mbits, val in _rows("q5k_worked.txt"):
        blk = np.zeros(176, dtype=np.uint8)
        _put_half(blk, 0, int(dbits, 16))
        _put_half(blk, 2, int(mbits, 16))
        blk[4:16] = np.frombuffer(bytes.fromhex(p), dtype=np.uint8)
        blk[16:48] = int(qhf, 16)
        blk[48:] = int(qsf, 16)
        out = orc.q5k_dequant(blk)
        exp = np.zeros(256, dtype=np.float32)
        exp[32 * int(s):32 * int(s) + 32] = float(val)
        assert np.array_equal(out, exp), (s, out[32 * int(s)], np.nonzero(out)[0][:4])


def pin_q6k_worked(orc):
    for t, sc, qlf, qhf, dbits, val in _rows("q6k_worked.txt"):
        blk = np.zeros(210, dtype=np.uint8)
        blk[0:128] = int(qlf, 16)
        blk[128:192] = int(qhf, 16)
        blk[192 + int(t)] = np.int8(int(sc)).view(np.uint8)
        _put_half(blk, 208, int(dbits, 16))
        out = orc.q6k_dequant(blk)
        exp = np.zeros(256, dtype=np.float32)
        exp[16 * int(t):16 * int(t) + 16] = float(val)
        assert np.array_equal(out, exp), (t, out[16 * int(t)], np.nonzero(out)[0][:4])


def pin_kquant_onehot(orc):
    for row in _rows("kquant_onehot.txt"):
        fmt, field, idx, val = row[0], row[1], int(row[2]), int(row[3], 16)
        listed = dict((int(a), float(b)) for a, b in (c.split(":") for c in row[4:]))
        if fmt in ("q4k", "q5k"):
            bb = 144 if fmt == "q4k" else 176
            blk = np.zeros(bb, dtype=np.uint8)
            _put_half(blk, 0, 0x3C00)
            blk[4:16] = [1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1]
            base = {"qs": 16 if fmt == "q4k" else 48, "qh": 16}[field]
            blk[base + idx] = val
            out = (orc.q4k_dequant if fmt == "q4k" else orc.q5k_dequant)(blk)
            exp = np.zeros(256, dtype=np.float32)
        else:
            blk = np.zeros(210, dtype=np.uint8)
            blk[192:208] = 1
            _put_half(blk, 208, 0x3C00)
            blk[{"ql": 0, "qh": 128}[field] + idx] = val
            out = orc.q6k_dequant(blk)
            exp = np.full(256, -32.0, dtype=np.float32)
        for j, w in listed.items():
            exp[j] = w
        assert np.array_equal(out, exp), (row, np.nonzero(out != exp)[0][:6])


def _random_kquant_blocks(rng, n, bb, half_offsets):
    blk = rng.integers(0, 256, size=(n, bb), dtype=np.uint8)
    for off in half_offsets:                  # finite fp16 fields
        h = rng.integers(0, 0x7C00, size=n).astype(np.uint16)
        h |= (rng.integers(0, 2, size=n).astype(np.uint16) << 15)
        blk[:, off:off + 2] = h.view(np.uint8).reshape(n, 2)
    return blk


def pin_kquant_numpy(orc):
    """Random blocks of each K-quant format: bit-exact agreement with the
    independent numpy decoders."""
    rng = np.random.default_rng(21)
    for bb, offs, fo, fn in ((144, (0, 2), orc.q4k_dequant, np_q4k_dequant),
                             (176, (0, 2), orc.q5k_dequant, np_q5k_dequant),
                             (210, (208,), orc.q6k_dequant, np_q6k_dequant)):
        blk = _random_kquant_blocks(rng, 512, bb, offs)
        got = fo(blk)
        ref = fn(blk)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), bb


def pin_mxfp4_worked(orc):
    for sb, e, i, byte, wl, wh in _rows("mxfp4_worked.txt"):
        sb, i = int(sb), int(i)
        blk = np.zeros(136, dtype=np.uint8)
        blk[0::17] = 127
        blk[17 * sb] = int(e)
        blk[17 * sb + 1 + i] = int(byte, 16)
        out = orc.mxfp4_dequant(blk)
        exp = np.zeros(256, dtype=np.float32)
        exp[32 * sb + i] = float(wl)
        exp[32 * sb + 16 + i] = float(wh)
        assert np.array_equal(out, exp), (sb, i, out[32 * sb + i], out[32 * sb + 16 + i])
        assert np.array_equal(np.signbit(out), np.signbit(exp)), (sb, i, "sign of zero")


def pin_mxfp4_numpy(orc):
    """Random MXFP4 units (scale bytes below 255): bit-exact agreement with
    the independent numpy decoder."""
    rng = np.random.default_rng(23)
    blk = rng.integers(0, 256, size=(512, 136), dtype=np.uint8)
    blk[:, 0::17] = rng.integers(0, 255, size=(512, 8), dtype=np.uint8)
    got = orc.mxfp4_dequant(blk)
    ref = np_mxfp4_dequant(blk)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def _worked_codebook():
    cb = np.zeros((256, 8), dtype=np.int8)
    cb[0] = [8, -8, 25, -25, 43, -43, 8, 8]
    cb[1] = [43, 43, 43, 43, -8, -8, -8, -8]
    cb[7] = [25] * 8
    return cb


def pin_cb2_worked(orc):
    cb = _worked_codebook()
    for row in _rows("cb2_worked.txt"):
        o, idx, sgn = int(row[0]), int(row[1]), int(row[2], 16)
        sc = [int(v, 16) for v in row[3:7]]
        d = int(row[7], 16)
        w = [float(v) for v in row[8:16]]
        blk = np.zeros(70, dtype=np.uint8)
        blk[:32] = 2
        blk[o] = idx
        blk[32 + o] = sgn
        blk[64:68] = sc
        blk[68:70] = [d & 0xFF, d >> 8]
        out = orc.cb2_dequant(blk, cb)
        exp = np.zeros(256, dtype=np.float32)
        exp[8 * o:8 * o + 8] = w
        assert np.array_equal(out, exp), (row, out[8 * o:8 * o + 8])


def pin_cb2_numpy(orc):
    rng = np.random.default_rng(3)
    cb = S.make_codebook(4)
    blk = rng.integers(0, 256, size=(256, 70), dtype=np.uint8)
    h = rng.integers(0, 0x7C00, size=256).astype(np.uint16)
    blk[:, 68:70] = h.view(np.uint8).reshape(256, 2)
    got = orc.cb2_dequant(blk, cb)
    ref = np_cb2_dequant(blk, cb)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def pin_route_worked(orc):
    for row in _rows("routing_worked.txt"):
        score = S.SCORE_SOFTMAX if row[0] == "softmax" else S.SCORE_SIGMOID
        k = int(row[1])
        logits = np.array([[float(v) for v in row[2].split(",")]], dtype=np.float32)
        ids = [int(v) for v in row[4].split(",")]
        w = [float(v) for v in row[5].split(",")]
        r = orc.route(logits, k, score)
        assert r["ids"][0].tolist() == ids, (row, r["ids"])
        assert np.allclose(r["weights"][0], w, rtol=0, atol=5e-12), (row, r["weights"])


def pin_route_bruteforce(orc):
    rng = np.random.default_rng(4)
    for score in (S.SCORE_SOFTMAX, S.SCORE_SIGMOID):
        for E, k in ((8, 2), (13, 5), (64, 6), (256, 8), (5, 5)):
            T = 9
            lg = rng.integers(-4, 5, size=(T, E)).astype(np.float32) * 0.5   # many exact ties
            if E > 8:
                lg[0, 3] = np.nan
            r = orc.route(lg, k, score)
            ids, w = np_route(lg, k, score)
            assert np.array_equal(r["ids"], ids)
            assert np.allclose(r["weights"], w, rtol=1e-13, atol=0)
            assert np.allclose(r["weights"].sum(axis=1), 1.0, rtol=0, atol=1e-12)
            flat = ids.reshape(-1)
            counts = np.bincount(flat, minlength=E)
            assert np.array_equal(r["counts"], counts)
            assert np.array_equal(r["offsets"], np.concatenate([[0], np.cumsum(counts)]))
            order = sorted(range(T * k), key=lambda a: (flat[a], a // k))
            assert r["perm"].tolist() == order


def pin_route_full_k(orc):
    """k = E: the ids are the whole stable descending argsort."""
    rng = np.random.default_rng(5)
    E = 16
    lg = rng.standard_normal((4, E)).astype(np.float32)
    lg[1, :] = 0.25
    r = orc.route(lg, E, S.SCORE_SIGMOID)
    for t in range(4):
        assert r["ids"][t].tolist() == sorted(range(E), key=lambda e: (-float(lg[t, e]), e))


def pin_forward_dense(orc):
    """Oracle forward against the dense numpy fp64 reference: the tiny
    workload, a padded-I layer, a sigmoid layer, a codebook layer, the two
    mixed layers (codebook gate/up with Q2_K down -- the shipping mix -- and
    the reverse, so that a format read for the wrong matrix fails), and
    layers in the K-quant formats."""
    layers = [S.make_layer(S.CONFIGS["tiny"]),
              small_layer(),
              small_layer(seed=12, I=256 + 40, score=S.SCORE_SIGMOID, logits_kind=S.LOGITS_UNIFORM),
              small_layer(seed=13, H=512, I=256, E=5, k=2, T=3, fmt=S.FMT_CB2, align=16),
              small_layer(seed=15, H=512, I=320, E=5, k=2, T=3, fmt=S.FMT_CB2, align=16,
                          down_fmt=S.FMT_Q2K),
              small_layer(seed=16, H=512, I=256, E=4, k=2, T=3, fmt=S.FMT_Q2K, align=16,
                          down_fmt=S.FMT_CB2),
              # the higher-bit routed formats: Q4_K gate/up with Q6_K down,
              # Q5_K throughout, and Q2_K gate/up with Q4_K down
              small_layer(seed=17, H=512, I=320, E=5, k=2, T=3, fmt=S.FMT_Q4K,
                          down_fmt=S.FMT_Q6K),
              small_layer(seed=18, H=512, I=256, E=4, k=2, T=3, fmt=S.FMT_Q5K),
              small_layer(seed=19, H=512, I=256, E=4, k=2, T=3, fmt=S.FMT_Q2K,
                          down_fmt=S.FMT_Q4K),
              small_layer(seed=20, H=512, I=320, E=4, k=2, T=3, fmt=S.FMT_MXFP4)]
    for L in layers:
        y, ids, w = orc.moe_forward(L, L["x"], L["logits"])
        ref = np_forward(L, L["x"], L["logits"])
        scale = np.abs(ref).max()
        assert scale > 0
        assert np.abs(y - ref).max() <= 1e-12 * scale, (L["name"], np.abs(y - ref).max(), scale)


def pin_forward_zero_scale(orc):
    """All-zero scale bytes in W_down => y == 0 exactly; zero scales in one
    expert's W_gate => that expert contributes nothing."""
    L = small_layer(seed=14)
    L["w_down"][:, :, :] = 0
    y, _, _ = orc.moe_forward(L, L["x"], L["logits"])
    assert np.all(y == 0.0)
    L = small_layer(seed=15, E=4, k=2, T=6)
    ids, _ = np_route(L["logits"], 2, L["score"])
    e0 = int(ids[0, 0])
    H = L["hidden"]
    nblk = H // 256
    for b in range(nblk):
        L["w_gate"][e0, :, 84 * b:84 * b + 16] = 0
    y, _, _ = orc.moe_forward(L, L["x"], L["logits"])
    ref = np_forward(L, L["x"], L["logits"])
    assert np.abs(y - ref).max() <= 1e-12 * np.abs(ref).max()
    # token 0's output now comes from slot 1 alone
    Wd = np_dense_weights(L, "w_down", L["inter"]).astype(np.float64)
    Wg = np_dense_weights(L, "w_gate", H).astype(np.float64)
    Wu = np_dense_weights(L, "w_up", H).astype(np.float64)
    assert np.all(Wg[e0] == 0)
    x0 = S.bf16_to_f32(L["x"][0]).astype(np.float64)
    _, w = np_route(L["logits"], 2, L["score"])
    e1 = int(ids[0, 1])
    g = Wg[e1] @ x0
    h = g / (1 + np.exp(-g)) * (Wu[e1] @ x0)
    assert np.allclose(y[0], w[0, 1] * (Wd[e1] @ h), rtol=1e-12, atol=1e-15)


def pin_forward_k1_single(orc):
    """One expert, k = 1: the layer is exactly that expert's FFN (weight 1)."""
    L = small_layer(seed=16, E=1, k=1, T=3)
    y, ids, w = orc.moe_forward(L, L["x"], L["logits"])
    assert np.all(ids == 0) and np.all(w == 1.0)
    for t in range(3):
        o = orc.expert_ffn(L, 0, L["x"][t])
        assert np.array_equal(y[t], o)
    ref = np_forward(L, L["x"], L["logits"])
    assert np.abs(y - ref).max() <= 1e-12 * np.abs(ref).max()


def pin_forward_scale_pow2(orc):
    """Doubling d and dmin of every W_down block (fp16 exponent + 1) doubles y
    exactly."""
    L = small_layer(seed=17)
    y1, _, _ = orc.moe_forward(L, L["x"], L["logits"])
    W = L["w_down"]
    nblk = -(-L["inter"] // 256)
    for b in range(nblk):
        for off in (80, 82):
            h = W[:, :, 84 * b + off:84 * b + off + 2].copy().view(np.uint16)
            nz = (h & 0x7FFF) != 0
            assert np.all(((h >> 10) & 31)[nz] < 30)
            h[nz] += 1 << 10
            W[:, :, 84 * b + off:84 * b + off + 2] = h.view(np.uint8)
    y2, _, _ = orc.moe_forward(L, L["x"], L["logits"])
    assert np.array_equal(y2, 2.0 * y1)


def pin_forward_relabel(orc):
    """Permuting the expert ids (weights and logit columns together) leaves y
    unchanged, bit for bit."""
    L = small_layer(seed=18, E=7, k=3, T=6)
    y1, ids1, _ = orc.moe_forward(L, L["x"], L["logits"])
    pi = np.array([3, 6, 0, 5, 1, 4, 2])           # new id of old expert e
    L2 = dict(L)
    for name in ("w_gate", "w_up", "w_down"):
        W = np.empty_like(L[name])
        W[pi] = L[name]
        L2[name] = W
    lg = np.empty_like(L["logits"])
    lg[:, pi] = L["logits"]
    y2, ids2, _ = orc.moe_forward(L2, L["x"], lg)
    assert np.array_equal(ids2, pi[ids1])
    assert np.array_equal(y1, y2)


def pin_quantizer_roundtrip(orc):
    """Encoder (input generator) -> oracle decoder round trip: every weight
    lands within one quantization step of its drawn value (Q2_K: one step of
    d * sc plus the min rounding; codebook: the 32-group's largest scale), and
    the reconstruction keeps most of the signal."""
    rng = np.random.default_rng(6)
    w = (0.02 * rng.standard_normal((64, 256))).astype(np.float32)
    blk = S.q2k_encode(w)
    rec = orc.q2k_dequant(blk).reshape(64, 256)
    d = blk[:, 80:82].copy().view(np.float16).astype(np.float64)
    dmin = blk[:, 82:84].copy().view(np.float16).astype(np.float64)
    step = np.repeat((blk[:, :16] & 15).astype(np.float64), 16, axis=1) * d
    bound = step * 0.5 + 0.5 * dmin + 0.5 * d * 3
    assert np.all(np.abs(rec - w) <= bound + 1e-7)
    assert np.linalg.norm(rec - w) / np.linalg.norm(w) < 0.5
    cb = S.make_codebook(4)
    blk = S.cb2_encode(w, cb)
    rec = orc.cb2_dequant(blk, cb).reshape(64, 256)
    assert np.all(np.sign(rec)[np.abs(w) > 1e-3] * np.sign(w)[np.abs(w) > 1e-3] >= 0)
    assert np.linalg.norm(rec - w) / np.linalg.norm(w) < 0.8


ALL_PINS = [
    pin_half_decode, pin_bf16_decode, pin_q2k_onehot, pin_q2k_scale_min,
    pin_q2k_zero_scale, pin_q2k_numpy, pin_cb2_worked, pin_cb2_numpy,
    pin_q4k_worked, pin_q5k_worked, pin_q6k_worked, pin_kquant_onehot, pin_kquant_numpy,
    pin_mxfp4_worked, pin_mxfp4_numpy,
    pin_route_worked, pin_route_bruteforce, pin_route_full_k,
    pin_forward_dense, pin_forward_zero_scale, pin_forward_k1_single,
    pin_forward_scale_pow2, pin_forward_relabel, pin_quantizer_roundtrip,
]
