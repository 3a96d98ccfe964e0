"""ds4g_q2k_dequant / ds4g_cb2_dequant against the oracle: fp32 bit-exact,
fp16 and bf16 equal to the round-to-nearest-even of the oracle's fp32."""
import numpy as np
import pytest
import torch

import bit_quantized_routed_route_b300 as D
import ds4g_synth as S
import oracle_pins as P

pytestmark = pytest.mark.gpu


def _rne_f16(f):
    # random d up to 65504 times a scale of 15 overflows fp16 on purpose: the
    # library's fp16 output must then be the same infinity as RNE gives
    with np.errstate(over="ignore"):
        return f.astype(np.float16).view(np.uint16)


def _random_q2k(n, seed):
    rng = np.random.default_rng(seed)
    blk = rng.integers(0, 256, size=(n, 84), dtype=np.uint8)
    for off in (80, 82):
        h = rng.integers(0, 0x7C00, size=n).astype(np.uint16)
        h |= rng.integers(0, 2, size=n).astype(np.uint16) << 15
        blk[:, off:off + 2] = h.view(np.uint8).reshape(n, 2)
    return blk


def _run(fn, blocks, n, dtype, *extra):
    dev = torch.device("cuda")
    bd = torch.from_numpy(np.ascontiguousarray(blocks).reshape(-1)).to(dev)
    tdt = {D.F32: torch.float32, D.F16: torch.float16, D.BF16: torch.bfloat16}[dtype]
    out = torch.full((n * 256,), float("nan"), dtype=tdt, device=dev)
    extra = [torch.from_numpy(e).to(dev) if isinstance(e, np.ndarray) else e for e in extra]
    if extra:
        D.check(fn(bd, n, extra[0], out, dtype))
    else:
        D.check(fn(bd, n, out, dtype))
    torch.cuda.synchronize()
    if dtype == D.F32:
        return out.cpu().numpy()
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("n", [1, 3, 37, 4096 + 5, 300_000])
def test_q2k_dequant_bit_exact(orc, n):
    blk = _random_q2k(n, n)
    ref = orc.q2k_dequant(blk)
    got = _run(D.q2k_dequant, blk, n, D.F32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(_run(D.q2k_dequant, blk, n, D.F16), _rne_f16(ref))
    assert np.array_equal(_run(D.q2k_dequant, blk, n, D.BF16), S.f32_to_bf16(ref))


def test_q2k_dequant_generated_rows(orc):
    W = S.make_experts(9, S.TENSOR_GATE, 2, 64, 4096, S.FMT_Q2K, 1344)
    ref = orc.q2k_dequant(W)
    got = _run(D.q2k_dequant, W, W.size // 84, D.F32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("n", [1, 2, 33, 70_001])
def test_cb2_dequant_bit_exact(orc, n):
    rng = np.random.default_rng(n)
    cb = S.make_codebook(4)
    blk = rng.integers(0, 256, size=(n, 70), dtype=np.uint8)
    h = rng.integers(0, 0x7C00, size=n).astype(np.uint16)
    blk[:, 68:70] = h.view(np.uint8).reshape(n, 2)
    ref = orc.cb2_dequant(blk, cb)
    got = _run(D.cb2_dequant, blk, n, D.F32, cb)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(_run(D.cb2_dequant, blk, n, D.F16, cb), _rne_f16(ref))
    assert np.array_equal(_run(D.cb2_dequant, blk, n, D.BF16, cb), S.f32_to_bf16(ref))


def test_dequant_worked_blocks(orc):
    """The hand-derived worked blocks go through the GPU too."""
    cb = P._worked_codebook()
    for row in P._rows("cb2_worked.txt"):
        o, idx, sgn = int(row[0]), int(row[1]), int(row[2], 16)
        blk = np.zeros(70, dtype=np.uint8)
        blk[:32] = 2
        blk[o], blk[32 + o] = idx, sgn
        blk[64:68] = [int(v, 16) for v in row[3:7]]
        d = int(row[7], 16)
        blk[68:70] = [d & 0xFF, d >> 8]
        got = _run(D.cb2_dequant, blk, 1, D.F32, cb)
        assert got[8 * o:8 * o + 8].tolist() == [float(v) for v in row[8:16]]
    for s, sb, fill, dbits, mbits, val in P._rows("q2k_scale_min.txt"):
        blk = np.zeros(84, dtype=np.uint8)
        blk[16:80] = int(fill, 16)
        blk[int(s)] = int(sb, 16)
        d, m = int(dbits, 16), int(mbits, 16)
        blk[80:84] = [d & 0xFF, d >> 8, m & 0xFF, m >> 8]
        got = _run(D.q2k_dequant, blk, 1, D.F32)
        exp = np.zeros(256, dtype=np.float32)
        exp[16 * int(s):16 * int(s) + 16] = float(val)
        assert np.array_equal(got, exp)


# ---------------------------------------------------------------------------
# Q4_K / Q5_K / Q6_K (the routed higher-bit formats)
# ---------------------------------------------------------------------------

KQ = {  # format: (block bytes, fp16 field offsets, library entry, oracle method)
    S.FMT_Q4K: (144, (0, 2), D.q4k_dequant, "q4k_dequant"),
    S.FMT_Q5K: (176, (0, 2), D.q5k_dequant, "q5k_dequant"),
    S.FMT_Q6K: (210, (208,), D.q6k_dequant, "q6k_dequant"),
    S.FMT_MXFP4: (136, (), D.mxfp4_dequant, "mxfp4_dequant"),
}


def _random_kquant(fmt, n, seed):
    bb, offs, _, _ = KQ[fmt]
    rng = np.random.default_rng(seed)
    blk = rng.integers(0, 256, size=(n, bb), dtype=np.uint8)
    for off in offs:
        h = rng.integers(0, 0x7C00, size=n).astype(np.uint16)
        h |= rng.integers(0, 2, size=n).astype(np.uint16) << 15
        blk[:, off:off + 2] = h.view(np.uint8).reshape(n, 2)
    if fmt == S.FMT_MXFP4:                       # scale bytes below 255 (255 is NaN)
        blk[:, 0::17] = rng.integers(0, 255, size=(n, 8), dtype=np.uint8)
    return blk


@pytest.mark.parametrize("fmt", [S.FMT_Q4K, S.FMT_Q5K, S.FMT_Q6K, S.FMT_MXFP4],
                         ids=["q4k", "q5k", "q6k", "mxfp4"])
@pytest.mark.parametrize("n", [1, 3, 37, 4096 + 5, 200_000])
def test_kquant_dequant_bit_exact(orc, fmt, n):
    _, _, fn, ref_name = KQ[fmt]
    blk = _random_kquant(fmt, n, 1000 * fmt + n)
    ref = getattr(orc, ref_name)(blk)
    got = _run(fn, blk, n, D.F32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(_run(fn, blk, n, D.F16), _rne_f16(ref))
    assert np.array_equal(_run(fn, blk, n, D.BF16), S.f32_to_bf16(ref))


@pytest.mark.parametrize("fmt", [S.FMT_Q4K, S.FMT_Q5K, S.FMT_Q6K, S.FMT_MXFP4],
                         ids=["q4k", "q5k", "q6k", "mxfp4"])
def test_kquant_dequant_generated_rows(orc, fmt):
    bb, _, fn, ref_name = KQ[fmt]
    W = S.make_experts(9, S.TENSOR_DOWN, 2, 64, 2048, fmt, 8 * bb)
    ref = getattr(orc, ref_name)(W)
    got = _run(fn, W, W.size // bb, D.F32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


class _GpuDecoders:
    """The library's K-quant kernels behind the oracle's method names, so
    the hand-derived worked and one-hot pins run against the GPU as well."""

    def q4k_dequant(self, blk):
        return _run(D.q4k_dequant, blk, blk.size // 144, D.F32)

    def q5k_dequant(self, blk):
        return _run(D.q5k_dequant, blk, blk.size // 176, D.F32)

    def q6k_dequant(self, blk):
        return _run(D.q6k_dequant, blk, blk.size // 210, D.F32)

    def mxfp4_dequant(self, blk):
        return _run(D.mxfp4_dequant, blk, blk.size // 136, D.F32)


@pytest.mark.parametrize("pin", [P.pin_q4k_worked, P.pin_q5k_worked, P.pin_q6k_worked,
                                 P.pin_kquant_onehot, P.pin_mxfp4_worked],
                         ids=lambda p: p.__name__)
def test_kquant_worked_blocks(pin):
    pin(_GpuDecoders())
