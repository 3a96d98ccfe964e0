"""Number-format facts that the tensor-core kernels' exactness claims rest
on, checked on the CPU with numpy's IEEE fp16 (no kernel or oracle code):

* MXFP4 (ds4 README mirror, "Model Weights": the ds4f-mxfp4 routed experts,
  read as OCP microscaling FP4): every E2M1 value times the block scale
  2^s is exact in fp16 for s in [-23, 13], and not for s = -24 or 14, which
  is the range outside which the kernels report DS4G_ERR_RANGE;
* Q4_K / Q5_K (same page, the routed K-quant formats): the integer q * sc
  (q < 32, sc < 64) and the constants -1024 * sc and -64 * sc used to form
  it are exact fp16 values, so n = v * S + C is exact;
* Q6_K: (q - 32) * sc reaches past fp16's exact integers, which is why its
  weights take the form fp16((q - 32) * fp16(d * sc)) with two roundings."""
import numpy as np

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def exact_in_fp16(v):
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):          # values past 65504 become inf: not exact
        return np.all(v.astype(np.float16).astype(np.float64) == v)


def test_e2m1_times_power_of_two_is_exact_in_fp16_from_2_pow_m23_to_2_pow_13():
    for s in range(-23, 14):
        vals = np.concatenate([E2M1, -E2M1]) * 2.0 ** s
        assert exact_in_fp16(vals), s
        # the scale itself is an fp16 value too (a subnormal below 2^-14)
        assert exact_in_fp16([2.0 ** s])
    # one step outside: 0.5 * 2^-24 underflows, 4 * 2^14 overflows
    assert not exact_in_fp16(E2M1 * 2.0 ** -24)
    assert not exact_in_fp16(E2M1 * 2.0 ** 14)


def test_e2m1_code_to_value_through_fp16_bits():
    # the low three bits placed at fp16 bits 9..11 give value * 2^-14 for every
    # code, subnormal 0.5 included (the magnitude grid of E2M1)
    for m in range(8):
        bits = np.array([m << 9], dtype=np.uint16)
        assert bits.view(np.float16)[0].astype(np.float64) == E2M1[m] * 2.0 ** -14


def test_k45_integer_products_are_exact_in_fp16():
    q = np.arange(32, dtype=np.float64)[:, None]
    sc = np.arange(64, dtype=np.float64)[None, :]
    assert (q * sc).max() == 1953
    assert exact_in_fp16(q * sc)
    assert exact_in_fp16(-1024.0 * sc) and exact_in_fp16(sc / 16.0) and exact_in_fp16(-64.0 * sc)
    # 1024 + q and 1024 + 16 q (+ 256 for the fifth bit) are exact too
    assert exact_in_fp16(1024.0 + np.arange(32)) and exact_in_fp16(1024.0 + 16.0 * np.arange(16) + 256.0)


def test_q6k_products_exceed_fp16_exact_integers():
    q = np.arange(64, dtype=np.float64)[:, None] - 32.0
    sc = np.arange(-128, 128, dtype=np.float64)[None, :]
    prod = q * sc
    assert np.abs(prod).max() == 4096
    assert not exact_in_fp16(prod)
    # while q - 32 itself, from v = 1024 + q, is exact
    assert exact_in_fp16((1024.0 + np.arange(64)) - 1056.0)


# ---------------------------------------------------------------------------
# Why the MXFP4 layers keep fp16 activations: the block-scaled tensor-core
# MMAs multiply MX-quantized activations (FP8 E4M3 or FP4 E2M1 elements, one
# power-of-two scale per 32 along K, scale exponent floor(log2 amax) minus
# the element format's largest exponent, per the OCP microscaling layout).
# Quantizing x that way alone, with everything else computed by the oracle,
# already costs far more than the 1e-3 per-token tolerance.
# ---------------------------------------------------------------------------

def _round_to_grid(v, mant_bits, emin, vmax):
    """Round-to-nearest-even onto a minifloat grid with `mant_bits` mantissa
    bits, smallest normal exponent `emin` (subnormals below) and largest
    finite value `vmax` (saturating)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    quantum = 2.0 ** (e - mant_bits)
    q = np.round(a / quantum) * quantum
    return np.sign(v) * np.minimum(q, vmax)


def _mx_quantize(x, mant_bits, emin, emax, vmax):
    """x [T x H] -> MX values: per 32 consecutive elements along H a scale
    2^(floor(log2 amax) - emax), elements rounded onto the element grid."""
    T, H = x.shape
    b = x.reshape(T, H // 32, 32)
    amax = np.abs(b).max(axis=2, keepdims=True)
    sexp = np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - emax
    scale = 2.0 ** sexp
    return (_round_to_grid(b / scale, mant_bits, emin, vmax) * scale).reshape(T, H)


def _per_token_rel_l2(y, ref):
    return np.linalg.norm(y - ref, axis=1) / np.linalg.norm(ref, axis=1)


def test_mx_quantized_activations_break_the_tolerance(orc):
    import ds4g_synth as S
    import oracle_pins as P
    layer = P.small_layer(seed=91, H=1024, I=512, E=8, k=2, T=16, fmt=S.FMT_MXFP4,
                          score=S.SCORE_SIGMOID)
    x = S.bf16_to_f32(layer["x"]).astype(np.float64)
    yref, _, _ = orc.moe_forward(layer, layer["x"], layer["logits"])
    errs = {}
    for name, (mant, emin, emax, vmax) in {"e4m3": (3, -6, 8, 448.0),
                                           "e2m1": (1, 0, 2, 6.0)}.items():
        xq = _mx_quantize(x, mant, emin, emax, vmax)
        # every MX value (at most 4 significant bits) is exact in bf16
        xb = S.f32_to_bf16(xq.astype(np.float32))
        assert np.array_equal(S.bf16_to_f32(xb).astype(np.float64), xq)
        y, _, _ = orc.moe_forward(layer, xb, layer["logits"])
        errs[name] = _per_token_rel_l2(y, yref).max()
    assert errs["e4m3"] > 5e-3, errs            # FP8 activations: several times the 1e-3 bar
    assert errs["e2m1"] > 5e-2, errs            # FP4 activations: far beyond it


def test_fp8_activation_terms_needed_for_the_tolerance(orc):
    """Splitting x into MX-FP8 terms, each quantizing the previous residual:
    two terms still leave more than 1e-3, three reproduce the bf16
    activations exactly (8 significant bits within three 4-bit terms), so a
    native FP8-activation MMA would need three MMAs per K step."""
    import ds4g_synth as S
    import oracle_pins as P
    layer = P.small_layer(seed=91, H=1024, I=512, E=8, k=2, T=16, fmt=S.FMT_MXFP4,
                          score=S.SCORE_SIGMOID)
    x = S.bf16_to_f32(layer["x"]).astype(np.float64)
    yref, _, _ = orc.moe_forward(layer, layer["x"], layer["logits"])
    q = lambda v: _mx_quantize(v, 3, -6, 8, 448.0)
    t1 = q(x)
    t2 = q(x - t1)
    t3 = q(x - t1 - t2)
    errs = []
    for xs in (t1 + t2, t1 + t2 + t3):
        y, _, _ = orc.moe_forward(layer, S.f32_to_bf16(xs.astype(np.float32)), layer["logits"])
        errs.append(_per_token_rel_l2(y, yref).max())
    assert errs[0] > 1e-3, errs
    assert np.array_equal(t1 + t2 + t3, x) and errs[1] == 0.0, errs
