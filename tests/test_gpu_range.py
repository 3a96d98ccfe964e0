"""Activations outside the comfortable fp16 range, on every device path.

The tensor-core and decode kernels multiply in fp16, whose full-precision
range (6.1e-5 .. 65504) is narrower than the bf16 activations'.  Each token
therefore enters scaled by a power of two chosen from its largest |x|, and h =
SiLU(g)*u leaves gate/up scaled by the square of that factor (times a fixed
2^-14), both undone exactly in fp32.  These tests feed tokens far from unit
scale and check the layer against the fp64 oracle with the usual tolerances:

  * x ~ N(0, 300^2) (h reaches ~1e5, beyond fp16);
  * one token whose largest |x| is near 6e4 (x itself at the edge of fp16);
  * one token ~N(0, 1e-4^2) (most of it subnormal in fp16 without scaling);
  * one all-zero token (its output must be exactly zero).
"""
import numpy as np
import pytest

import bit_quantized_routed_route_b300 as D
import ds4g_synth as S
import oracle_pins as P
from gpu_helpers import check_output, check_routing, oracle_tokens, run_forward, to_device

pytestmark = pytest.mark.gpu


def ranged_x(T: int, H: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H)).astype(np.float64) * 300.0
    x[1] = rng.standard_normal(H) * 1.2e4          # max |x| ~ 5e4 .. 6e4
    x[1] *= 6.0e4 / np.abs(x[1]).max()
    x[2] = rng.standard_normal(H) * 1e-4
    x[3] = 0.0
    return S.f32_to_bf16(x.astype(np.float32))


@pytest.mark.parametrize("kw,flags", [
    (dict(H=1024, I=512, E=8, k=2, T=5), 0),                               # mma.sync decode
    (dict(H=4096, I=512, E=8, k=2, T=7), 0),                               # same, x converted ahead
    (dict(H=1024, I=512, E=8, k=2, T=12), 0),                              # tcgen05 decode
    (dict(H=1024, I=512, E=8, k=2, T=40, align=16), D.FORCE_TC),           # tensor-core kernels
    (dict(H=512, I=256, E=5, k=2, T=9, fmt=S.FMT_CB2, align=16), 0),       # codebook, tensor core
    (dict(H=512, I=200, E=7, k=3, T=17, fmt=S.FMT_CB2, align=2), 0),       # general kernels
    (dict(H=1024, I=512, E=8, k=2, T=12, fmt=S.FMT_Q5K, down_fmt=S.FMT_Q4K), 0),   # K-quant, tensor core
    (dict(H=1024, I=512, E=8, k=2, T=12, fmt=S.FMT_MXFP4), 0),            # MXFP4, tensor core
], ids=["decode_mma_sync", "decode_mma_sync_xp", "decode_tcgen05", "tensor_core", "codebook_tc", "general",
        "kquant_tc", "mxfp4_tc"])
def test_large_and_small_activations(orc, kw, flags):
    layer = P.small_layer(seed=41 + kw["T"], **kw)
    T, H = layer["x"].shape
    layer["x"] = ranged_x(T, H, seed=7 + T)
    L = to_device(layer, flags=flags)
    y, routing = run_forward(L, layer["x"], layer["logits"])
    check_routing(routing, orc.route(layer["logits"], layer["top_k"], layer["score"]))
    yref = oracle_tokens(orc, layer, layer["x"], layer["logits"])
    assert np.abs(yref[0]).max() > 1e3                  # the big tokens really are big
    assert np.all(y[3] == 0.0) and np.all(yref[3] == 0.0)
    check_output(y, yref)
    # the small token is checked on its own scale too (max-abs is global)
    err = np.linalg.norm(y[2] - yref[2]) / np.linalg.norm(yref[2])
    assert err <= 1e-3, f"tiny-magnitude token: relative L2 {err:.3e}"
