"""The decode kernels (small expert segments, Q2_K) against the oracle over
token counts 1..32 (ragged segment chunks), padded inter sizes, expert counts
below and above a warp, and several layer widths."""
import numpy as np
import pytest
import torch

import bit_quantized_routed_route_b300 as D
import ds4g_synth as S
import oracle_pins as P
from gpu_helpers import cached_layer, check_output, check_routing, run_forward, to_device

pytestmark = pytest.mark.gpu

CASES = [
    dict(H=256, I=128, E=8, k=2, T=1),
    dict(H=512, I=320, E=6, k=3, T=2),
    dict(H=768, I=512, E=16, k=4, T=3),
    dict(H=1024, I=256, E=5, k=5, T=5),         # every expert busy, segments of 5
    dict(H=512, I=768, E=64, k=6, T=8),
    dict(H=512, I=256, E=3, k=2, T=9),          # segments longer than one token chunk
    dict(H=2048, I=512, E=33, k=8, T=17),
    dict(H=1024, I=1024, E=256, k=8, T=32),
    dict(H=4096, I=1536, E=64, k=6, T=1),       # the single-token decode shape
    dict(H=512, I=512, E=2, k=2, T=32, score=S.SCORE_SIGMOID, logits_kind=S.LOGITS_UNIFORM),
]


@pytest.mark.parametrize("kw", CASES, ids=lambda kw: "H{H}_I{I}_E{E}_k{k}_T{T}".format(**kw))
def test_decode_path(orc, kw):
    layer = P.small_layer(seed=kw["H"] + kw["I"] + kw["T"], **kw)
    L = to_device(layer, flags=D.FORCE_GEMV)                   # decode kernels at every T
    assert D.moe_forward_launches(L.desc, kw["T"]) == 2        # reset/convert, fused decode kernel
    y, routing = run_forward(L, layer["x"], layer["logits"])
    check_routing(routing, orc.route(layer["logits"], layer["top_k"], layer["score"]))
    yref, _, _ = orc.moe_forward(layer, layer["x"], layer["logits"])
    check_output(y, yref)


@pytest.mark.parametrize("T", [1, 2, 5, 8, 12, 32])
def test_decode_full_width_layer(orc, T):
    """The 7168/2048/256/top-8 layer on the decode kernels (the first T tokens
    of the 32-token workload; from 4 tokens on the call would take the
    tensor-core kernels unless forced): 2352-byte gate/up rows copied whole,
    672-byte W_down rows padded to 688 bytes in shared memory, and down
    stages that fit two experts' tiles and h rows plus a third tile without
    its h rows (the one-vector kernel must start a new stage there, as it
    reads h from shared memory only); 12 and 32 tokens on the tcgen05 decode
    kernel."""
    layer = cached_layer("decode_32tok")
    x, lg = layer["x"][:T], layer["logits"][:T]
    L = to_device(layer, flags=D.FORCE_GEMV)
    assert D.moe_forward_launches(L.desc, T) == 2
    y, routing, st = run_forward(L, x, lg, with_status=True)
    assert st == D.OK
    check_routing(routing, orc.route(lg, layer["top_k"], layer["score"]))
    yref, _, _ = orc.moe_forward(layer, x, lg)
    check_output(y, yref)


def test_decode_is_deterministic():
    layer = P.small_layer(seed=5, H=1024, I=512, E=16, k=4, T=7)
    L = to_device(layer, flags=D.FORCE_GEMV)
    y1, _ = run_forward(L, layer["x"], layer["logits"])
    y2, _ = run_forward(L, layer["x"], layer["logits"])
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_decode_matches_tensor_core_path_closely(orc):
    """The tcgen05 path (forced) and the mma.sync decode path agree with each
    other to the same tolerance."""
    layer = P.small_layer(seed=9, H=2048, I=768, E=12, k=3, T=4, align=16)
    y_dec, _ = run_forward(to_device(layer), layer["x"], layer["logits"])
    y_gen, _ = run_forward(to_device(layer, flags=D.FORCE_TC), layer["x"], layer["logits"])
    check_output(y_dec, y_gen.astype(np.float64))
