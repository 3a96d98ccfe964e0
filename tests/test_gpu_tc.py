"""The tensor-core (tcgen05) path of ds4g_moe_forward against the oracle:
routing bit-exact, per-token relative L2 <= 1e-3 and max-abs <= 5e-3 *
max|ref| on the output.

The path runs by itself for layers whose rows are multiples of 16 bytes (every
format; Q2_K from 4 tokens on); DS4G_FORCE_TC sends the others to it.
Cases span several 128-row weight tiles and several 128-token tiles, with
ragged tails on both (inter not a multiple of 128, segments longer than one
token tile), a single expert, k = E, and the full-size decode layer."""
import numpy as np
import pytest

import bit_quantized_routed_route_b300 as D
import ds4g_synth as S
import oracle_pins as P
from gpu_helpers import cached_layer, check_output, check_routing, run_forward, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kw", [
    dict(H=256, I=128, E=8, k=2, T=4),                     # one tile of each; I < 256
    dict(H=512, I=320, E=6, k=3, T=40),                    # ragged inter (rows >= inter read as zero)
    dict(H=1024, I=256, E=5, k=2, T=200),                  # segments of > 128 tokens
    dict(H=1024, I=512, E=1, k=1, T=300),                  # one expert, three token tiles
    dict(H=2048, I=384, E=33, k=5, T=70),                  # E not a multiple of 32
    dict(H=768, I=1024, E=4, k=4, T=33),                   # k = E, every expert busy
])
def test_tc_forward_small_layers(orc, kw):
    layer = P.small_layer(seed=1000 + kw["H"] + kw["T"], align=16, **kw)
    L = to_device(layer, flags=D.FORCE_TC)
    y, routing = run_forward(L, layer["x"], layer["logits"])
    check_routing(routing, orc.route(layer["logits"], layer["top_k"], layer["score"]))
    yref, _, _ = orc.moe_forward(layer, layer["x"], layer["logits"])
    check_output(y, yref)


@pytest.mark.parametrize("kw", [
    dict(H=256, I=128, E=8, k=2, T=12),                    # one block per row; I < 256
    dict(H=512, I=256, E=5, k=2, T=40),                    # 70-byte blocks at every 2-byte offset
    dict(H=1024, I=384, E=7, k=3, T=150),                  # ragged inter; segments over 128 tokens
    dict(H=2048, I=512, E=33, k=5, T=70),
])
def test_tc_forward_codebook_layers(orc, kw):
    """The codebook-2-bit format on the tensor-core kernels (rows padded to
    16 bytes)."""
    layer = P.small_layer(seed=2000 + kw["H"] + kw["T"], fmt=S.FMT_CB2, align=16,
                          score=S.SCORE_SIGMOID, **kw)
    L = to_device(layer, flags=D.FORCE_TC)
    y, routing = run_forward(L, layer["x"], layer["logits"])
    check_routing(routing, orc.route(layer["logits"], layer["top_k"], layer["score"]))
    yref, _, _ = orc.moe_forward(layer, layer["x"], layer["logits"])
    check_output(y, yref)


def test_tc_forward_decode_layer_forced(orc):
    """The 7168/2048/256/top-8 layer at 32 tokens, forced onto the
    tensor-core kernels, on a sample of tokens."""
    layer = cached_layer("decode_32tok")
    L = to_device(layer, flags=D.FORCE_TC)
    y, routing = run_forward(L, layer["x"], layer["logits"])
    check_routing(routing, orc.route(layer["logits"], layer["top_k"], layer["score"]))
    tok = np.array([0, 13, 31], dtype=np.int32)
    yref, _, _ = orc.moe_forward(layer, layer["x"], layer["logits"], tok)
    check_output(y[tok], yref)


def test_tc_matches_general_path():
    """Both device paths on the same layer agree within the output tolerance."""
    layer = P.small_layer(seed=5, H=1024, I=512, E=7, k=3, T=150, align=16)
    L = to_device(layer, flags=D.FORCE_TC)
    y_tc, _ = run_forward(L, layer["x"], layer["logits"])
    y_gv, _ = run_forward(L.with_flags(D.FORCE_GEMV), layer["x"], layer["logits"])
    check_output(y_tc, y_gv.astype(np.float64))


def test_tc_is_deterministic():
    layer = P.small_layer(seed=9, H=1024, I=256, E=4, k=2, T=130, align=16)
    L = to_device(layer, flags=D.FORCE_TC)
    y1, _ = run_forward(L, layer["x"], layer["logits"])
    y2, _ = run_forward(L, layer["x"], layer["logits"])
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_tc_forced_on_unaligned_rows_is_rejected():
    layer = P.small_layer(seed=3, H=512, I=256, E=4, k=2, T=8)      # 168-byte rows
    L = to_device(layer, flags=D.FORCE_TC)
    assert L.workspace_bytes(8) == 0
    with pytest.raises(D.DS4GError):
        run_forward(L, layer["x"], layer["logits"])


@pytest.mark.parametrize("kw", [
    dict(H=1024, I=512, E=6, k=2, T=70, fmt=S.FMT_CB2, down_fmt=S.FMT_Q2K, align=16),
    dict(H=512, I=320, E=5, k=3, T=150, fmt=S.FMT_CB2, down_fmt=S.FMT_Q2K, align=16),
    dict(H=1024, I=512, E=4, k=2, T=40, fmt=S.FMT_Q2K, down_fmt=S.FMT_CB2, align=16),
    dict(H=512, I=200, E=5, k=2, T=20, fmt=S.FMT_CB2, down_fmt=S.FMT_Q2K, align=2),   # general
], ids=["cb2_q2k", "cb2_q2k_ragged_I", "q2k_cb2", "cb2_q2k_general"])
def test_mixed_format_layers(orc, kw):
    """W_gate / W_up in one format and W_down in the other (the shipping mix
    is codebook gate/up with Q2_K down): the tensor-core kernels run each
    matrix through its own dequantizer, h in the order the down kernel's
    format needs; 2-byte aligned rows take the general kernels."""
    layer = P.small_layer(seed=3000 + kw["H"] + kw["T"], score=S.SCORE_SIGMOID, **kw)
    L = to_device(layer)
    y, routing = run_forward(L, layer["x"], layer["logits"])
    check_routing(routing, orc.route(layer["logits"], layer["top_k"], layer["score"]))
    yref, _, _ = orc.moe_forward(layer, layer["x"], layer["logits"])
    check_output(y, yref)


@pytest.mark.parametrize("kw", [
    dict(H=512, I=512, E=8, k=2, T=12),                       # units at window offsets 0 and 8
    dict(H=1024, I=320, E=6, k=3, T=150),                     # ragged inter; segments over 128 tokens
    dict(H=2048, I=1024, E=33, k=5, T=70),                    # E not a multiple of 32
    dict(H=1024, I=512, E=1, k=1, T=300),                     # one expert, three token tiles
    dict(H=1024, I=512, E=5, k=2, T=40, down_fmt=S.FMT_Q2K, align=16),   # MXFP4 gate/up, Q2_K down
    dict(H=1024, I=512, E=5, k=2, T=40, down_fmt=S.FMT_CB2, align=16),   # h in natural order
    dict(H=1024, I=512, E=5, k=2, T=40, fmt=S.FMT_CB2, down_fmt=S.FMT_MXFP4, align=16),
], ids=["offsets", "ragged_I", "E33", "one_expert", "mx_q2k", "mx_cb2", "cb2_mx"])
def test_tc_forward_mxfp4_layers(orc, kw):
    """MXFP4 matrices on the tensor-core kernels: each code byte becomes an
    fp16 pair of E2M1 values, times the block's power-of-two scale (exact for
    these weights, so the status word stays clear), alone or mixed with the
    2-bit formats in one layer."""
    kw = dict(dict(fmt=S.FMT_MXFP4), **kw)
    layer = P.small_layer(seed=5000 + kw["H"] + kw["T"], score=S.SCORE_SIGMOID, **kw)
    L = to_device(layer, flags=D.FORCE_TC)
    y, routing, st = run_forward(L, layer["x"], layer["logits"], with_status=True)
    assert st == D.OK
    check_routing(routing, orc.route(layer["logits"], layer["top_k"], layer["score"]))
    yref, _, _ = orc.moe_forward(layer, layer["x"], layer["logits"])
    check_output(y, yref)


@pytest.mark.parametrize("kw", [
    dict(H=512, I=512, E=8, k=2, T=12, fmt=S.FMT_Q4K),
    dict(H=1024, I=320, E=6, k=3, T=150, fmt=S.FMT_Q5K),                  # ragged inter; > 128 tokens
    dict(H=1024, I=1800, E=5, k=2, T=40, fmt=S.FMT_Q4K, down_fmt=S.FMT_Q6K),   # Q6_K at every even offset
    dict(H=2048, I=512, E=33, k=5, T=70, fmt=S.FMT_Q5K, down_fmt=S.FMT_Q4K),
    dict(H=1024, I=512, E=1, k=1, T=300, fmt=S.FMT_Q4K, down_fmt=S.FMT_Q5K),   # one expert, three tiles
    dict(H=1024, I=2048, E=4, k=2, T=24, fmt=S.FMT_Q5K, down_fmt=S.FMT_Q6K),
    dict(H=1024, I=512, E=5, k=2, T=40, fmt=S.FMT_CB2, down_fmt=S.FMT_Q4K, align=16),
    dict(H=1024, I=512, E=5, k=2, T=40, fmt=S.FMT_Q4K, down_fmt=S.FMT_Q2K, align=16),
    dict(H=1024, I=512, E=5, k=2, T=40, fmt=S.FMT_MXFP4, down_fmt=S.FMT_Q5K),
], ids=["q4k", "q5k_ragged_I", "q4k_q6k", "q5k_q4k_E33", "q4k_q5k_one_expert", "q5k_q6k",
        "cb2_q4k", "q4k_q2k", "mx_q5k"])
def test_tc_forward_kquant_layers(orc, kw):
    """The Q4_K / Q5_K super-blocks (gate/up or down) and Q6_K (down) on the
    tensor-core kernels, in natural order (h too), alone or mixed with the
    other formats in one layer."""
    layer = P.small_layer(seed=6000 + kw["H"] + kw["T"], score=S.SCORE_SIGMOID, **kw)
    L = to_device(layer, flags=D.FORCE_TC)
    y, routing, st = run_forward(L, layer["x"], layer["logits"], with_status=True)
    assert st == D.OK
    check_routing(routing, orc.route(layer["logits"], layer["top_k"], layer["score"]))
    yref, _, _ = orc.moe_forward(layer, layer["x"], layer["logits"])
    check_output(y, yref)


def test_tc_mxfp4_scale_outside_fp16_range_is_reported(orc):
    """A block scale of 2^-30 (exact in the fp32 definition; its weights fall
    below fp16's smallest subnormal): the tensor-core kernels round those
    weights and the status word reads DS4G_ERR_RANGE, while the GEMV kernels
    compute the layer in fp32 with the status word clear.  Both stay within
    the tolerance here, the rounded weights being that small."""
    layer = P.small_layer(seed=77, H=512, I=512, E=4, k=2, T=16, fmt=S.FMT_MXFP4,
                          score=S.SCORE_SIGMOID)
    layer["w_up"][:, 0, 17] = 97          # scale byte of block 1, row 0, every expert
    yref, _, _ = orc.moe_forward(layer, layer["x"], layer["logits"])
    L = to_device(layer)
    y_tc, _, st_tc = run_forward(L, layer["x"], layer["logits"], with_status=True)
    assert st_tc == D.ERR_RANGE
    check_output(y_tc, yref)
    y_gv, _, st_gv = run_forward(L.with_flags(D.FORCE_GEMV), layer["x"], layer["logits"],
                                 with_status=True)
    assert st_gv == D.OK
    check_output(y_gv, yref)


@pytest.mark.parametrize("theta,fmt", [(8, S.FMT_Q2K), (8, S.FMT_CB2), (1000, S.FMT_Q2K),
                                        (1, S.FMT_CB2)],
                         ids=["q2k_theta8", "cb2_theta8", "all_light", "all_heavy"])
def test_per_segment_split(orc, theta, fmt):
    """tc_min_tokens = theta: segments of fewer than theta tokens run on the
    GEMV kernels, the others on the tensor-core kernels, in one call.  The
    layer's biased routing gives both kinds (with theta 8); theta 1000 sends
    every segment to the GEMV kernels, theta 1 none."""
    layer = P.small_layer(seed=4000 + theta, H=1024, I=384, E=24, k=4, T=96, fmt=fmt, align=16,
                          score=S.SCORE_SIGMOID, logits_kind=S.LOGITS_BIASED)
    counts = orc.route(layer["logits"], layer["top_k"], layer["score"])["counts"]
    if theta == 8:
        assert (counts >= 8).any() and ((counts > 0) & (counts < 8)).any()
    L = to_device(layer, tc_min_tokens=theta)
    y, routing = run_forward(L, layer["x"], layer["logits"])
    check_routing(routing, orc.route(layer["logits"], layer["top_k"], layer["score"]))
    yref, _, _ = orc.moe_forward(layer, layer["x"], layer["logits"])
    check_output(y, yref)
    # the split result is deterministic too
    y2, _ = run_forward(L, layer["x"], layer["logits"])
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))
