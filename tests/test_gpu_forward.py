"""ds4g_moe_forward against the oracle on the synthetic workloads and on small
edge-case layers: routing bit-exact, per-token relative L2 <= 1e-3 and
max-abs <= 5e-3 * max|ref| on the output.

Full-size workloads run at their full token counts (the launch configuration
the benchmark times).  The oracle checks every token of the decode-sized
workloads (up to 32 tokens, the K-quant and MXFP4 layers among them); for
prefill_2048, codebook_512, mixed_2048 and mxfp4_2048 it checks at least 64
tokens
chosen to reach every code path (first and last token of the heaviest
segments, both sides of each 128-token tile boundary in them, tokens routed
to one-token segments, then seeded random ones).  Its result for a token does
not depend on the other tokens."""
import numpy as np
import pytest
import torch

import bit_quantized_routed_route_b300 as D
import ds4g_synth as S
import oracle_pins as P
from gpu_helpers import (boundary_tokens, cached_layer, check_output, check_routing,
                         oracle_tokens, run_forward, to_device)

pytestmark = pytest.mark.gpu

SAMPLE = {"tiny": None, "decode_1tok": None, "decode_32tok": None, "prefill_2048": 64,
          "codebook_512": 64, "mixed_2048": 64, "kquant_32tok": None, "mxfp4_32tok": None,
          "mxfp4_2048": 64}


@pytest.mark.parametrize("name", list(S.CONFIGS))
def test_forward_workloads(orc, name):
    layer = cached_layer(name)
    L = to_device(layer)
    y, routing = run_forward(L, layer["x"], layer["logits"])
    k, score = layer["top_k"], layer["score"]
    rref = orc.route(layer["logits"], k, score)
    check_routing(routing, rref)
    T = layer["tokens"]
    tok = None if SAMPLE[name] is None else boundary_tokens(rref, k, T, SAMPLE[name], 1234)
    yref = oracle_tokens(orc, layer, layer["x"], layer["logits"], tok)
    yy = y if tok is None else y[tok]
    check_output(yy, yref)
    if tok is not None:
        assert len(tok) >= 64


@pytest.mark.parametrize("kw", [
    dict(H=256, I=128, E=8, k=2, T=4),                     # tiny shape, I < 256
    dict(H=512, I=320, E=6, k=3, T=5),                     # ragged I (padded down K)
    dict(H=768, I=256, E=33, k=5, T=70),                   # E not a multiple of 32; T > 64
    dict(H=256, I=256, E=1, k=1, T=3),                     # one expert
    dict(H=512, I=512, E=4, k=4, T=40),                    # k = E, every expert busy
    dict(H=1024, I=384, E=16, k=2, T=1, score=S.SCORE_SIGMOID, logits_kind=S.LOGITS_UNIFORM),
    dict(H=512, I=256, E=5, k=2, T=9, fmt=S.FMT_CB2, align=16),
    dict(H=512, I=200, E=7, k=3, T=17, fmt=S.FMT_CB2, align=2),
    # the routed higher-bit formats (general kernels)
    dict(H=512, I=320, E=5, k=2, T=9, fmt=S.FMT_Q4K, down_fmt=S.FMT_Q6K),
    dict(H=768, I=256, E=6, k=3, T=40, fmt=S.FMT_Q5K),
    dict(H=512, I=200, E=4, k=2, T=3, fmt=S.FMT_Q2K, down_fmt=S.FMT_Q5K),
    dict(H=256, I=512, E=3, k=3, T=2, fmt=S.FMT_Q4K, score=S.SCORE_SIGMOID,
         logits_kind=S.LOGITS_UNIFORM),
    dict(H=512, I=320, E=5, k=2, T=9, fmt=S.FMT_MXFP4),
    dict(H=768, I=256, E=4, k=2, T=6, fmt=S.FMT_MXFP4, down_fmt=S.FMT_Q6K),
])
def test_forward_edge_layers(orc, kw):
    layer = P.small_layer(seed=sum(kw.get(x, 0) for x in ("H", "I", "E", "T")), **kw)
    L = to_device(layer)
    y, routing = run_forward(L, layer["x"], layer["logits"])
    check_routing(routing, orc.route(layer["logits"], layer["top_k"], layer["score"]))
    yref, _, _ = orc.moe_forward(layer, layer["x"], layer["logits"])
    check_output(y, yref)


def test_forward_zero_scale_expert_gives_exact_zero(orc):
    layer = P.small_layer(seed=21, E=4, k=1, T=6)
    layer["w_down"][:, :, :] = 0
    y, _ = run_forward(to_device(layer), layer["x"], layer["logits"])
    assert np.all(y == 0.0)


def test_forward_is_deterministic():
    layer = cached_layer("tiny")
    L = to_device(layer)
    y1, _ = run_forward(L, layer["x"], layer["logits"])
    y2, _ = run_forward(L, layer["x"], layer["logits"])
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_host_entry_point_matches_device_entry_point():
    layer = cached_layer("decode_1tok")
    L = to_device(layer)
    y_dev, _ = run_forward(L, layer["x"], layer["logits"])
    T, H = layer["x"].shape
    x_h = torch.from_numpy(layer["x"].view(np.int16)).pin_memory()
    l_h = torch.from_numpy(layer["logits"]).pin_memory()
    y_h = torch.empty((T, H), dtype=torch.float32).pin_memory()
    ws_bytes = L.workspace_bytes(T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    D.check(D.moe_forward_host(L.desc, x_h, l_h, T, y_h, ws, ws_bytes))
    assert np.array_equal(y_h.numpy().view(np.uint32), y_dev.view(np.uint32))


def test_forced_tensor_core_refuses_unaligned_kquant_rows():
    """The tensor-core kernels stage whole 16-byte windows: forcing them on a
    layer whose Q6_K W_down rows (two 210-byte blocks) are not a multiple of
    16 bytes returns DS4G_ERR_LAYOUT without touching y."""
    layer = P.small_layer(seed=5, H=512, I=256, E=4, k=2, T=40, fmt=S.FMT_Q4K,
                          down_fmt=S.FMT_Q6K)
    L = to_device(layer, flags=D.FORCE_TC)
    dev = torch.device("cuda")
    T, H = layer["x"].shape
    x = torch.from_numpy(layer["x"].view(np.int16)).to(dev)
    lg = torch.from_numpy(layer["logits"]).to(dev)
    y = torch.full((T, H), 7.0, dtype=torch.float32, device=dev)
    ws = torch.empty(L.workspace_bytes(T), dtype=torch.uint8, device=dev)
    assert D.moe_forward(L.desc, x, lg, T, y, ws) == D.ERR_LAYOUT
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
