"""ds4g_moe_forward_noalloc: the layer for callers that cannot allocate device
memory (a plugin whose host runtime owns every allocation, or a serving loop
that must not call cudaMalloc once running).  Its scratch is a static device
array inside the library.  Checked against the workspace entry point,
ds4g_moe_forward, on two calls in a row (the second call reuses the array
the first one left behind): both run the same deterministic kernels, so the
outputs must be bit-identical, which also shows that nothing a call leaves
in the array leaks into the next one.  One case is forced onto the
tensor-core kernels, one is the codebook format.  Collected last so that a
stop-at-first-failure run has already run every other test."""
import numpy as np
import pytest
import torch

import bit_quantized_routed_route_b300 as D
import ds4g_synth as S
import oracle_pins as P
from gpu_helpers import cached_layer, check_output, run_forward, to_device

pytestmark = pytest.mark.gpu


def _dev_inputs(layer):
    dev = torch.device("cuda")
    x = torch.from_numpy(np.ascontiguousarray(layer["x"]).view(np.int16)).to(dev)
    lg = torch.from_numpy(np.ascontiguousarray(layer["logits"])).to(dev)
    return x, lg


def _small(which):
    if which == "small":
        return P.small_layer(seed=77, H=1024, I=320, E=12, k=3, T=5), 0
    if which == "small_tc":            # segments over one 128-token tile
        return P.small_layer(seed=78, H=1024, I=256, E=4, k=2, T=200, align=16), D.FORCE_TC
    if which == "small_codebook":
        return P.small_layer(seed=79, H=512, I=256, E=5, k=2, T=40, fmt=S.FMT_CB2, align=16,
                             score=S.SCORE_SIGMOID), 0
    return cached_layer(which), 0


@pytest.mark.parametrize("which", ["decode_1tok", "small", "small_tc", "small_codebook"])
def test_noalloc_matches_workspace_entry_point_twice(which):
    layer, flags = _small(which)
    L = to_device(layer, flags=flags)
    y_ws, _ = run_forward(L, layer["x"], layer["logits"])      # ds4g_moe_forward
    x, lg = _dev_inputs(layer)
    T, H = layer["x"].shape
    assert L.workspace_bytes(T) <= D.NOALLOC_SCRATCH_BYTES
    for _ in range(2):
        y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        D.check(D.moe_forward_noalloc(L.desc, x, lg, T, y))
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        check_output(got, y_ws.astype(np.float64))
        assert np.array_equal(got.view(np.uint32), y_ws.view(np.uint32)), \
            "no-alloc output differs from the workspace entry point's"


def test_noalloc_rejects_plans_beyond_the_static_scratch():
    layer = cached_layer("decode_1tok")
    L = to_device(layer)
    T = 2048                                   # a prefill-sized call
    assert L.workspace_bytes(T) > D.NOALLOC_SCRATCH_BYTES
    H, E = layer["hidden"], layer["n_experts"]
    x = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    lg = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    y = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    assert D.moe_forward_noalloc(L.desc, x, lg, T, y) == D.ERR_WORKSPACE


def test_noalloc_status_reports_a_timeout_then_ok():
    """ds4g_moe_noalloc_status reads the static scratch's status word: a
    call whose producers issue nothing (DS4G_DEBUG_STALL, 2 ms waits) reads
    DS4G_ERR_TIMEOUT; the next normal call reads DS4G_OK and is exact."""
    layer, _ = _small("small")
    L = to_device(layer)
    y_ws, _ = run_forward(L, layer["x"], layer["logits"])
    x, lg = _dev_inputs(layer)
    T, H = layer["x"].shape
    stalled = L.with_flags(D.DEBUG_STALL)
    y = torch.empty((T, H), dtype=torch.float32, device="cuda")
    D.check(D.moe_forward_noalloc(stalled.desc, x, lg, T, y))
    st, v = D.moe_noalloc_status(stalled.desc, T)
    assert st == D.OK and v == D.ERR_TIMEOUT
    D.check(D.moe_forward_noalloc(L.desc, x, lg, T, y))
    st, v = D.moe_noalloc_status(L.desc, T)
    assert st == D.OK and v == D.OK
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_ws.view(np.uint32))
