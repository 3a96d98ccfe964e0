"""ds4g_moe_forward_noalloc: the layer for callers that cannot allocate device
memory (a plugin whose host runtime owns every allocation, or a serving loop
that must not call cudaMalloc once running).  Its scratch is a static device
array inside the library.  Checked against the workspace entry point,
ds4g_moe_forward, with the layer tolerance, on two calls in a row (the second
call reuses the array the first one left behind).  Collected last so that a
stop-at-first-failure run has already run every other test."""
import numpy as np
import pytest
import torch

import bit_quantized_routed_route_b300 as D
import oracle_pins as P
from gpu_helpers import cached_layer, check_output, run_forward, to_device

pytestmark = pytest.mark.gpu


def _dev_inputs(layer):
    dev = torch.device("cuda")
    x = torch.from_numpy(np.ascontiguousarray(layer["x"]).view(np.int16)).to(dev)
    lg = torch.from_numpy(np.ascontiguousarray(layer["logits"])).to(dev)
    return x, lg


@pytest.mark.parametrize("which", ["decode_1tok", "small"])
def test_noalloc_matches_workspace_entry_point_twice(which):
    layer = cached_layer(which) if which != "small" else P.small_layer(
        seed=77, H=1024, I=320, E=12, k=3, T=5)
    L = to_device(layer)
    y_ws, _ = run_forward(L, layer["x"], layer["logits"])      # ds4g_moe_forward
    x, lg = _dev_inputs(layer)
    T, H = layer["x"].shape
    for _ in range(2):
        y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        D.check(D.moe_forward_noalloc(L.desc, x, lg, T, y))
        torch.cuda.synchronize()
        check_output(y.cpu().numpy(), y_ws.astype(np.float64))


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
