"""Failure detection on the device without a fault: with the DS4G_DEBUG_STALL
test hook the decode kernels' copy producers issue nothing, the consumers'
bounded waits (2 ms) expire, the kernels return early and the workspace
status word reads DS4G_ERR_TIMEOUT.  The context stays usable: the next
normal call on the same workspace succeeds and is correct."""
import numpy as np
import pytest
import torch

import bit_quantized_routed_route_b300 as D
import oracle_pins as P
from gpu_helpers import check_output, to_device

pytestmark = pytest.mark.gpu


def test_bounded_wait_expires_and_reports_timeout(orc):
    layer = P.small_layer(seed=31, H=1024, I=512, E=8, k=2, T=3)
    T, H = layer["x"].shape
    dev = torch.device("cuda")
    x = torch.from_numpy(layer["x"].view(np.int16)).to(dev)
    lg = torch.from_numpy(layer["logits"]).to(dev)
    y = torch.zeros((T, H), dtype=torch.float32, device=dev)
    L = to_device(layer)
    ws_bytes = L.workspace_bytes(T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    stalled = L.with_flags(D.DEBUG_STALL)
    D.check(D.moe_forward(stalled.desc, x, lg, T, y, ws, ws_bytes))
    st, dev_status = D.moe_device_status(stalled.desc, T, ws, ws_bytes)
    assert st == D.OK and dev_status == D.ERR_TIMEOUT

    D.check(D.moe_forward(L.desc, x, lg, T, y, ws, ws_bytes))
    st, dev_status = D.moe_device_status(L.desc, T, ws, ws_bytes)
    assert st == D.OK and dev_status == D.OK
    torch.cuda.synchronize()
    yref, _, _ = orc.moe_forward(layer, layer["x"], layer["logits"])
    check_output(y.cpu().numpy(), yref)
