"""Failure detection on the device without a fault: with the DS4G_DEBUG_STALL
test hook the kernels' copy producers issue nothing, the consumers' bounded
waits (2 ms) expire, the kernels return early (the tcgen05 kernels after
freeing their tensor memory) and the workspace status word reads
DS4G_ERR_TIMEOUT.  The context stays usable: the next normal call on the
same workspace succeeds and is correct.  Each kernel family is covered: the
mma.sync decode kernel (3 tokens), the tcgen05 decode kernel (12 tokens) and
the tensor-core prefill kernels (forced)."""
import numpy as np
import pytest
import torch

import bit_quantized_routed_route_b300 as D
import oracle_pins as P
from gpu_helpers import check_output, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,flags", [(3, 0), (12, D.FORCE_GEMV), (3, D.FORCE_TC)],
                         ids=["decode_mma_sync", "decode_tcgen05", "tensor_core"])
def test_bounded_wait_expires_and_reports_timeout(orc, T, flags):
    layer = P.small_layer(seed=31, H=1024, I=512, E=8, k=2, T=T, align=16)
    T, H = layer["x"].shape
    dev = torch.device("cuda")
    x = torch.from_numpy(layer["x"].view(np.int16)).to(dev)
    lg = torch.from_numpy(layer["logits"]).to(dev)
    y = torch.zeros((T, H), dtype=torch.float32, device=dev)
    L = to_device(layer, flags=flags)
    ws_bytes = L.workspace_bytes(T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    stalled = L.with_flags(flags | D.DEBUG_STALL)
    D.check(D.moe_forward(stalled.desc, x, lg, T, y, ws, ws_bytes))
    st, dev_status = D.moe_device_status(stalled.desc, T, ws, ws_bytes)
    assert st == D.OK and dev_status == D.ERR_TIMEOUT

    D.check(D.moe_forward(L.desc, x, lg, T, y, ws, ws_bytes))
    st, dev_status = D.moe_device_status(L.desc, T, ws, ws_bytes)
    assert st == D.OK and dev_status == D.OK
    torch.cuda.synchronize()
    yref, _, _ = orc.moe_forward(layer, layer["x"], layer["logits"])
    check_output(y.cpu().numpy(), yref)
