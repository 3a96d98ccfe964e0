"""Failure detection on the device without a fault: with the DS4G_DEBUG_STALL
test hook the kernels' copy producers issue nothing, the consumers' bounded
waits (2 ms) expire, the kernels return early (the tcgen05 kernels after
freeing their tensor memory) and the workspace status word reads
DS4G_ERR_TIMEOUT.  The context stays usable: the next normal call on the
same workspace succeeds and is correct.  Each kernel family is covered: the
mma.sync decode kernel (3 tokens), the tcgen05 decode kernel (12 tokens), the
tensor-core kernels (forced; and with a codebook W_down, which has its own
down kernel; and in MXFP4)."""
import numpy as np
import pytest
import torch

import bit_quantized_routed_route_b300 as D
import ds4g_synth as S
import oracle_pins as P
from gpu_helpers import check_output, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,flags,fmt", [(3, 0, S.FMT_Q2K), (12, D.FORCE_GEMV, S.FMT_Q2K),
                                         (3, D.FORCE_TC, S.FMT_Q2K), (12, 0, S.FMT_CB2),
                                         (12, 0, S.FMT_MXFP4)],
                         ids=["decode_mma_sync", "decode_tcgen05", "tensor_core",
                              "tensor_core_codebook_down", "tensor_core_mxfp4"])
def test_bounded_wait_expires_and_reports_timeout(orc, T, flags, fmt):
    layer = P.small_layer(seed=31, H=1024, I=512, E=8, k=2, T=T, align=16, fmt=fmt)
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
