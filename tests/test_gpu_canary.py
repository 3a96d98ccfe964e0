"""Nothing outside the caller's buffers is written: the workspace is followed
by 4 KB of canary bytes and y by two canary rows, and after a call on each
kind of path (decode kernels, tensor-core kernels in several formats, GEMV
kernels) both are unchanged.  The call's result is checked against the oracle
too, so the canaries sit next to a call that really ran."""
import numpy as np
import pytest
import torch

import bit_quantized_routed_route_b300 as D
import ds4g_synth as S
import oracle_pins as P
from gpu_helpers import check_output, to_device

pytestmark = pytest.mark.gpu

CANARY = 0xA5
TAIL = 4096


@pytest.mark.parametrize("kw,flags", [
    (dict(H=1024, I=512, E=8, k=2, T=3), 0),                                     # mma.sync decode
    (dict(H=1024, I=512, E=8, k=2, T=12), D.FORCE_GEMV),                         # tcgen05 decode
    (dict(H=1024, I=512, E=8, k=2, T=40, align=16), 0),                          # tensor core, Q2_K
    (dict(H=1024, I=512, E=8, k=2, T=40, fmt=S.FMT_MXFP4), 0),                   # tensor core, MXFP4
    (dict(H=1024, I=2048, E=6, k=2, T=20, fmt=S.FMT_Q4K, down_fmt=S.FMT_Q6K), 0),  # tensor core, K-quant
    (dict(H=512, I=200, E=7, k=3, T=17, fmt=S.FMT_CB2, align=2), 0),            # GEMV kernels
], ids=["decode_mma_sync", "decode_tcgen05", "tc_q2k", "tc_mxfp4", "tc_kquant", "gemv"])
def test_no_write_outside_workspace_and_output(orc, kw, flags):
    layer = P.small_layer(seed=97 + kw["T"], score=S.SCORE_SIGMOID, **kw)
    L = to_device(layer, flags=flags)
    T, H = layer["x"].shape
    dev = torch.device("cuda")
    x = torch.from_numpy(layer["x"].view(np.int16)).to(dev)
    lg = torch.from_numpy(layer["logits"]).to(dev)
    ws_bytes = L.workspace_bytes(T)
    ws = torch.full((ws_bytes + TAIL,), CANARY, dtype=torch.uint8, device=dev)
    y_all = torch.full((T + 2, H), float("nan"), dtype=torch.float32, device=dev)
    D.check(D.moe_forward(L.desc, x, lg, T, y_all[:T], ws, ws_bytes))
    torch.cuda.synchronize()
    assert bool((ws[ws_bytes:] == CANARY).all())
    assert bool(torch.isnan(y_all[T:]).all())
    yref, _, _ = orc.moe_forward(layer, layer["x"], layer["logits"])
    check_output(y_all[:T].cpu().numpy(), yref)
