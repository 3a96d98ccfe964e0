"""ds4g_expert_cache: layers whose experts live in page-locked host memory,
a few of them resident in device slots, uploaded on misses.

The cache runs the ordinary kernels on the slots, so its output must be
bit-identical to ds4g_moe_forward on a device-resident copy of the same
weights, on every path (decode, tensor-core, general kernels), call after
call while experts are evicted and uploaded again.  Also checked: the LRU
choice of victims, the hit / miss / byte accounting, the refusal of a call
that routes to more experts than there are slots, and that an out-of-range
slot map entry is reported in the device status word instead of reading
outside the weight tensors."""
import ctypes

import numpy as np
import pytest
import torch

import bit_quantized_routed_route_b300 as D
import ds4g_synth as S
import oracle_pins as P
from gpu_helpers import check_output, run_forward, to_device

pytestmark = pytest.mark.gpu


def _host_cache(layer, n_slots, flags=0):
    t = {n: torch.from_numpy(layer[n]).pin_memory() for n in ("w_gate", "w_up", "w_down")}
    cb = layer.get("codebook")
    cbd = None if cb is None else torch.from_numpy(cb).cuda()
    c = D.ExpertCache(layer["hidden"], layer["inter"], layer["n_experts"], layer["top_k"],
                      layer["score"], layer["format"], t["w_gate"], t["w_up"], t["w_down"],
                      n_slots, codebook=cbd, flags=flags, down_fmt=layer.get("down_format"))
    c._keep = (t, cbd)
    return c


def _cache_forward(c, x_np, lg_np):
    dev = torch.device("cuda")
    T = x_np.shape[0]
    x = torch.from_numpy(x_np.view(np.int16)).to(dev)
    lg = torch.from_numpy(lg_np).to(dev)
    y = torch.full((T, c.host.desc.hidden), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(max(c.workspace_bytes(T), 1), dtype=torch.uint8, device=dev)
    st = c.forward(x, lg, y, ws)
    torch.cuda.synchronize()
    return st, y.cpu().numpy()


def _expert_bytes(layer):
    return 2 * layer["gate_up_expert_stride"] + layer["down_expert_stride"]


def lru_model(calls, n_slots):
    """The documented policy, call by call: hits keep their slot; each miss
    (in expert order) takes a free slot, else the least recently used slot
    of an expert this call does not route to (ties -> lowest slot).  Yields
    the running (hits, misses)."""
    owner, stamp, slot_of = [-1] * n_slots, [0] * n_slots, {}
    hits = misses = 0
    for now, routed in enumerate(calls, 1):
        for e in routed:
            if e in slot_of:
                stamp[slot_of[e]] = now
        for e in sorted(routed):
            if e in slot_of:
                hits += 1
                continue
            v = -1
            for sl in range(n_slots):
                if stamp[sl] == now:
                    continue
                if owner[sl] < 0:
                    v = sl
                    break
                if v < 0 or stamp[sl] < stamp[v]:
                    v = sl
            if owner[v] >= 0:
                del slot_of[owner[v]]
            owner[v], slot_of[e], stamp[v] = e, v, now
            misses += 1
        yield hits, misses


def _budget_logits(rng, T, E, n_slots):
    """Logits whose top-k all come from one random set of n_slots experts."""
    keep = rng.choice(E, size=n_slots, replace=False)
    lg = (rng.standard_normal((T, E)) - 8.0).astype(np.float32)
    lg[:, keep] = rng.standard_normal((T, n_slots)).astype(np.float32) * 2.0
    return lg


@pytest.mark.parametrize("kw,flags", [
    (dict(H=1024, I=512, E=16, k=2, T=5), 0),                               # decode kernels
    (dict(H=512, I=256, E=12, k=3, T=40, align=16), D.FORCE_TC),            # tensor-core kernels
    (dict(H=512, I=320, E=10, k=2, T=9, fmt=S.FMT_Q4K, down_fmt=S.FMT_Q6K), 0),   # general
    (dict(H=512, I=256, E=10, k=2, T=7, fmt=S.FMT_CB2, align=16), 0),       # codebook
    (dict(H=512, I=2048, E=10, k=2, T=9, fmt=S.FMT_Q4K, down_fmt=S.FMT_Q6K), 0),  # K-quant, tensor core
    (dict(H=512, I=512, E=10, k=2, T=9, fmt=S.FMT_MXFP4), 0),              # MXFP4, tensor core
], ids=["decode", "tensor_core", "kquant", "codebook", "kquant_tc", "mxfp4_tc"])
def test_cache_matches_device_forward(orc, kw, flags):
    layer = P.small_layer(seed=61 + kw["T"], **kw)
    E, k, T = layer["n_experts"], layer["top_k"], layer["x"].shape[0]
    n_slots = E // 2
    c = _host_cache(layer, n_slots, flags=flags)
    L = to_device(layer, flags=flags)
    rng = np.random.default_rng(5)
    calls = [_budget_logits(rng, T, E, n_slots) for _ in range(8)]
    routed = [set(orc.route(lg, k, layer["score"])["ids"].ravel().tolist()) for lg in calls]
    for i, (lg, expect) in enumerate(zip(calls, lru_model(routed, n_slots))):
        st, y = _cache_forward(c, layer["x"], lg)
        assert st == D.OK, D.status_string(st)
        yd, _ = run_forward(L, layer["x"], lg)
        assert np.array_equal(y.view(np.uint32), yd.view(np.uint32)), f"call {i}"
        h, m, b = c.stats()
        assert (h, m) == expect, (i, (h, m), expect)
        assert b == m * _expert_bytes(layer)
    assert m > len(routed[0])                 # experts were evicted and uploaded again
    yref, _, _ = orc.moe_forward(layer, layer["x"], calls[-1])
    check_output(y, yref)
    c.close()


def _one_token_logits(E, picks):
    lg = np.full((1, E), -4.0, dtype=np.float32)
    for i, e in enumerate(picks):
        lg[0, e] = 4.0 - i
    return lg


def test_cache_evicts_least_recently_used():
    """A worked sequence on 3 slots (hits, misses after each call):
    {0,1} -> (0,2); {1,2} -> (1,3): expert 2 takes the free slot;
    {3,1} -> (2,4): expert 0 (last used in call 1) is evicted;
    {0,2} -> (3,5): slots of 3 and 1 were both last used in call 3, the lower
    slot (expert 3's) goes; {1,3} -> (4,6): expert 1 hits, expert 3 evicts
    expert 0 (slots of 0 and 2 last used in call 4, lower slot first)."""
    layer = P.small_layer(seed=71, H=512, I=256, E=8, k=2, T=1)
    c = _host_cache(layer, n_slots=3)
    L = to_device(layer)
    x = layer["x"]
    steps = [((0, 1), (0, 2)), ((1, 2), (1, 3)), ((3, 1), (2, 4)), ((0, 2), (3, 5)),
             ((1, 3), (4, 6))]
    for picks, expect in steps:
        lg = _one_token_logits(8, picks)
        st, y = _cache_forward(c, x, lg)
        assert st == D.OK
        yd, _ = run_forward(L, x, lg)
        assert np.array_equal(y.view(np.uint32), yd.view(np.uint32))
        assert c.stats()[:2] == expect, (picks, c.stats(), expect)
    assert [e for e in lru_model([set(p) for p, _ in steps], 3)] == [e for _, e in steps]
    c.close()


def test_cache_refuses_calls_beyond_its_slots():
    layer = P.small_layer(seed=72, H=512, I=256, E=8, k=2, T=3)
    c = _host_cache(layer, n_slots=3)
    lg = np.full((3, 8), -4.0, dtype=np.float32)
    for t in range(3):
        lg[t, 2 * t] = 3.0
        lg[t, 2 * t + 1] = 2.0                          # six distinct experts > 3 slots
    st, y = _cache_forward(c, layer["x"], lg)
    assert st == D.ERR_UNSUPPORTED
    assert np.all(np.isnan(y))
    assert c.stats()[:2] == (0, 0)
    c.close()


@pytest.mark.parametrize("kw,flags", [
    (dict(H=1024, I=512, E=8, k=2, T=3), 0),                                # decode kernels
    (dict(H=512, I=256, E=8, k=2, T=40, align=16), D.FORCE_TC),             # tensor-core kernels
    (dict(H=512, I=320, E=8, k=2, T=5), D.FORCE_GEMV),                      # general kernels
], ids=["decode", "tensor_core", "general"])
def test_bad_slot_map_is_reported_not_read(kw, flags):
    """Every expert mapped to slot 7 of a 2-slot layer: the kernels read slot
    0 instead and the workspace status word reads DS4G_ERR_INVALID."""
    layer = P.small_layer(seed=73, **kw)
    L = to_device(layer, flags=flags)
    dev = torch.device("cuda")
    d = D.MoeDesc.from_buffer_copy(L.desc)
    smap = torch.full((layer["n_experts"],), 7, dtype=torch.int32, device=dev)
    d.n_slots = 2
    d.expert_slot = smap.data_ptr()
    T, H = layer["x"].shape
    x = torch.from_numpy(layer["x"].view(np.int16)).to(dev)
    lg = torch.from_numpy(layer["logits"]).to(dev)
    y = torch.empty((T, H), dtype=torch.float32, device=dev)
    ws = torch.empty(D.moe_workspace_bytes(d, T), dtype=torch.uint8, device=dev)
    D.check(D.moe_forward(d, x, lg, T, y, ws))
    st, v = D.moe_device_status(d, T, ws)
    assert st == D.OK and v == D.ERR_INVALID
    # the device is fine afterwards: a correct map gives the plain result
    smap.copy_(torch.arange(layer["n_experts"], dtype=torch.int32, device=dev))
    d.n_slots = layer["n_experts"]
    D.check(D.moe_forward(d, x, lg, T, y, ws))
    st, v = D.moe_device_status(d, T, ws)
    assert st == D.OK and v == D.OK
    yd, _ = run_forward(L, layer["x"], layer["logits"])
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().view(np.uint32), yd.view(np.uint32))
