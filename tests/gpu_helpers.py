"""Helpers for the GPU parity tests: move a synthetic layer to the device, run
the library through its C ABI, and compare against the oracle with the
layer's tolerances."""
from __future__ import annotations

import numpy as np
import torch

import bit_quantized_routed_route_b300 as D
import ds4g_synth as S

# Tolerances of the layer output (per token, and over the whole tensor).
REL_L2_TOL = 1e-3
MAX_ABS_TOL = 5e-3
WEIGHT_REL_TOL = 1e-6

_layers = {}


def cached_layer(name: str) -> dict:
    """One synthetic layer per configuration name per process."""
    if name not in _layers:
        _layers[name] = S.make_layer(S.CONFIGS[name])
    return _layers[name]


def to_device(layer: dict, flags: int = 0, tc_min_tokens: int = 0) -> D.Layer:
    dev = torch.device("cuda")
    key = "_dev"
    if key not in layer:
        cb = layer.get("codebook")
        layer[key] = dict(
            w_gate=torch.from_numpy(layer["w_gate"]).to(dev),
            w_up=torch.from_numpy(layer["w_up"]).to(dev),
            w_down=torch.from_numpy(layer["w_down"]).to(dev),
            codebook=None if cb is None else torch.from_numpy(cb).to(dev),
        )
    t = layer[key]
    return D.Layer(layer["hidden"], layer["inter"], layer["n_experts"], layer["top_k"],
                   layer["score"], layer["format"], t["w_gate"], t["w_up"], t["w_down"],
                   t["codebook"], flags=flags, tc_min_tokens=tc_min_tokens,
                   down_fmt=layer.get("down_format"))


def run_forward(L: D.Layer, x: np.ndarray, logits: np.ndarray, with_status: bool = False):
    """Runs ds4g_moe_forward; returns (y fp32 numpy, routing dict of numpy
    arrays read back through ds4g_moe_routing_view), and with `with_status`
    the workspace status word (ds4g_moe_device_status) third."""
    dev = torch.device("cuda")
    T = x.shape[0]
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev)
    ld = torch.from_numpy(np.ascontiguousarray(logits)).to(dev)
    H, E, k = L.desc.hidden, L.desc.n_experts, L.desc.top_k
    y = torch.full((T, H), float("nan"), dtype=torch.float32, device=dev)
    ws_bytes = L.workspace_bytes(T)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    D.check(D.moe_forward(L.desc, xd, ld, T, y, ws, ws_bytes))
    torch.cuda.synchronize()
    st, v = D.moe_routing_view(L.desc, T, ws, ws_bytes)
    D.check(st)

    def grab(addr, n, dtype):
        out = torch.empty(n, dtype=dtype, device=dev)
        if n:
            nbytes = n * out.element_size()
            # copy from the raw workspace address through a byte view of ws
            off = addr - ws.data_ptr()
            out.view(torch.uint8).copy_(ws[off:off + nbytes])
        return out.cpu().numpy()

    A = T * k
    routing = dict(ids=grab(v["ids"], A, torch.int32).reshape(T, k),
                   weights=grab(v["weights"], A, torch.float32).reshape(T, k),
                   counts=grab(v["counts"], E, torch.int32),
                   offsets=grab(v["offsets"], E + 1, torch.int32),
                   perm=grab(v["perm"], A, torch.int32))
    if with_status:
        st, dev_status = D.moe_device_status(L.desc, T, ws, ws_bytes)
        D.check(st)
        return y.cpu().numpy(), routing, dev_status
    return y.cpu().numpy(), routing


def oracle_tokens(orc, layer: dict, x: np.ndarray, logits: np.ndarray, tokens=None):
    """The oracle's y for the listed tokens (all when None), computed on all
    host cores: the oracle is re-entrant and ctypes releases the GIL, so the
    tokens are split across threads.  Returns fp64 [n x H]."""
    import concurrent.futures as cf
    import os
    T = x.shape[0]
    tok = np.arange(T, dtype=np.int32) if tokens is None else np.asarray(tokens, dtype=np.int32)
    n_thr = max(1, min(len(tok), os.cpu_count() or 1))
    parts = np.array_split(tok, n_thr)
    with cf.ThreadPoolExecutor(n_thr) as ex:
        outs = list(ex.map(lambda tk: orc.moe_forward(layer, x, logits, tk)[0], parts))
    return np.concatenate(outs, axis=0)


def boundary_tokens(route: dict, k: int, T: int, n_total: int, seed: int) -> np.ndarray:
    """Tokens that exercise every code path of a large call: the first and
    last token of the three heaviest expert segments and the tokens on both
    sides of each 128-token tile boundary inside them, tokens routed to
    one-token segments, then seeded random tokens up to n_total."""
    counts, offsets, perm = route["counts"], route["offsets"], route["perm"]
    picks = []
    for e in np.argsort(-counts, kind="stable")[:3]:
        n = int(counts[e])
        pos = {0, n - 1}
        for b in range(128, n, 128):
            pos.update((b - 1, b))
        picks += [int(perm[offsets[e] + q]) // k for q in sorted(pos) if 0 <= q < n]
    for e in np.nonzero(counts == 1)[0][:16]:
        picks.append(int(perm[offsets[e]]) // k)
    out = list(dict.fromkeys(picks))
    rng = np.random.default_rng(seed)
    for t in rng.permutation(T):
        if len(out) >= n_total:
            break
        if int(t) not in out:
            out.append(int(t))
    return np.sort(np.array(out, dtype=np.int32))


def check_output(y: np.ndarray, yref: np.ndarray, rel_l2=REL_L2_TOL, max_abs=MAX_ABS_TOL):
    """Per-token relative L2 <= rel_l2 and max-abs <= max_abs * max|ref|; a
    token whose reference is exactly zero must be exactly zero."""
    assert np.all(np.isfinite(y)), "non-finite output"
    err = y.astype(np.float64) - yref
    ref_n = np.linalg.norm(yref, axis=1)
    err_n = np.linalg.norm(err, axis=1)
    zero = ref_n == 0
    assert np.all(err_n[zero] == 0), "token with zero reference is not zero"
    rel = err_n[~zero] / ref_n[~zero]
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= rel_l2, f"per-token relative L2 {worst:.3e} > {rel_l2}"
    scale = np.abs(yref).max()
    mx = float(np.abs(err).max())
    assert mx <= max_abs * scale, f"max-abs {mx:.3e} > {max_abs} * {scale:.3e}"
    return worst, mx / scale if scale else 0.0


def check_routing(routing: dict, ref: dict, tokens=None):
    """ids / counts / offsets / perm bit-exact, weights within 1e-6 relative."""
    ids = routing["ids"] if tokens is None else routing["ids"][tokens]
    rids = ref["ids"] if tokens is None else ref["ids"][tokens]
    assert np.array_equal(ids, rids)
    w = routing["weights"] if tokens is None else routing["weights"][tokens]
    rw = ref["weights"] if tokens is None else ref["weights"][tokens]
    assert np.all(np.abs(w - rw) <= WEIGHT_REL_TOL * np.abs(rw) + 1e-30)
    if tokens is None:
        for key in ("counts", "offsets", "perm"):
            assert np.array_equal(routing[key], ref[key]), key
