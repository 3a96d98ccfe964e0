"""ds4g_route_topk against the oracle: ids, counts, offsets and perm
bit-exact; weights within 1e-6 relative."""
import numpy as np
import pytest
import torch

import bit_quantized_routed_route_b300 as D
import ds4g_synth as S
from gpu_helpers import WEIGHT_REL_TOL

pytestmark = pytest.mark.gpu


def gpu_route(logits, k, score):
    dev = torch.device("cuda")
    T, E = logits.shape
    lg = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(dev)
    ids = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device=dev)
    counts = torch.full((E,), -7, dtype=torch.int32, device=dev)
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    perm = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
    D.check(D.route_topk(lg, T, E, k, score, ids, w, counts, offsets, perm))
    torch.cuda.synchronize()
    return dict(ids=ids.cpu().numpy(), weights=w.cpu().numpy(), counts=counts.cpu().numpy(),
                offsets=offsets.cpu().numpy(), perm=perm.cpu().numpy())


def compare(got, ref):
    assert np.array_equal(got["ids"], ref["ids"])
    assert np.array_equal(got["counts"], ref["counts"])
    assert np.array_equal(got["offsets"], ref["offsets"])
    assert np.array_equal(got["perm"], ref["perm"])
    rw, w = ref["weights"], got["weights"]
    both_nan = np.isnan(rw) & np.isnan(w)      # softmax over k picks that are all -inf
    ok = np.abs(w - rw) <= WEIGHT_REL_TOL * np.abs(rw) + 1e-30
    assert np.all(ok | both_nan)


@pytest.mark.parametrize("name", list(S.CONFIGS))
def test_route_configs(orc, name):
    c = S.CONFIGS[name]
    lg = S.make_logits(c.seed, c.logits, c.tokens, c.n_experts, c.top_k)
    compare(gpu_route(lg, c.top_k, c.score), orc.route(lg, c.top_k, c.score))


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (1, 256, 8), (5, 33, 7), (64, 200, 8), (65, 8, 8),
                                   (700, 64, 6), (3000, 256, 8), (129, 31, 3)])
@pytest.mark.parametrize("score", [D.SCORE_SOFTMAX, D.SCORE_SIGMOID])
def test_route_shapes_with_ties_and_nan(orc, T, E, k, score):
    rng = np.random.default_rng(T * 1000 + E)
    lg = (rng.integers(-6, 7, size=(T, E)) * 0.25).astype(np.float32)   # many exact ties
    lg[rng.random((T, E)) < 0.02] = np.nan
    lg[rng.random((T, E)) < 0.02] = -np.inf
    compare(gpu_route(lg, k, score), orc.route(lg, k, score))


def test_route_empty():
    dev = torch.device("cuda")
    counts = torch.full((8,), 5, dtype=torch.int32, device=dev)
    offsets = torch.full((9,), 5, dtype=torch.int32, device=dev)
    lg = torch.zeros((1, 8), device=dev)
    ids = torch.zeros((1, 2), dtype=torch.int32, device=dev)
    w = torch.zeros((1, 2), device=dev)
    D.check(D.route_topk(lg, 0, 8, 2, 0, ids, w, counts, offsets, None))
    torch.cuda.synchronize()
    assert counts.cpu().tolist() == [0] * 8 and offsets.cpu().tolist() == [0] * 9
