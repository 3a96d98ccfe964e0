"""Host checks of the seeded input generator (no GPU)."""
import numpy as np
import pytest
import torch

import ds4g_synth as S


def test_weights_do_not_depend_on_thread_count():
    a = S.make_experts(7, S.TENSOR_GATE, 3, 24, 512, S.FMT_Q2K, 168, n_threads=1)
    b = S.make_experts(7, S.TENSOR_GATE, 3, 24, 512, S.FMT_Q2K, 168, n_threads=5)
    assert np.array_equal(a, b)
    cb = S.make_codebook(4)
    a = S.make_experts(7, S.TENSOR_UP, 2, 10, 768, S.FMT_CB2, 224, cb, n_threads=1)
    b = S.make_experts(7, S.TENSOR_UP, 2, 10, 768, S.FMT_CB2, 224, cb, n_threads=3)
    assert np.array_equal(a, b)


def test_seeds_and_tensors_give_distinct_streams():
    a = S.make_experts(1, S.TENSOR_GATE, 1, 4, 256, S.FMT_Q2K, 84)
    b = S.make_experts(1, S.TENSOR_UP, 1, 4, 256, S.FMT_Q2K, 84)
    c = S.make_experts(2, S.TENSOR_GATE, 1, 4, 256, S.FMT_Q2K, 84)
    assert not np.array_equal(a, b) and not np.array_equal(a, c)


def test_row_padding_is_zero():
    w = S.make_experts(3, S.TENSOR_DOWN, 2, 8, 128, S.FMT_Q2K, 96)
    assert np.all(w[:, :, 84:] == 0)
    # columns 128..255 of the single block are zero weights: sub-blocks 8..15
    # carry zero scale bytes and zero quants
    assert np.all(w[:, :, 8:16] == 0)
    assert np.all(w[:, :, 16 + 32 + 0:16 + 64] & 0 == 0)


def test_normals_have_unit_moments():
    x = S.bf16_to_f32(S.make_x(0, 64, 4096)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01


@pytest.mark.parametrize("kind", [S.LOGITS_NORMAL, S.LOGITS_UNIFORM, S.LOGITS_BIASED])
def test_logit_margin(kind):
    lg = S.make_logits(5, kind, 300, 256, 8)
    s = -np.sort(-lg.astype(np.float64), axis=1)
    assert np.all(s[:, 7] - s[:, 8] >= 1e-3)
    if kind == S.LOGITS_UNIFORM:
        assert lg.min() >= 0 and lg.max() < 1


def test_biased_logits_give_uneven_loads():
    lg = S.make_logits(3, S.LOGITS_BIASED, 2048, 256, 8)
    top = np.argsort(-lg, axis=1)[:, :8]
    counts = np.bincount(top.reshape(-1), minlength=256)
    assert counts.max() > 4 * counts.mean()


def test_zipf_logits_skew_and_margin():
    lg = S.make_logits(4, S.LOGITS_ZIPF, 512, 256, 8)
    s = -np.sort(-lg.astype(np.float64), axis=1)
    assert np.all(s[:, 7] - s[:, 8] >= 1.0)
    top = np.argsort(-lg, axis=1)[:, :8]
    counts = np.sort(np.bincount(top.reshape(-1), minlength=256))[::-1]
    assert counts[0] >= 0.8 * 512          # the most popular expert is in most tokens
    assert counts[:16].sum() > counts[16:].sum()


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    f = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        np.array([0.0, -0.0, 1e-40, 3.4e38, np.inf, -np.inf], dtype=np.float32)])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(S.f32_to_bf16(f), ref)
    L = S.lib()
    for v in f[:2000]:
        assert L.syn_f32_to_bf16(float(v)) == S.f32_to_bf16(np.array([v]))[0]


def test_double_to_half_matches_numpy():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 5, 20000),
                        [0.0, 65504.0, 65519.99, 65520.0, 6.0e-8, 2.9e-8, 3.0e-8]])
    with np.errstate(over="ignore"):          # 65520 rounds to infinity on purpose
        ref = v.astype(np.float16).view(np.uint16)
    L = S.lib()
    got = np.array([L.syn_double_to_half(float(x)) for x in v], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_codebook_values():
    cb = S.make_codebook(4)
    assert cb.shape == (256, 8)
    assert set(np.unique(cb).tolist()) == {-43, -25, -8, 8, 25, 43}
    assert np.array_equal(cb, S.make_codebook(4))


def test_config_table():
    c = S.CONFIGS
    assert (c["decode_1tok"].hidden, c["decode_1tok"].inter, c["decode_1tok"].n_experts,
            c["decode_1tok"].top_k, c["decode_1tok"].tokens) == (4096, 1536, 64, 6, 1)
    assert c["codebook_512"].row_bytes(7168) == 1968
    assert c["prefill_2048"].row_bytes(7168) == 2352
    assert c["decode_1tok"].row_bytes(1536) == 504
