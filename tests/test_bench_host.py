"""Host-side pieces of the benchmark, on the CPU: the algorithmic byte and
FLOP counts the roofline divides by (against figures derived by hand from
the block sizes), and the rule that recorded DRAM traffic is reported only
while the profiled kernel's sources are unchanged."""
import json

import pytest

import bench
import ds4g_synth as S


@pytest.mark.parametrize("name,gate_bytes,down_bytes", [
    # Q2_K: 84 bytes per 256 weights; down rows padded to whole super-blocks
    ("tiny", 128 * 1 * 84, 256 * 1 * 84),            # inter 128 < 256: one padded block per row
    ("decode_1tok", 1536 * 16 * 84, 4096 * 6 * 84),   # 2,064,384 and 2,064,384 bytes
    ("decode_32tok", 2048 * 28 * 84, 7168 * 8 * 84),  # 4,816,896 and 4,816,896 bytes
    # codebook format: 70 bytes per 256 weights
    ("codebook_512", 2048 * 28 * 70, 7168 * 8 * 70),  # 4,014,080 and 4,014,080 bytes
    # each matrix in its own format
    ("mixed_2048", 2048 * 28 * 70, 7168 * 8 * 84),    # codebook gate/up, Q2_K down
    ("kquant_32tok", 2048 * 28 * 144, 7168 * 8 * 210),  # Q4_K gate/up, Q6_K down
    ("mxfp4_32tok", 2048 * 28 * 136, 7168 * 8 * 136),   # eight 17-byte blocks per 256 weights
])
def test_layer_bytes_per_expert(name, gate_bytes, down_bytes):
    assert bench.layer_bytes(S.CONFIGS[name]) == (gate_bytes, down_bytes)


def test_decode_1tok_bytes_touched():
    # six experts of three matrices: 37,158,912 bytes of weights per token
    gu, dn = bench.layer_bytes(S.CONFIGS["decode_1tok"])
    assert 6 * (2 * gu + dn) == 37_158_912


def test_recorded_traffic_needs_unchanged_sources(tmp_path, monkeypatch):
    f = tmp_path / "traffic.json"
    good = bench.kernel_source_hash("decode")
    f.write_text(json.dumps({"decode_1tok": {"decode": {"dram_bytes_per_launch": 123.0,
                                                        "source_hash": good}},
                             "prefill_2048": {"tc_gateup": {"dram_bytes_per_launch": 456.0,
                                                            "source_hash": "0" * 16}}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.measured_traffic("decode", "decode_1tok") == 123.0
    assert bench.measured_traffic("tc_gateup", "prefill_2048") is None     # stale hash
    assert bench.measured_traffic("decode", "tiny") is None                # never profiled


def test_source_hash_ignores_comments_and_blank_lines(tmp_path, monkeypatch):
    csrc = tmp_path / "bit_quantized_routed_route_b300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.KERNEL_SOURCES, "probe", ("k.cu",))
    (csrc / "k.cu").write_text("int a = 1;\n")
    h0 = bench.kernel_source_hash("probe")
    (csrc / "k.cu").write_text("// a comment\n\nint a = 1;  // trailing\n")
    assert bench.kernel_source_hash("probe") == h0
    (csrc / "k.cu").write_text("int a = 2;\n")
    assert bench.kernel_source_hash("probe") != h0


@pytest.mark.parametrize("name", list(S.CONFIGS))
def test_layer_path_mirrors_the_library(name):
    """The benchmark's own statement of which kernels run (`layer_path`, used
    for the roofline) agrees with the library's choice, read through
    ds4g_moe_forward_launches on the workload's descriptor (host arithmetic
    only): decode = 2 launches, tensor core = routing + 5, general = routing + 3."""
    import bit_quantized_routed_route_b300 as D
    from test_abi import layer_desc
    cfg = S.CONFIGS[name]
    d = layer_desc(cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k, fmt=cfg.format,
                   align=cfg.row_align, down_fmt=cfg.dn_format)
    route = 1 if cfg.tokens <= 64 else 2
    expect = {"decode": 2, "tc": route + 5, "general": route + 3}[bench.layer_path(cfg)]
    assert D.moe_forward_launches(d, cfg.tokens) == expect

