"""The C-ABI library on the CPU (no GPU calls): it loads, exports every symbol
that include/ds4g.h declares, and rejects bad arguments on the host before
any launch."""
import ctypes
import os
import re

import pytest

import bit_quantized_routed_route_b300 as D

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ds4g.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DS4G_API\s+[\w\s\*]+?\b(ds4g_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    assert set(D.EXPORTED) <= set(names), names
    assert len(names) >= 9


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(D.LIBRARY)
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings():
    assert D.abi_version() == 3
    assert D.status_string(D.OK) == "ok"
    for s in range(1, 9):
        assert D.status_string(s) not in ("ok", "unknown status")
    assert D.status_string(99) == "unknown status"


FAKE = 1 << 20   # a 256-byte aligned address that is never dereferenced


def desc(**kw):
    d = D.MoeDesc()
    d.hidden, d.inter, d.n_experts, d.top_k = 256, 128, 8, 2
    d.score, d.format, d.flags, d.tc_min_tokens = D.SCORE_SOFTMAX, D.FMT_Q2K, 0, 0
    d.down_format, d.n_slots = D.FMT_Q2K, 0
    d.w_gate = d.w_up = d.w_down = FAKE
    d.gate_up_row_bytes, d.down_row_bytes = 84, 84
    d.gate_up_expert_stride, d.down_expert_stride = 128 * 84, 256 * 84
    d.codebook = None
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def fwd(d, T=4, ws_bytes=None, ws=FAKE, x=FAKE, logits=FAKE, y=FAKE):
    if ws_bytes is None:
        ws_bytes = max(D.moe_workspace_bytes(d, T), 1)
    return D.lib().ds4g_moe_forward(ctypes.byref(d), x, logits, T, y, ws, ws_bytes, None)


def test_workspace_size_is_positive_and_grows_with_T():
    d = desc()
    a, b = D.moe_workspace_bytes(d, 4), D.moe_workspace_bytes(d, 400)
    assert 0 < a < b and a % 256 == 0


def test_noalloc_scratch_covers_a_32_token_decode_of_the_7168_layer():
    # the static scratch size is stated in the header and mirrored in Python
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "ds4g.h")).read()
    m = re.search(r"#define DS4G_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", hdr)
    assert m and int(m.group(1)) << int(m.group(2)) == D.NOALLOC_SCRATCH_BYTES
    H, I, E, k = 7168, 2048, 256, 8
    row = H // 256 * 84
    d = desc(hidden=H, inter=I, n_experts=E, top_k=k, score=D.SCORE_SIGMOID,
             gate_up_row_bytes=row, down_row_bytes=I // 256 * 84,
             gate_up_expert_stride=I * row, down_expert_stride=H * (I // 256 * 84))
    assert 0 < D.moe_workspace_bytes(d, 32) <= D.NOALLOC_SCRATCH_BYTES
    assert D.moe_workspace_bytes(d, 2048) > D.NOALLOC_SCRATCH_BYTES


@pytest.mark.parametrize("kw,code", [
    (dict(hidden=300), D.ERR_SHAPE),
    (dict(hidden=0), D.ERR_SHAPE),
    (dict(inter=0), D.ERR_SHAPE),
    (dict(n_experts=0), D.ERR_INVALID),
    (dict(n_experts=257), D.ERR_INVALID),
    (dict(top_k=9, n_experts=16), D.ERR_INVALID),
    (dict(top_k=3, n_experts=2), D.ERR_INVALID),
    (dict(score=2), D.ERR_INVALID),
    (dict(format=6), D.ERR_INVALID),
    (dict(down_format=6), D.ERR_INVALID),
    (dict(format=D.FMT_Q6K, gate_up_row_bytes=210, gate_up_expert_stride=128 * 224),
     D.ERR_INVALID),                                                       # Q6_K is down-only
    (dict(down_format=D.FMT_Q4K, down_row_bytes=146), D.ERR_LAYOUT),       # Q4_K rows % 4
    (dict(n_slots=1), D.ERR_INVALID),                       # slots without a map
    (dict(n_slots=-1), D.ERR_INVALID),
    (dict(expert_slot=FAKE), D.ERR_INVALID),                # a map without slots
    (dict(n_slots=4, expert_slot=FAKE + 2), D.ERR_LAYOUT),
    (dict(down_format=D.FMT_CB2, down_row_bytes=70), D.ERR_INVALID),      # no codebook
    (dict(flags=D.FORCE_GEMV | D.FORCE_TC), D.ERR_INVALID),
    (dict(flags=64), D.ERR_INVALID),
    (dict(tc_min_tokens=-1), D.ERR_INVALID),
    (dict(w_up=None), D.ERR_INVALID),
    (dict(format=D.FMT_CB2, gate_up_row_bytes=70, down_row_bytes=70,
          gate_up_expert_stride=128 * 80, down_expert_stride=256 * 80), D.ERR_INVALID),
    (dict(gate_up_row_bytes=80), D.ERR_LAYOUT),
    (dict(gate_up_row_bytes=86), D.ERR_LAYOUT),
    (dict(gate_up_expert_stride=100 * 84), D.ERR_LAYOUT),
    (dict(down_expert_stride=256 * 84 + 4), D.ERR_LAYOUT),
    (dict(w_gate=FAKE + 8), D.ERR_LAYOUT),
    (dict(flags=D.FORCE_TC), D.ERR_LAYOUT),
])
def test_forward_rejects_bad_descriptors(kw, code):
    d = desc(**kw)
    assert fwd(d, ws_bytes=1 << 30) == code
    assert D.moe_workspace_bytes(d, 4) == 0


def test_forward_rejects_bad_calls():
    d = desc()
    need = D.moe_workspace_bytes(d, 4)
    assert fwd(d, T=-1, ws_bytes=need) == D.ERR_INVALID
    assert fwd(d, T=D.lib().ds4g_abi_version() * 70000, ws_bytes=1 << 40) == D.ERR_SHAPE
    assert fwd(d, ws_bytes=need - 1) == D.ERR_WORKSPACE
    assert fwd(d, ws=FAKE + 16, ws_bytes=need) == D.ERR_WORKSPACE
    assert fwd(d, x=None, ws_bytes=need) == D.ERR_INVALID
    assert fwd(d, x=FAKE + 2, ws_bytes=need) == D.ERR_LAYOUT
    assert fwd(d, y=FAKE + 4, ws_bytes=need) == D.ERR_LAYOUT
    # T == 0 is a no-op that touches nothing
    assert fwd(d, T=0, ws=None, x=None, logits=None, y=None, ws_bytes=0) == D.OK
    assert D.lib().ds4g_moe_forward(None, FAKE, FAKE, 4, FAKE, FAKE, 1 << 30, None) == D.ERR_INVALID


def test_host_entry_point_validates_first():
    d = desc()
    L = D.lib()
    assert L.ds4g_moe_forward_host(ctypes.byref(d), FAKE, FAKE, 4, FAKE, FAKE, 10, None) == D.ERR_WORKSPACE
    assert L.ds4g_moe_forward_host(ctypes.byref(desc(hidden=100)), FAKE, FAKE, 4, FAKE, FAKE, 1 << 30,
                                   None) == D.ERR_SHAPE


def test_route_topk_validation():
    L = D.lib()
    assert L.ds4g_route_topk(None, 4, 8, 2, 0, FAKE, FAKE, None, None, None, None) == D.ERR_INVALID
    assert L.ds4g_route_topk(FAKE, 4, 8, 9, 0, FAKE, FAKE, None, None, None, None) == D.ERR_INVALID
    assert L.ds4g_route_topk(FAKE, 4, 8, 4, 3, FAKE, FAKE, None, None, None, None) == D.ERR_INVALID
    assert L.ds4g_route_topk(FAKE, 4, 300, 4, 0, FAKE, FAKE, None, None, None, None) == D.ERR_INVALID
    assert L.ds4g_route_topk(FAKE, -1, 8, 2, 0, FAKE, FAKE, None, None, None, None) == D.ERR_INVALID
    assert L.ds4g_route_topk(FAKE, 70000, 8, 2, 0, FAKE, FAKE, None, None, None, None) == D.ERR_SHAPE
    assert L.ds4g_route_topk(FAKE + 2, 4, 8, 2, 0, FAKE, FAKE, None, None, None, None) == D.ERR_LAYOUT


def test_dequant_validation():
    L = D.lib()
    assert L.ds4g_q2k_dequant(FAKE, 0, FAKE, D.F32, None) == D.OK          # no-op
    assert L.ds4g_q2k_dequant(FAKE, -1, FAKE, D.F32, None) == D.ERR_INVALID
    assert L.ds4g_q2k_dequant(FAKE, 4, FAKE, 7, None) == D.ERR_INVALID
    assert L.ds4g_q2k_dequant(None, 4, FAKE, D.F32, None) == D.ERR_INVALID
    assert L.ds4g_q2k_dequant(FAKE + 2, 4, FAKE, D.F32, None) == D.ERR_LAYOUT
    assert L.ds4g_q2k_dequant(FAKE, 4, FAKE + 4, D.F16, None) == D.ERR_LAYOUT
    assert L.ds4g_cb2_dequant(FAKE, 4, None, FAKE, D.F32, None) == D.ERR_INVALID
    assert L.ds4g_cb2_dequant(FAKE + 1, 4, FAKE, FAKE, D.F32, None) == D.ERR_LAYOUT
    for fn, balign in ((L.ds4g_q4k_dequant, 4), (L.ds4g_q5k_dequant, 4), (L.ds4g_q6k_dequant, 2),
                       (L.ds4g_mxfp4_dequant, 4)):
        assert fn(FAKE, 0, FAKE, D.F32, None) == D.OK
        assert fn(FAKE, -1, FAKE, D.F32, None) == D.ERR_INVALID
        assert fn(FAKE, 4, FAKE, 3, None) == D.ERR_INVALID
        assert fn(None, 4, FAKE, D.F32, None) == D.ERR_INVALID
        assert fn(FAKE + balign // 2, 4, FAKE, D.F32, None) == D.ERR_LAYOUT
        assert fn(FAKE, 4, FAKE + 8, D.BF16, None) == D.ERR_LAYOUT


def test_routing_view_points_inside_the_workspace():
    d = desc()
    need = D.moe_workspace_bytes(d, 4)
    st, v = D.moe_routing_view(d, 4, FAKE, need)
    assert st == D.OK
    for name in ("ids", "weights", "counts", "offsets", "perm"):
        assert FAKE <= v[name] < FAKE + need and (v[name] - FAKE) % 256 == 0
    assert len({v[n] for n in v}) == 5
    st, _ = D.moe_routing_view(d, 4, FAKE, need - 1)
    assert st == D.ERR_WORKSPACE

def layer_desc(H, I, E, k, fmt=None, flags=0, align=1, down_fmt=None, tc_min_tokens=0):
    """A descriptor with packed (or `align`-padded) rows at a fake address;
    W_down in `down_fmt` (default: fmt)."""
    fmt = D.FMT_Q2K if fmt is None else fmt
    down_fmt = fmt if down_fmt is None else down_fmt
    sizes = {D.FMT_Q2K: 84, D.FMT_CB2: 70, D.FMT_Q4K: 144, D.FMT_Q5K: 176, D.FMT_Q6K: 210,
             D.FMT_MXFP4: 136}
    bb, dbb = sizes[fmt], sizes[down_fmt]
    gr, dr = H // 256 * bb, -(-I // 256) * dbb
    gr, dr = -(-gr // align) * align, -(-dr // align) * align
    return desc(hidden=H, inter=I, n_experts=E, top_k=k, format=fmt, down_format=down_fmt,
                flags=flags, tc_min_tokens=tc_min_tokens, gate_up_row_bytes=gr, down_row_bytes=dr,
                gate_up_expert_stride=-(-I * gr // 16) * 16,
                down_expert_stride=-(-H * dr // 16) * 16,
                codebook=FAKE if D.FMT_CB2 in (fmt, down_fmt) else None)


def test_mixed_format_descriptor_is_accepted():
    """Codebook gate/up with Q2_K down (the shipping mix) and the reverse:
    each matrix's rows are checked against its own block size."""
    d = layer_desc(7168, 2048, 256, 8, fmt=D.FMT_CB2, down_fmt=D.FMT_Q2K, align=16)
    assert (d.gate_up_row_bytes, d.down_row_bytes) == (1968, 672)
    assert D.moe_workspace_bytes(d, 64) > 0
    d = layer_desc(512, 256, 4, 2, fmt=D.FMT_Q2K, down_fmt=D.FMT_CB2)
    assert (d.gate_up_row_bytes, d.down_row_bytes) == (168, 70)
    assert D.moe_workspace_bytes(d, 4) > 0
    # W_down rows sized for the gate/up format are too short
    d = layer_desc(512, 512, 4, 2, fmt=D.FMT_CB2, down_fmt=D.FMT_Q2K)
    d.down_row_bytes = 2 * 70
    assert D.moe_workspace_bytes(d, 4) == 0


@pytest.mark.parametrize("shape,T,kw,launches", [
    # decode kernels (reset + fused layer): Q2_K, inter % 16 == 0, up to 3
    # vectors, or up to 32 where the tensor-core kernels cannot stage the rows
    # (504-byte W_down rows here)
    ((4096, 1536, 64, 6), 1, {}, 2),
    ((4096, 1536, 64, 6), 32, {}, 2),
    ((7168, 2048, 256, 8), 3, {}, 2),
    # tensor-core path from 4 vectors: routing (1 launch up to 64 tokens, else
    # 2) + token exponents, prep/gather, gate/up, down, combine
    ((7168, 2048, 256, 8), 4, {}, 1 + 5),
    ((7168, 2048, 256, 8), 32, {}, 1 + 5),
    ((7168, 2048, 256, 8), 33, {}, 1 + 5),
    ((7168, 2048, 256, 8), 65, {}, 2 + 5),
    # rows that are not multiples of 16 bytes: GEMV kernels (routing + 3)
    ((512, 320, 8, 2), 100, {}, 2 + 3),
    # the codebook format never takes the decode kernels
    ((7168, 2048, 256, 8), 1, dict(fmt=D.FMT_CB2, align=16), 1 + 5),
    ((7168, 2048, 256, 8), 1, dict(fmt=D.FMT_CB2), 1 + 3),
    # mixed formats never take the (Q2_K-only) decode kernels
    ((7168, 2048, 256, 8), 1, dict(fmt=D.FMT_CB2, down_fmt=D.FMT_Q2K, align=16), 1 + 5),
    ((7168, 2048, 256, 8), 1, dict(fmt=D.FMT_Q2K, down_fmt=D.FMT_CB2), 1 + 5),   # 560-byte rows
    ((7168, 1024, 256, 8), 1, dict(fmt=D.FMT_Q2K, down_fmt=D.FMT_CB2), 1 + 3),   # 280-byte rows
    # FORCE_GEMV keeps the decode kernels where they apply and rules out the
    # tensor-core kernels elsewhere; FORCE_TC needs 16-byte rows (504-byte down rows here)
    ((4096, 1536, 64, 6), 1, dict(flags=D.FORCE_GEMV), 2),
    ((7168, 2048, 256, 8), 100, dict(flags=D.FORCE_GEMV), 2 + 3),
    ((7168, 2048, 256, 8), 32, dict(flags=D.FORCE_GEMV), 2),
    ((4096, 1536, 64, 6), 1, dict(flags=D.FORCE_TC), 0),
    # per-segment split on the tensor-core path: + GEMV gate/up and down
    ((7168, 2048, 256, 8), 2048, dict(tc_min_tokens=16), 2 + 5 + 2),
    ((7168, 2048, 256, 8), 3, dict(tc_min_tokens=16), 2),         # decode kernels: no split
    # the Q4_K / Q5_K / Q6_K and MXFP4 formats take the tensor-core kernels at
    # every T when their rows are multiples of 16 bytes (Q6_K: I_pad a multiple
    # of 2048; MXFP4: an even number of 136-byte units), alone or mixed
    ((7168, 2048, 256, 8), 32, dict(fmt=D.FMT_Q4K, down_fmt=D.FMT_Q6K), 1 + 5),
    ((7168, 2048, 256, 8), 2048, dict(fmt=D.FMT_Q5K), 2 + 5),
    ((7168, 2048, 256, 8), 1, dict(fmt=D.FMT_Q2K, down_fmt=D.FMT_Q4K), 1 + 5),
    ((7168, 2048, 256, 8), 64, dict(fmt=D.FMT_Q4K, flags=D.FORCE_TC), 1 + 5),
    ((7168, 2048, 256, 8), 32, dict(fmt=D.FMT_MXFP4), 1 + 5),
    ((7168, 2048, 256, 8), 1, dict(fmt=D.FMT_MXFP4, down_fmt=D.FMT_Q2K), 1 + 5),
    ((7168, 2048, 256, 8), 2048, dict(fmt=D.FMT_MXFP4, down_fmt=D.FMT_Q6K), 2 + 5),
    # otherwise the GEMV kernels: 408-byte MXFP4 rows, 420-byte Q6_K rows
    ((768, 512, 8, 2), 100, dict(fmt=D.FMT_MXFP4), 2 + 3),
    ((768, 512, 8, 2), 100, dict(fmt=D.FMT_MXFP4, flags=D.FORCE_TC), 0),
    ((7168, 512, 256, 8), 32, dict(fmt=D.FMT_Q4K, down_fmt=D.FMT_Q6K), 1 + 3),
])
def test_path_choice_by_launch_count(shape, T, kw, launches):
    """The per-call path choice documented under ds4g_moe_forward ("Path"),
    read through ds4g_moe_forward_launches (pure host arithmetic)."""
    assert D.moe_forward_launches(layer_desc(*shape, **kw), T) == launches


def test_expert_cache_create_validates_first():
    """The cache's create checks its descriptor and slot count on the host
    before it allocates anything."""
    L = D.lib()
    h = ctypes.c_void_p()
    assert L.ds4g_expert_cache_create(None, 4, ctypes.byref(h)) == D.ERR_INVALID
    assert L.ds4g_expert_cache_create(ctypes.byref(desc()), 4, None) == D.ERR_INVALID
    assert L.ds4g_expert_cache_create(ctypes.byref(desc()), 1, ctypes.byref(h)) == D.ERR_INVALID  # < top_k
    assert L.ds4g_expert_cache_create(ctypes.byref(desc()), 9, ctypes.byref(h)) == D.ERR_INVALID  # > E
    assert L.ds4g_expert_cache_create(ctypes.byref(desc(n_slots=4, expert_slot=FAKE)), 4,
                                      ctypes.byref(h)) == D.ERR_INVALID
    assert L.ds4g_expert_cache_create(ctypes.byref(desc(hidden=300)), 4, ctypes.byref(h)) == D.ERR_SHAPE
    assert h.value is None
    assert L.ds4g_expert_cache_workspace_bytes(None, 4) == 0
    assert L.ds4g_expert_cache_forward(None, FAKE, FAKE, 4, FAKE, FAKE, 1 << 20, None) == D.ERR_INVALID
    assert L.ds4g_expert_cache_stats(None, None, None, None) == D.ERR_INVALID
    L.ds4g_expert_cache_destroy(None)          # no-op
